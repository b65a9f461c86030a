// Block-scaled grouped matmul for small (decode-sized) groups, with FP8 E4M3
// or bf16 weights:
//   out[r, c] = sum_b s[g, b, c] * sum_{kk in block b} lhs[r, kk] * W(g, c, kk) + bias[g, c]
// (page "tpu-inference 0.12.0.dev20251213 -> 0.13.2.dev20251230", gmm.py:
// _accum multiplies each quant block's partial sum by rhs_scale[g, b, 0, n] on
// the block's last k tile and adds rhs_bias once; rhs_scale [G, nb, 1, n],
// block width k // nb).  Accumulation is fp32 across blocks with one final
// rounding (the pages round the running result to the output dtype after
// every block; this kernel keeps it in fp32 registers instead).
//
// The weight tile is the MMA's M side (128 rows of n) and the group's tokens
// its N side (16 per item), so a group of a few rows costs one pass over its
// weights.  Per 128-wide k step:
//   warp 0      TMA: raw weight tile [128 n x 128 k] (e4m3: 16 KB) and the
//               token tile [16 rows x 128 k] bf16 into stage s
//   warps 6-13  (e4m3 only) decode the raw tile to bf16 into the K-major,
//               128-byte-swizzled A operand of stage s
//   warp 1      TMEM owner; issues 8 tcgen05.mma 128x16x16 into the
//               accumulator slot of the current quant block
//   warps 2-5   per quant block: TMEM -> registers, multiply by the block's
//               scale for this lane's n, add into fp32 registers; at the end of
//               the item add the bias, round and store the token rows
// For bf16 weights the TMA writes the A operand directly and warps 6-13 idle.
//
// e4m3fn -> bf16 is exact: every e4m3fn value is a bf16 value.  The decoder
// places the 7 exponent/mantissa bits of the code at bf16 bits 4..10 (giving
// the bf16 number 2^-120 times the code's value, subnormals included) and
// multiplies by 2^120; the two NaN codes (0x7F, 0xFF) are mapped to NaN.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "worklist.cuh"

namespace gmmk {
namespace {

constexpr int BMW = 128;  // weight rows (n) per item = MMA M
constexpr int BT = 16;    // tokens per item = MMA N
constexpr int KS = 128;   // k per pipeline step
constexpr int STAGES = 4;
constexpr int NACC = 8;  // TMEM accumulator slots, one per quant block in flight
constexpr int kConvWarps = 8;
constexpr int kConvThreads = kConvWarps * 32;
constexpr int kMaxGroups = 1024;
constexpr uint32_t A_BYTES = BMW * KS * 2;  // bf16 operand: two 64-wide k atoms
constexpr uint32_t RAW_BYTES = BMW * KS;    // e4m3 tile
constexpr uint32_t B_BYTES = BT * KS * 2;   // token tile: two 64-wide k atoms
constexpr uint32_t TMEM_COLS = NACC * BT;

constexpr uint32_t OFF_A = 0;
constexpr uint32_t OFF_RAW = OFF_A + STAGES * A_BYTES;
constexpr uint32_t OFF_B = OFF_RAW + STAGES * RAW_BYTES;
constexpr uint32_t OFF_CTRL = OFF_B + STAGES * B_BYTES;
constexpr uint32_t OFF_FULL = OFF_CTRL;  // TMA bytes landed
constexpr uint32_t OFF_AFULL = OFF_FULL + 8 * STAGES;  // A operand decoded
constexpr uint32_t OFF_EMPTY = OFF_AFULL + 8 * STAGES;  // MMA done with the stage
constexpr uint32_t OFF_ACCF = OFF_EMPTY + 8 * STAGES;
constexpr uint32_t OFF_ACCE = OFF_ACCF + 8 * NACC;
constexpr uint32_t OFF_DONE = OFF_ACCE + 8 * NACC;
constexpr uint32_t OFF_TMEM = OFF_DONE + 8;
constexpr uint32_t OFF_ABORT = OFF_TMEM + 4;
constexpr uint32_t OFF_OFFS = OFF_CTRL + 512;
constexpr uint32_t OFF_TILES = OFF_OFFS + 4 * (kMaxGroups + 4);
constexpr uint32_t SMEM_USED = OFF_TILES + 4 * (kMaxGroups + 4);
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(OFF_ABORT + 4 <= OFF_OFFS, "control block overlaps the tables");

struct Params {
  const int32_t* group_sizes;
  int32_t num_total_groups, group_offset, num_local_groups;
  int32_t m, n, k;
  const float* scale;
  int32_t num_blocks;
  const void* bias;
  int32_t bias_f32;
  void* out;
  uint32_t* err;
};

// 16 e4m3fn codes (one 16-byte chunk, lowest k first) -> 16 bf16 (8 words).
// Per pair of codes: the two bytes go to the high byte of each 16-bit half,
// their 7 exponent/mantissa bits move to bf16 bits 4..10 (a bf16 number equal
// to 2^-120 times the code's value, subnormal codes included), a bf16x2 fma
// multiplies by 2^120 (exact) and the sign bit is merged back.  The two NaN
// codes (low 7 bits all ones) would come out as +-480; a chunk holding one is
// rare, so it is found with a zero-byte test and fixed on a separate path.
__device__ __forceinline__ void decode16(const uint4 raw, uint32_t (&o)[8]) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  uint32_t nan_any = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t t = ~w[i] & 0x7F7F7F7Fu;  // a zero byte marks a NaN code
    nan_any |= (t - 0x01010101u) & 0x80808080u;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t v = __byte_perm(w[i], 0u, h == 0 ? 0x1404u : 0x3424u);
      const uint32_t mag = (v >> 4) & 0x07F007F0u;
      uint32_t y;
      asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(y) : "r"(mag), "r"(0x7B807B80u), "r"(0u));
      o[2 * i + h] = y | (v & 0x80008000u);
    }
  }
  if (nan_any != 0u) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t v = __byte_perm(w[i], 0u, h == 0 ? 0x1404u : 0x3424u);
        if ((v & 0x00007F00u) == 0x00007F00u) o[2 * i + h] = (o[2 * i + h] & 0xFFFF0000u) | 0x7FC0u;
        if ((v & 0x7F000000u) == 0x7F000000u) o[2 * i + h] = (o[2 * i + h] & 0x0000FFFFu) | 0x7FC00000u;
      }
    }
  }
}

template <bool kE4M3, bool kOutF32>
__global__ void __launch_bounds__(kE4M3 ? 192 + kConvThreads : 192, 1)
    gemm_scaled_kernel(const __grid_constant__ CUtensorMap tm_lhs, const __grid_constant__ CUtensorMap tm_rhs,
                       const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + OFF_ABORT);
  int32_t* offs = reinterpret_cast<int32_t*>(smem + OFF_OFFS);
  int32_t* tiles = reinterpret_cast<int32_t*>(smem + OFF_TILES);
  auto full_bar = [&](uint32_t s) { return sbase + OFF_FULL + 8 * s; };
  auto afull_bar = [&](uint32_t s) { return sbase + OFF_AFULL + 8 * s; };
  auto empty_bar = [&](uint32_t s) { return sbase + OFF_EMPTY + 8 * s; };
  auto accf_bar = [&](uint32_t b) { return sbase + OFF_ACCF + 8 * b; };
  auto acce_bar = [&](uint32_t b) { return sbase + OFF_ACCE + 8 * b; };
  const uint32_t done_bar = sbase + OFF_DONE;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(afull_bar(s), kConvThreads);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < NACC; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), 128);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch(&tm_lhs);
    tma_prefetch(&tm_rhs);
  }
  if (warp == 1) {
    tmem_alloc(sbase + OFF_TMEM, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 2) {
    build_group_offsets(p.group_sizes, p.num_total_groups, p.m, offs, p.err);
    build_tile_prefix(offs, p.group_offset, p.num_local_groups, BT, tiles);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + OFF_TMEM);

  const int32_t t_tiles = tiles[p.num_local_groups];  // token chunks over all local groups
  const int32_t n_tiles = (p.n + BMW - 1) / BMW;
  const int32_t ksteps = p.k / KS;                     // k % 128 == 0 on this path
  const int32_t nb = p.scale != nullptr ? p.num_blocks : 1;
  const int32_t steps_per_block = ksteps / nb;         // (k / nb) % 128 == 0 on this path
  const int32_t total = t_tiles * n_tiles;
  // Items: token chunks outer, the weight tiles of the chunk's group inner.
  auto item_of = [&](int32_t w) {
    return decode_gemm_tile(w, t_tiles, n_tiles, n_tiles, tiles, offs, p.group_offset, p.num_local_groups, BT);
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, pend_mask = 0;
      uint32_t pend_par[STAGES];
      bool ok = true;
      for (int32_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
        const GemmTile t = item_of(w);
        for (int32_t ks = 0; ks < ksteps; ++ks) {
          if (!wait_bar(empty_bar(stage), phase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, (kE4M3 ? RAW_BYTES : A_BYTES) + B_BYTES);
          if constexpr (kE4M3) {
            tma_load_3d(sbase + OFF_RAW + stage * RAW_BYTES, &tm_rhs, fb, ks * KS, t.n_tile * BMW, t.local_group);
          } else {
#pragma unroll
            for (int h = 0; h < 2; ++h)
              tma_load_3d(sbase + OFF_A + stage * A_BYTES + h * (A_BYTES / 2), &tm_rhs, fb, ks * KS + 64 * h,
                          t.n_tile * BMW, t.local_group);
          }
#pragma unroll
          for (int h = 0; h < 2; ++h)
            tma_load_2d(sbase + OFF_B + stage * B_BYTES + h * (B_BYTES / 2), &tm_lhs, fb, ks * KS + 64 * h, t.row0);
          pend_par[stage] = phase;
          pend_mask |= 1u << stage;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        for (int s = 0; s < STAGES; ++s)
          if (pend_mask >> s & 1u) drain_bar(full_bar(s), pend_par[s]);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    constexpr uint32_t kIdesc = idesc_bf16(BMW, BT, false, false);
    uint32_t stage = 0, phase = 0, slot = 0, slot_phase = 0;
    bool ok = true;
    for (int32_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
      for (int32_t ks = 0; ks < ksteps; ++ks) {
        const int32_t in_block = ks % steps_per_block;
        if (in_block == 0) {
          if (!wait_bar(acce_bar(slot), slot_phase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
        }
        if (!wait_bar(full_bar(stage), phase, abort_flag, p.err)) {
          ok = false;
          break;
        }
        if constexpr (kE4M3) {
          if (!wait_bar(afull_bar(stage), phase, abort_flag, p.err)) {
            ok = false;
            break;
          }
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a0 = sbase + OFF_A + stage * A_BYTES;
          const uint32_t b0 = sbase + OFF_B + stage * B_BYTES;
          const uint32_t d_tmem = tmem_base + slot * BT;
#pragma unroll
          for (int kk = 0; kk < KS / 16; ++kk) {
            const int h = kk >> 2;
            const uint64_t ad = sw128_desc(a0 + h * (A_BYTES / 2) + (kk & 3) * 32, 16, 1024);
            const uint64_t bd = sw128_desc(b0 + h * (B_BYTES / 2) + (kk & 3) * 32, 16, 1024);
            mma_bf16_ss(d_tmem, ad, bd, kIdesc, (in_block | kk) != 0 ? 1u : 0u);
          }
          mma_commit(empty_bar(stage));
          if (in_block == steps_per_block - 1) mma_commit(accf_bar(slot));
        }
        __syncwarp();
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
        if (in_block == steps_per_block - 1) {
          if (++slot == NACC) {
            slot = 0;
            slot_phase ^= 1u;
          }
        }
      }
    }
    if (lane == 0) {
      mma_commit(done_bar);
      drain_bar(done_bar, 0);
    }
    __syncwarp();
  } else if (warp < 6) {
    // ---------------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const int wrow = quarter * 32 + lane;  // weight row in the tile = output column
    uint32_t slot = 0, slot_phase = 0;
    bool ok = true;
    for (int32_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
      const GemmTile t = item_of(w);
      const int32_t col = t.n_tile * BMW + wrow;
      const bool col_ok = col < p.n;
      float acc[BT];
#pragma unroll
      for (int i = 0; i < BT; ++i) acc[i] = 0.f;
      const float* srow = p.scale != nullptr ? p.scale + int64_t(t.local_group) * nb * p.n + col : nullptr;
      float s_next = (srow != nullptr && col_ok) ? __ldg(srow) : 1.f;
      for (int32_t b = 0; b < nb; ++b) {
        const float s = s_next;
        if (srow != nullptr && col_ok && b + 1 < nb) s_next = __ldg(srow + int64_t(b + 1) * p.n);
        if (!wait_bar(accf_bar(slot), slot_phase, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t v[BT];
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
            "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
            "tcgen05.wait::ld.sync.aligned;"
            : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
              "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
            : "r"(tmem_base + (uint32_t(quarter * 32) << 16) + slot * BT)
            : "memory");
        tc_fence_before();
        mbar_arrive(acce_bar(slot));
#pragma unroll
        for (int i = 0; i < BT; ++i) acc[i] = fmaf(s, __uint_as_float(v[i]), acc[i]);
        if (++slot == NACC) {
          slot = 0;
          slot_phase ^= 1u;
        }
      }
      if (!ok) break;
      if (!col_ok) continue;
      float bias = 0.f;
      if (p.bias != nullptr) {
        const int64_t bi = int64_t(t.local_group) * p.n + col;
        bias = p.bias_f32 ? __ldg(static_cast<const float*>(p.bias) + bi)
                          : __bfloat162float(static_cast<const __nv_bfloat16*>(p.bias)[bi]);
      }
#pragma unroll
      for (int i = 0; i < BT; ++i) {
        const int32_t row = t.row0 + i;
        if (row < t.row_end) {
          const float r = acc[i] + bias;
          if constexpr (kOutF32)
            static_cast<float*>(p.out)[int64_t(row) * p.n + col] = r;
          else
            static_cast<__nv_bfloat16*>(p.out)[int64_t(row) * p.n + col] = __float2bfloat16_rn(r);
        }
      }
    }
    // Rows outside [offs[first local], offs[last local + 1]) are zero.
    const int64_t row_bytes = int64_t(p.n) * (kOutF32 ? 4 : 2);
    const int64_t lo_bytes = int64_t(offs[p.group_offset]) * row_bytes;
    const int64_t hi_begin = int64_t(offs[p.group_offset + p.num_local_groups]) * row_bytes;
    const int64_t n_lo = lo_bytes / 16;
    const int64_t n_all = n_lo + (int64_t(p.m) * row_bytes - hi_begin) / 16;
    const int64_t stride = int64_t(gridDim.x) * 128;
    for (int64_t i = int64_t(blockIdx.x) * 128 + (threadIdx.x - 64); i < n_all; i += stride) {
      const int64_t byte = i < n_lo ? i * 16 : hi_begin + (i - n_lo) * 16;
      st_global_v4(static_cast<uint8_t*>(p.out) + byte, 0u, 0u, 0u, 0u);
    }
  } else if constexpr (kE4M3) {
    // ---------------------------------------------------------------- e4m3 -> bf16 decoders
    // Unit u of a stage = (row r, 16-byte raw chunk c) with r = u % 8 + 8 * (u / 64)
    // and c = (u / 8) % 8, so the 8 lanes of each quarter-warp (one shared-memory
    // phase of a 16-byte access) take the same chunk of 8 consecutive rows.
    // Raw row r holds k [0, 128) as 8 chunks at positions c ^ (r % 8); the bf16
    // A operand holds k [0, 64) and [64, 128) in two atoms whose rows hold 8
    // chunks of 8 bf16 at positions j ^ (r % 8): the 8 lanes of a phase hit 8
    // different positions on every load and store.
    const int ct = threadIdx.x - 192;
    uint32_t stage = 0, phase = 0;
    bool ok = true;
    for (int32_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
      for (int32_t ks = 0; ks < ksteps; ++ks) {
        if (!wait_bar(full_bar(stage), phase, abort_flag, p.err)) {
          ok = false;
          break;
        }
        const uint32_t raw0 = sbase + OFF_RAW + stage * RAW_BYTES;
        const uint32_t a0 = sbase + OFF_A + stage * A_BYTES;
#pragma unroll
        for (int i = 0; i < (BMW * 8) / kConvThreads; ++i) {
          const int u = ct + i * kConvThreads;
          const int r = (u & 7) + ((u >> 6) << 3), c = (u >> 3) & 7, sw = r & 7;
          uint4 raw;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(raw.x), "=r"(raw.y), "=r"(raw.z), "=r"(raw.w)
                       : "r"(raw0 + r * 128 + ((c ^ sw) << 4)));
          uint32_t o[8];
          decode16(raw, o);
          const uint32_t atom = a0 + (c >> 2) * (A_BYTES / 2) + r * 128;
          const int j = (c & 3) * 2;
          st_shared_v4(atom + ((j ^ sw) << 4), o[0], o[1], o[2], o[3]);
          st_shared_v4(atom + (((j + 1) ^ sw) << 4), o[4], o[5], o[6], o[7]);
        }
        fence_proxy_async_smem();
        mbar_arrive(afull_bar(stage));
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

template <bool kE4M3, bool kOutF32>
cudaError_t launch_impl(const ScaledLaunch& L, int grid, cudaStream_t stream) {
  auto kern = gemm_scaled_kernel<kE4M3, kOutF32>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(SMEM_BYTES));
  if (e != cudaSuccess) return e;
  Params p{L.group_sizes, L.num_total_groups, L.group_offset, L.num_local_groups, L.m, L.n, L.k, L.scale,
           L.num_blocks, L.bias, L.bias_f32, L.out, L.err};
  kern<<<grid, kE4M3 ? 192 + kConvThreads : 192, SMEM_BYTES, stream>>>(L.tm_lhs, L.tm_rhs, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_scaled(const ScaledLaunch& p, bool rhs_e4m3, bool out_f32, int grid, cudaStream_t stream) {
  if (rhs_e4m3) return out_f32 ? launch_impl<true, true>(p, grid, stream) : launch_impl<true, false>(p, grid, stream);
  return out_f32 ? launch_impl<false, true>(p, grid, stream) : launch_impl<false, false>(p, grid, stream);
}

}  // namespace gmmk
