// Forward grouped matmul on SM pairs: the same computation as gemm_bf16.cu
// (page "tpu-inference 0.12.0.dev20251213 -> 0.13.2.dev20251230", gmm.py: gmm
// without quant blocks; NT weights [L, n, k] or NN [L, k, n] read in place),
// with 256 x 256 output tiles computed by a cluster of two CTAs on two SMs
// through tcgen05.mma.cta_group::2.
//
// Each CTA of the pair loads its own 128 lhs rows and its own 128 of the 256
// weight rows (n) per 64-wide k step, 32 KB instead of 48 KB for a 128 x 256
// tile on one SM; the tensor cores of the pair exchange the weight halves.  So
// every SM pulls a third less from L2 and writes a third less into shared
// memory per MMA, and the smaller stage leaves room for a 6-deep ring.
//
// Roles, per CTA (192 threads):
//   warp 0     TMA producer (both CTAs); completion bytes of both CTAs'
//              copies land on the stage's full barrier in the leader CTA
//   warp 1     TMEM (512 columns, allocated by both CTAs together); in the
//              leader CTA it also issues the MMAs (M = 256 over the pair,
//              N = 256, K = 16) and commits to barriers in both CTAs
//   warps 2-5  epilogue of this CTA's 128 rows; they release the accumulator
//              by arriving on the leader's barrier
// Work items are (group, 256-row block from the group's first row, n tile);
// the second CTA's rows may run past the group and are masked at the store.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "worklist.cuh"

namespace gmmk {
namespace {

constexpr int BM = 128;      // rows per CTA
constexpr int PAIR_M = 256;  // rows per pair tile
constexpr int BN = 256;      // n per pair tile; each CTA holds 128
constexpr int BK = 64;
constexpr int STAGES = 6;
constexpr int kThreads = 192;
constexpr int kMaxGroups = 1024;
constexpr uint32_t A_BYTES = BM * BK * 2;
constexpr uint32_t B_BYTES = (BN / 2) * BK * 2;
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t TMEM_COLS = 2 * BN;

constexpr uint32_t OFF_A = 0;
constexpr uint32_t OFF_B = STAGES * A_BYTES;
constexpr uint32_t OFF_CTRL = STAGES * STAGE_BYTES;
constexpr uint32_t OFF_FULL = OFF_CTRL;
constexpr uint32_t OFF_EMPTY = OFF_FULL + 8 * STAGES;
constexpr uint32_t OFF_ACCF = OFF_EMPTY + 8 * STAGES;
constexpr uint32_t OFF_ACCE = OFF_ACCF + 16;
constexpr uint32_t OFF_DONE = OFF_ACCE + 16;
constexpr uint32_t OFF_TMEM = OFF_DONE + 8;
constexpr uint32_t OFF_ABORT = OFF_TMEM + 4;
constexpr uint32_t OFF_REPORT = OFF_ABORT + 4;  // pair_report's barrier and count (leader's)
constexpr uint32_t OFF_RWORD = OFF_REPORT + 8;
constexpr uint32_t OFF_OFFS = OFF_CTRL + 256;
constexpr uint32_t OFF_TILES = OFF_OFFS + 4 * (kMaxGroups + 4);
constexpr uint32_t SMEM_USED = OFF_TILES + 4 * (kMaxGroups + 4);
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(OFF_RWORD + 4 <= OFF_OFFS && OFF_REPORT % 8 == 0, "control block overlaps the tables");

struct Params {
  const int32_t* group_sizes;
  int32_t num_total_groups, group_offset, num_local_groups;
  int32_t m, n, k;
  void* out;
  const void* bias;
  int32_t bias_f32;
  uint32_t* err;
  int32_t raster;
  int32_t zero_rest;  // zero the rows outside the local groups (gmm) or leave them (gmm_into)
  const int32_t* group_offset_dev;  // NULL, or the device scalar that replaces group_offset
  long long wait_limit;             // bound of every pipeline wait, in clock cycles
  int32_t drop_stage;               // 0, or s > 0: the first pair's second CTA stops before its s-th stage (test)
};

template <bool kOutF32>
__device__ __forceinline__ void store_row_chunk(const Params& p, int32_t row, int32_t col0, int32_t lgroup,
                                                const uint32_t (&v)[32]) {
  float f[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
  if (p.bias != nullptr) {
    const int64_t bidx = int64_t(lgroup) * p.n + col0;
    if (p.bias_f32) {
      const float* b = static_cast<const float*>(p.bias) + bidx;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (col0 + i < p.n) f[i] += __ldg(b + i);
    } else {
      const __nv_bfloat16* b = static_cast<const __nv_bfloat16*>(p.bias) + bidx;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (col0 + i < p.n) f[i] += __bfloat162float(b[i]);
    }
  }
  if constexpr (kOutF32) {
    float* o = static_cast<float*>(p.out) + int64_t(row) * p.n + col0;
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (col0 + 4 * q < p.n)
        st_global_v4(o + 4 * q, __float_as_uint(f[4 * q]), __float_as_uint(f[4 * q + 1]),
                     __float_as_uint(f[4 * q + 2]), __float_as_uint(f[4 * q + 3]));
  } else {
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) + int64_t(row) * p.n + col0;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (col0 + 8 * q < p.n)
        st_global_v4(o + 8 * q, pack_bf16x2(f[8 * q], f[8 * q + 1]), pack_bf16x2(f[8 * q + 2], f[8 * q + 3]),
                     pack_bf16x2(f[8 * q + 4], f[8 * q + 5]), pack_bf16x2(f[8 * q + 6], f[8 * q + 7]));
  }
}

template <bool kNT, bool kOutF32>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_bf16_2sm_kernel(const __grid_constant__ CUtensorMap tm_lhs, const __grid_constant__ CUtensorMap tm_rhs,
                         const Params p) {
  int32_t go;
  if (!resolve_group_offset(p.group_offset_dev, p.group_offset, p.num_total_groups, p.num_local_groups, p.err, go))
    return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int32_t pair = blockIdx.x >> 1;
  const int32_t npairs = gridDim.x >> 1;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + OFF_ABORT);
  int32_t* offs = reinterpret_cast<int32_t*>(smem + OFF_OFFS);
  int32_t* tiles = reinterpret_cast<int32_t*>(smem + OFF_TILES);
  auto full_bar = [&](uint32_t s) { return sbase + OFF_FULL + 8 * s; };
  auto empty_bar = [&](uint32_t s) { return sbase + OFF_EMPTY + 8 * s; };
  auto accf_bar = [&](uint32_t b) { return sbase + OFF_ACCF + 8 * b; };
  auto acce_bar = [&](uint32_t b) { return sbase + OFF_ACCE + 8 * b; };
  const uint32_t done_bar = sbase + OFF_DONE;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);   // the leader's expect_tx; bytes from both CTAs
      mbar_init(empty_bar(s), 1);  // the leader's MMA commit, multicast to both
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);  // MMA commit, multicast to both
      mbar_init(acce_bar(b), 8);  // one lane of each epilogue warp of both CTAs
    }
    mbar_init(done_bar, 1);
    mbar_init(sbase + OFF_REPORT, 1);  // the follower's pair_report
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch(&tm_lhs);
    tma_prefetch(&tm_rhs);
  }
  if (warp == 1) {
    tmem_alloc_pair(sbase + OFF_TMEM, TMEM_COLS);
    tmem_relinquish_pair();
  }
  if (warp == 2) {
    build_group_offsets(p.group_sizes, p.num_total_groups, p.m, offs, p.err);
    build_tile_prefix(offs, go, p.num_local_groups, PAIR_M, tiles);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + OFF_TMEM);

  const int32_t m_tiles = tiles[p.num_local_groups];
  const int32_t n_tiles = (p.n + BN - 1) / BN;
  const int32_t k_blocks = (p.k + BK - 1) / BK;
  const int32_t total = m_tiles * n_tiles;
  auto tile_of = [&](int32_t w) {
    return decode_gemm_tile(w, m_tiles, n_tiles, p.raster, tiles, offs, go, p.num_local_groups,
                            PAIR_M);
  };

  uint32_t issued = 0;  // producer: stages of the pair's sequence this CTA issued (leader: armed)
  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer (both CTAs)
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int32_t w = pair; w < total && ok; w += npairs) {
        const GemmTile t = tile_of(w);
        const int32_t row = t.row0 + int32_t(rank) * BM;
        const int32_t ncol = t.n_tile * BN + int32_t(rank) * (BN / 2);
        for (int32_t kb = 0; kb < k_blocks; ++kb) {
          if (!wait_bar(empty_bar(stage), phase ^ 1u, abort_flag, p.err, p.wait_limit)) {
            ok = false;
            break;
          }
          if (blockIdx.x == 1 && issued + 1 == uint32_t(p.drop_stage)) {
            // timeout test: the follower stops issuing, so the leader's wait for
            // this stage's bytes runs out
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(full_bar(stage), 2 * STAGE_BYTES);
          const uint32_t fb = mapa_shared(full_bar(stage), 0);
          const uint32_t a_dst = sbase + OFF_A + stage * A_BYTES;
          const uint32_t b_dst = sbase + OFF_B + stage * B_BYTES;
          tma_load_2d_pair(a_dst, &tm_lhs, fb, kb * BK, row);
          if constexpr (kNT) {
            tma_load_3d_pair(b_dst, &tm_rhs, fb, kb * BK, ncol, t.local_group);
          } else {
#pragma unroll
            for (int j = 0; j < BN / 128; ++j)
              tma_load_3d_pair(b_dst + j * 8192u, &tm_rhs, fb, ncol + 64 * j, kb * BK, t.local_group);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!leader) pair_report(sbase + OFF_REPORT, sbase + OFF_RWORD, issued);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (leader CTA)
    if (leader) {
      constexpr uint32_t kIdesc = idesc_bf16(PAIR_M, BN, false, !kNT);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int32_t w = pair; w < total && ok; w += npairs) {
        if (!wait_bar_cluster(acce_bar(acc), acc_phase ^ 1u, abort_flag, p.err, p.wait_limit)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int32_t kb = 0; kb < k_blocks; ++kb) {
          if (!wait_bar(full_bar(stage), phase, abort_flag, p.err, p.wait_limit)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (lane == 0) {
            const uint32_t a0 = sbase + OFF_A + stage * A_BYTES;
            const uint32_t b0 = sbase + OFF_B + stage * B_BYTES;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint64_t ad = sw128_desc(a0 + kk * 32, 16, 1024);
              const uint64_t bd =
                  kNT ? sw128_desc(b0 + kk * 32, 16, 1024) : sw128_desc(b0 + kk * 2048, 8192, 1024);
              mma_bf16_ss_pair(d_tmem, ad, bd, kIdesc, (kb | kk) != 0 ? 1u : 0u);
            }
            mma_commit_pair(empty_bar(stage), 0x3);
          }
          __syncwarp();
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (lane == 0) mma_commit_pair(accf_bar(acc), 0x3);
        __syncwarp();
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (lane == 0) {
        mma_commit_pair(done_bar, 0x1);
        drain_bar(done_bar, 0);
      }
      __syncwarp();
    }
  } else {
    // ---------------------------------------------------------------- epilogue (both CTAs)
    const int quarter = warp & 3;
    const int row_in_tile = int(rank) * BM + quarter * 32 + lane;
    uint32_t acc = 0, acc_phase = 0;
    for (int32_t w = pair; w < total; w += npairs) {
      const GemmTile t = tile_of(w);
      if (!wait_bar(accf_bar(acc), acc_phase, abort_flag, p.err, p.wait_limit)) break;
      tc_fence_after();
      const int32_t row = t.row0 + row_in_tile;
      const bool valid = row < t.row_end;
      const uint32_t tbase = tmem_base + (uint32_t(quarter * 32) << 16) + acc * BN;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t v[32];
        tmem_ld_32cols(tbase + c * 32, v);
        if (c == BN / 32 - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(acce_bar(acc), 0));
        }
        const int32_t col0 = t.n_tile * BN + c * 32;
        if (valid && col0 < p.n) store_row_chunk<kOutF32>(p, row, col0, t.local_group, v);
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // Rows outside [offs[first local], offs[last local + 1]) are zero, unless the
    // caller keeps them (gmm_into).
    if (p.zero_rest) {
      const int64_t row_bytes = int64_t(p.n) * (kOutF32 ? 4 : 2);
      const int64_t lo_bytes = int64_t(offs[go]) * row_bytes;
      const int64_t hi_begin = int64_t(offs[go + p.num_local_groups]) * row_bytes;
      const int64_t n_lo = lo_bytes / 16;
      const int64_t n_all = n_lo + (int64_t(p.m) * row_bytes - hi_begin) / 16;
      const int64_t stride = int64_t(gridDim.x) * 128;
      for (int64_t i = int64_t(blockIdx.x) * 128 + (threadIdx.x - 64); i < n_all; i += stride) {
        const int64_t byte = i < n_lo ? i * 16 : hi_begin + (i - n_lo) * 16;
        st_global_v4(static_cast<uint8_t*>(p.out) + byte, 0u, 0u, 0u, 0u);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (leader && warp == 0 && lane == 0 && *abort_flag) {
    st_shared_cluster_u32(mapa_shared(sbase + OFF_ABORT, 1), 1u);  // the follower's waits end too
    pair_drain<STAGES>(full_bar(0), sbase + OFF_REPORT, sbase + OFF_RWORD, issued, p.wait_limit,
                       [](uint32_t) { return STAGE_BYTES; });
  }
  cluster_sync();  // the leader's MMAs and every copy are done; no signal targets either CTA any more
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

template <bool kNT, bool kOutF32>
cudaError_t launch_impl(const GemmLaunch& L, int max_ctas, cudaStream_t stream) {
  auto kern = gemm_bf16_2sm_kernel<kNT, kOutF32>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(SMEM_BYTES));
  if (e != cudaSuccess) return e;
  // One pair per co-resident cluster slot (persistent kernel).
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(max_ctas & ~1);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
  if (e != cudaSuccess) return e;
  if (clusters < 1) return cudaErrorLaunchOutOfResources;
  const int grid = 2 * (clusters < max_ctas / 2 ? clusters : max_ctas / 2);
  Params p{L.group_sizes, L.num_total_groups, L.group_offset, L.num_local_groups, L.m, L.n, L.k, L.out, L.bias,
           L.bias_f32, L.err, L.raster, L.zero_rest, L.group_offset_dev,
           L.wait_limit > 0 ? (long long)L.wait_limit : kWaitLimitCycles, L.drop_stage};
  kern<<<grid, kThreads, SMEM_BYTES, stream>>>(L.tm_lhs, L.tm_rhs, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_bf16_2sm(const GemmLaunch& p, bool nt, bool out_f32, int max_ctas, cudaStream_t stream) {
  if (nt) return out_f32 ? launch_impl<true, true>(p, max_ctas, stream) : launch_impl<true, false>(p, max_ctas, stream);
  return out_f32 ? launch_impl<false, true>(p, max_ctas, stream) : launch_impl<false, false>(p, max_ctas, stream);
}

}  // namespace gmmk
