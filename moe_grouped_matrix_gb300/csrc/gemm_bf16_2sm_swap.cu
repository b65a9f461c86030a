// Forward grouped matmul on SM pairs with the operands' roles swapped, for
// groups of tens to a few hundred rows (Zipf-routed experts): the same
// computation as gemm_bf16.cu (page "tpu-inference 0.12.0.dev20251213 ->
// 0.13.2.dev20251230", gmm.py: gmm without quant blocks; NT [L, n, k] or NN
// [L, k, n] weights read in place).
//
// 256 weight rows (n) are the M side of tcgen05.mma.cta_group::2, 128 in each
// CTA of the pair; up to 256 of a group's rows are its N side, split in halves
// between the two CTAs.  N is the chunk's row count rounded up to 32 and set
// at run time in the instruction descriptor, so a group's last chunk wastes at
// most 31 rows of MMA work (256-row tiles of rows waste up to 255: 1.5x the
// useful work on Zipf-routed experts, against ~1.05x here), while each SM still
// loads only its own 128 weight rows and half of the chunk's rows per k step.
//
// Roles, per CTA (192 threads):
//   warp 0     TMA producer (both CTAs): this CTA's 128 weight rows and its
//              N/2 chunk rows per 128-wide k step (two 64-wide boxes each, 3
//              stages of 64 KB); bytes of both CTAs' copies
//              land on the stage's full barrier in the leader CTA
//   warp 1     TMEM (512 columns, allocated by both CTAs together); in the
//              leader CTA it also issues the MMAs (M = 256, N, K = 16)
//   warps 2-5  epilogue of this CTA's 128 weight rows: lane = output column;
//              for each of the chunk's rows a warp stores 32 consecutive columns
// Work items are (group, 256-row chunk, 256-wide n tile), chunks outer.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "worklist.cuh"

namespace gmmk {
namespace {

constexpr int BW = 128;      // weight rows per CTA (its half of the MMA's M = 256)
constexpr int PAIR_W = 256;  // weight rows (n) per pair tile
constexpr int CHUNK = 256;   // largest N: rows of a group per item
constexpr int BK = 128;      // k per stage: two 64-wide boxes, adjacent in k, per operand
constexpr int KH = BK / 64;
constexpr int STAGES = 3;
constexpr int kThreads = 192;
constexpr int kMaxGroups = 1024;
constexpr uint32_t A_HALF = BW * 64 * 2;               // this CTA's weight rows over 64 k
constexpr uint32_t A_BYTES = KH * A_HALF;
constexpr uint32_t B_HALF = (CHUNK / 2) * 64 * 2;      // up to half a chunk of rows over 64 k
constexpr uint32_t B_BYTES = KH * B_HALF;
constexpr uint32_t TBOX_BYTES = 64 * 64 * 2;           // one {64 k, 64 rows} box of rows
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t TMEM_COLS = 2 * CHUNK;

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

// Rows of the item's chunk, and the MMA N covering them (a multiple of 32, so
// each CTA of the pair holds a multiple of 16 of them).
__device__ __forceinline__ int32_t chunk_rows(const GemmTile& t) { return min(CHUNK, t.row_end - t.row0); }
__device__ __forceinline__ int32_t chunk_n(const GemmTile& t) { return (chunk_rows(t) + 31) & ~31; }

template <bool kNT, bool kOutF32>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_bf16_2sm_swap_kernel(const __grid_constant__ CUtensorMap tm_lhs, const __grid_constant__ CUtensorMap tm_rhs,
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
    build_tile_prefix(offs, go, p.num_local_groups, CHUNK, tiles);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + OFF_TMEM);

  const int32_t t_tiles = tiles[p.num_local_groups];  // 256-row chunks over all local groups
  const int32_t n_tiles = (p.n + PAIR_W - 1) / PAIR_W;
  const int32_t k_blocks = (p.k + BK - 1) / BK;
  const int32_t total = t_tiles * n_tiles;
  // chunks outer, the n tiles of the chunk's group inner
  auto tile_of = [&](int32_t w) {
    return decode_gemm_tile(w, t_tiles, n_tiles, n_tiles, tiles, offs, go, p.num_local_groups, CHUNK);
  };

  // the bytes one CTA's copies of a stage of work item w carry
  auto cta_stage_bytes = [&](int32_t w) {
    return A_BYTES + uint32_t(KH * ((chunk_n(tile_of(w)) / 2 + 63) / 64)) * TBOX_BYTES;
  };

  uint32_t issued = 0;  // producer: stages of the pair's sequence this CTA issued (leader: armed)
  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer (both CTAs)
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int32_t w = pair; w < total && ok; w += npairs) {
        const GemmTile t = tile_of(w);
        const int32_t half = chunk_n(t) / 2;  // rows of the chunk this CTA holds
        const int32_t nbox = (half + 63) / 64;
        const int32_t trow = t.row0 + int32_t(rank) * half;
        const int32_t wrow = t.n_tile * PAIR_W + int32_t(rank) * BW;
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
          if (leader) mbar_arrive_expect_tx(full_bar(stage), 2u * (A_BYTES + uint32_t(KH * nbox) * TBOX_BYTES));
          const uint32_t fb = mapa_shared(full_bar(stage), 0);
          const uint32_t a_dst = sbase + OFF_A + stage * A_BYTES;
          const uint32_t b_dst = sbase + OFF_B + stage * B_BYTES;
#pragma unroll
          for (int kh = 0; kh < KH; ++kh) {
            const int32_t kc = kb * BK + 64 * kh;  // past k the boxes are zero-filled
            if constexpr (kNT) {
              tma_load_3d_pair(a_dst + kh * A_HALF, &tm_rhs, fb, kc, wrow, t.local_group);
            } else {
#pragma unroll
              for (int j = 0; j < BW / 64; ++j)
                tma_load_3d_pair(a_dst + kh * A_HALF + j * 8192u, &tm_rhs, fb, wrow + 64 * j, kc, t.local_group);
            }
            for (int32_t j = 0; j < nbox; ++j)
              tma_load_2d_pair(b_dst + kh * B_HALF + j * TBOX_BYTES, &tm_lhs, fb, kc, trow + 64 * j);
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
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int32_t w = pair; w < total && ok; w += npairs) {
        const GemmTile t = tile_of(w);
        // A = weights (K-major for NT, MN-major for NN), B = the chunk's rows (K-major)
        const uint32_t idesc = idesc_bf16(2 * BW, chunk_n(t), !kNT, false);
        if (!wait_bar_cluster(acce_bar(acc), acc_phase ^ 1u, abort_flag, p.err, p.wait_limit)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * CHUNK;
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
              const uint32_t ah = a0 + (kk / 4) * A_HALF, bh = b0 + (kk / 4) * B_HALF;
              const int kq = kk % 4;
              const uint64_t ad =
                  kNT ? sw128_desc(ah + kq * 32, 16, 1024) : sw128_desc(ah + kq * 2048, 8192, 1024);
              const uint64_t bd = sw128_desc(bh + kq * 32, 16, 1024);
              mma_bf16_ss_pair(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
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
    // TMEM lane = this CTA's weight row = output column; TMEM column = row of the chunk.
    const int quarter = warp & 3;
    uint32_t acc = 0, acc_phase = 0;
    for (int32_t w = pair; w < total; w += npairs) {
      const GemmTile t = tile_of(w);
      const int32_t rows = chunk_rows(t), ncols = chunk_n(t);
      const int32_t col = t.n_tile * PAIR_W + int32_t(rank) * BW + quarter * 32 + lane;
      const bool col_ok = col < p.n;
      float bias = 0.f;
      if (p.bias != nullptr && col_ok) {
        const int64_t bi = int64_t(t.local_group) * p.n + col;
        bias = p.bias_f32 ? __ldg(static_cast<const float*>(p.bias) + bi)
                          : __bfloat162float(static_cast<const __nv_bfloat16*>(p.bias)[bi]);
      }
      if (!wait_bar(accf_bar(acc), acc_phase, abort_flag, p.err, p.wait_limit)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (uint32_t(quarter * 32) << 16) + acc * CHUNK;
#pragma unroll 1
      for (int32_t c0 = 0; c0 < ncols; c0 += 32) {
        uint32_t v[32];
        tmem_ld_32cols(tbase + c0, v);
        if (c0 + 32 >= ncols) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(acce_bar(acc), 0));
        }
        if (col_ok) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (c0 + i < rows) {
              const int64_t o = int64_t(t.row0 + c0 + i) * p.n + col;
              const float r = __uint_as_float(v[i]) + bias;
              if constexpr (kOutF32)
                static_cast<float*>(p.out)[o] = r;
              else
                static_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(r);
            }
          }
        }
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
    // stage i of the sequence belongs to the pair's (i / k_blocks)-th work item
    pair_drain<STAGES>(full_bar(0), sbase + OFF_REPORT, sbase + OFF_RWORD, issued, p.wait_limit,
                       [&](uint32_t i) { return cta_stage_bytes(pair + int32_t(i / uint32_t(k_blocks)) * npairs); });
  }
  cluster_sync();  // the leader's MMAs and every copy are done; no signal targets either CTA any more
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

template <bool kNT, bool kOutF32>
cudaError_t launch_impl(const GemmLaunch& L, int max_ctas, cudaStream_t stream) {
  auto kern = gemm_bf16_2sm_swap_kernel<kNT, kOutF32>;
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

cudaError_t launch_gemm_bf16_2sm_swap(const GemmLaunch& p, bool nt, bool out_f32, int max_ctas, cudaStream_t stream) {
  if (nt) return out_f32 ? launch_impl<true, true>(p, max_ctas, stream) : launch_impl<true, false>(p, max_ctas, stream);
  return out_f32 ? launch_impl<false, true>(p, max_ctas, stream) : launch_impl<false, false>(p, max_ctas, stream);
}

}  // namespace gmmk
