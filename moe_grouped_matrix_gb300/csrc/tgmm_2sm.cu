// Backward weight gradient per group on SM pairs: the same computation as
// tgmm.cu, out[g, kk, c] = sum_{r in group group_offset + g} lhs[r, kk] * dout[r, c]
// (page "Megablox: transposed-RHS gmm_v2 kernel for the backward dlhs", Context:
// the drhs of the grouped matmul; page "tpu-inference ...", gmm.py
// make_group_metadata: every group, empty ones included, gets its output), with
// 256 x 256 output tiles computed by a cluster of two CTAs through
// tcgen05.mma.cta_group::2.
//
// Every output tile streams all of its group's rows.  Each CTA of the pair
// loads its own 128 lhs columns (A, MN-major) and its 128 of the tile's 256 dout
// columns (B, MN-major) per 64-row chunk: 512 bytes per row instead of the 768
// a 128 x 256 tile on one SM needs, so the same shared memory holds a 5-deep ring
// (320 rows in flight per SM instead of 192).  On the 128-expert workload this
// runs as fast as the one-SM kernel (the output write stream sets both), which
// stays the default; this one is selected per call (gmm_options.tgmm_kernel).
//
// A group's last chunk may run into the next group's rows.  Their products must
// not enter the sum, and zero rows of B (dout) suffice for that whatever A
// holds.  Both CTAs' copies complete on the leader's full barrier, so the
// leader's MMA warp, once a tail chunk has landed, zeroes those B rows in its
// own shared memory and, through st.shared::cluster, in the peer's, fences them
// to the async proxy and issues: no handshake between the CTAs per chunk.
//
// Roles, per CTA (192 threads):
//   warp 0     TMA producer for this CTA's operand halves; completion bytes of
//              both CTAs' copies land on the stage's full barrier in the leader
//   warp 1     TMEM (512 columns, allocated by both CTAs together); in the
//              leader it zeroes tail rows and issues the MMAs (M = 256 over the
//              pair, N = 256, K = 16), committing to barriers in both CTAs
//   warps 2-5  epilogue of this CTA's 128 output rows: TMEM -> 128-byte-
//              swizzled shared-memory slices -> TMA bulk tensor stores (the TMA
//              clips the k and n tails); empty groups' tiles are written as
//              zeros without TMEM
// Work items are (local group, 256-wide k pair tile, 256-wide n tile).
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "worklist.cuh"

namespace gmmk {
namespace {

constexpr int BM = 128;      // output rows (lhs columns) per CTA
constexpr int PAIR_M = 256;  // output rows per pair tile
constexpr int BN = 256;      // output columns (dout columns) per pair tile; each CTA loads 128
constexpr int BR = 64;       // contraction rows per stage
constexpr int STAGES = 5;
constexpr int kThreads = 192;
constexpr int kMaxGroups = 1024;
constexpr uint32_t BOX_BYTES = 64 * 64 * 2;            // one 64-feature x 64-row box
constexpr uint32_t A_BYTES = (BM / 64) * BOX_BYTES;      // this CTA's 128 lhs columns
constexpr uint32_t B_BYTES = (BN / 2 / 64) * BOX_BYTES;  // this CTA's 128 dout columns
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr uint32_t SLICE_BYTES = 32 * 128;  // one warp's 32 rows x 128 bytes of output

constexpr uint32_t OFF_A = 0;
constexpr uint32_t OFF_B = STAGES * A_BYTES;
constexpr uint32_t OFF_OUT = STAGES * STAGE_BYTES;  // 4 warps x 2 slices
constexpr uint32_t OFF_CTRL = OFF_OUT + 8 * SLICE_BYTES;
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
constexpr uint32_t SMEM_USED = OFF_OFFS + 4 * (kMaxGroups + 4);
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(OFF_RWORD + 4 <= OFF_OFFS && OFF_REPORT % 8 == 0, "control block overlaps the tables");

struct Params {
  const int32_t* group_sizes;
  int32_t num_total_groups, group_offset, num_local_groups;
  int32_t m, n, k;
  void* out;
  uint32_t* err;
  long long wait_limit;  // bound of every pipeline wait, in clock cycles
  int32_t drop_stage;    // 0, or s > 0: the first pair's second CTA stops before its s-th stage (test)
};

// One warp writes its 32 rows x 128 bytes (32 fp32 or 64 bf16 columns) into a
// swizzled slice: row `lane`, 16-byte chunk j at position j ^ (lane % 8), the
// layout a 128-byte-swizzled TMA box of {128 bytes, 32 rows} expects.
template <bool kOutF32>
__device__ __forceinline__ void stage_row(uint32_t slice, int lane, const float* f) {
  const uint32_t row = slice + uint32_t(lane) * 128u;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t dst = row + ((uint32_t(j) ^ uint32_t(lane & 7)) << 4);
    if constexpr (kOutF32) {
      st_shared_v4(dst, __float_as_uint(f[4 * j]), __float_as_uint(f[4 * j + 1]), __float_as_uint(f[4 * j + 2]),
                   __float_as_uint(f[4 * j + 3]));
    } else {
      st_shared_v4(dst, pack_bf16x2(f[8 * j], f[8 * j + 1]), pack_bf16x2(f[8 * j + 2], f[8 * j + 3]),
                   pack_bf16x2(f[8 * j + 4], f[8 * j + 5]), pack_bf16x2(f[8 * j + 6], f[8 * j + 7]));
    }
  }
}

// Zeroes rows [valid, valid rounded up to 16) of this stage's B boxes in both
// CTAs (the rows belong to the next group or lie past m).  A row is 128
// contiguous bytes (the swizzle permutes 16-byte chunks within a row only).
// All 32 lanes of the leader's MMA warp, lanes over (row, 16-byte chunk).
__device__ __forceinline__ void zero_b_tail(uint32_t b0, int32_t valid, int lane) {
  constexpr int kB = int(B_BYTES / BOX_BYTES);
  const uint32_t b0_peer = mapa_shared(b0, 1);
  const int32_t zrows = ((valid + 15) & ~15) - valid;
  const uint32_t chunk = uint32_t(lane & 7) * 16u;
#pragma unroll
  for (int box = 0; box < kB; ++box) {
    for (int32_t zr = lane >> 3; zr < zrows; zr += 4) {
      const uint32_t off = uint32_t(box) * BOX_BYTES + uint32_t(valid + zr) * 128u + chunk;
      st_shared_v4(b0 + off, 0u, 0u, 0u, 0u);
      st_shared_cluster_v4(b0_peer + off, 0u, 0u, 0u, 0u);
    }
  }
  fence_proxy_async_smem();
  fence_proxy_async_cluster();
  __syncwarp();
}

template <bool kOutF32>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    tgmm_2sm_kernel(const __grid_constant__ CUtensorMap tm_lhs, const __grid_constant__ CUtensorMap tm_dout,
                    const __grid_constant__ CUtensorMap tm_out, const Params p) {
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
    tma_prefetch(&tm_dout);
    tma_prefetch(&tm_out);
  }
  if (warp == 1) {
    tmem_alloc_pair(sbase + OFF_TMEM, TMEM_COLS);
    tmem_relinquish_pair();
  }
  if (warp == 2) build_group_offsets(p.group_sizes, p.num_total_groups, p.m, offs, p.err);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + OFF_TMEM);

  const int32_t k_pairs = (p.k + PAIR_M - 1) / PAIR_M;
  const int32_t n_tiles = (p.n + BN - 1) / BN;
  const int32_t per_group = k_pairs * n_tiles;
  const int32_t total = p.num_local_groups * per_group;
  // Work item w covers local group g = w / per_group; its rows start at
  // loffs[g] (offsets run over all groups) and it writes out[g].
  const int32_t* loffs = offs + p.group_offset;

  uint32_t issued = 0;  // producer: stages of the pair's sequence this CTA issued (leader: armed)
  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer (both CTAs)
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int32_t w = pair; w < total && ok; w += npairs) {
        const int32_t g = w / per_group;
        const int32_t r = w - g * per_group;
        const int32_t kp = r / n_tiles, nt = r - kp * n_tiles;
        const int32_t row_begin = loffs[g], rows = loffs[g + 1] - loffs[g];
        const int32_t kc = kp * PAIR_M + int32_t(rank) * BM;        // this CTA's lhs columns
        const int32_t nc = nt * BN + int32_t(rank) * (BN / 2);      // this CTA's dout columns
        for (int32_t c = 0; c * BR < rows; ++c) {
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
          const int32_t row = row_begin + c * BR;
#pragma unroll
          for (int j = 0; j < BM / 64; ++j) tma_load_2d_pair(a_dst + j * BOX_BYTES, &tm_lhs, fb, kc + 64 * j, row);
#pragma unroll
          for (int j = 0; j < BN / 128; ++j) tma_load_2d_pair(b_dst + j * BOX_BYTES, &tm_dout, fb, nc + 64 * j, row);
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
    if (leader) {
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      // -------------------------------------------------------------- MMA issuer (leader CTA)
      constexpr uint32_t kIdesc = idesc_bf16(PAIR_M, BN, true, true);
      uint32_t acc = 0, acc_phase = 0;
      for (int32_t w = pair; w < total && ok; w += npairs) {
        const int32_t g = w / per_group;
        const int32_t rows = loffs[g + 1] - loffs[g];
        if (rows == 0) continue;  // the epilogues write zeros; no accumulator is used
        if (!wait_bar_cluster(acce_bar(acc), acc_phase ^ 1u, abort_flag, p.err, p.wait_limit)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int32_t c = 0; c * BR < rows; ++c) {
          if (!wait_bar(full_bar(stage), phase, abort_flag, p.err, p.wait_limit)) {
            ok = false;
            break;
          }
          const uint32_t a0 = sbase + OFF_A + stage * A_BYTES;
          const uint32_t b0 = sbase + OFF_B + stage * B_BYTES;
          const int32_t valid = min(BR, rows - c * BR);
          const int32_t ksteps = (valid + 15) / 16, kfull = valid / 16;
          auto issue = [&](int32_t k0, int32_t k1) {
            for (int32_t kk = k0; kk < k1; ++kk) {
              const uint64_t ad = sw128_desc(a0 + kk * 2048, BOX_BYTES, 1024);
              const uint64_t bd = sw128_desc(b0 + kk * 2048, BOX_BYTES, 1024);
              mma_bf16_ss_pair(d_tmem, ad, bd, kIdesc, (c | kk) != 0 ? 1u : 0u);
            }
          };
          tc_fence_after();
          // the 16-row blocks of this group's rows only go first; the tail block
          // is fixed up while they run
          if (lane == 0) issue(0, kfull);
          if (kfull < ksteps) {
            zero_b_tail(b0, valid, lane);
            tc_fence_after();
            if (lane == 0) issue(kfull, ksteps);
          }
          if (lane == 0) mma_commit_pair(empty_bar(stage), 0x3);
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
    constexpr int kColsPerBox = kOutF32 ? 32 : 64;  // 128 bytes of output per row
    const int quarter = warp & 3;
    const uint32_t slices = sbase + OFF_OUT + uint32_t(quarter) * 2u * SLICE_BYTES;
    uint32_t slot = 0;
    // Hands the slice `slot` to this warp: the store issued from it two boxes
    // ago has finished reading shared memory.
    auto acquire_slice = [&]() {
      if (lane == 0) tma_store_wait_read<1>();
      __syncwarp();
      return slices + slot * SLICE_BYTES;
    };
    auto release_slice = [&](int32_t col, int32_t krow0, int32_t g) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_3d_hint(&tm_out, slices + slot * SLICE_BYTES, col, krow0, g, l2_policy_evict_first());
        tma_store_commit();
      }
      slot ^= 1u;
    };
    uint32_t acc = 0, acc_phase = 0;
    for (int32_t w = pair; w < total; w += npairs) {
      const int32_t g = w / per_group;
      const int32_t r = w - g * per_group;
      const int32_t kp = r / n_tiles, nt = r - kp * n_tiles;
      const int32_t rows = loffs[g + 1] - loffs[g];
      const int32_t krow0 = kp * PAIR_M + int32_t(rank) * BM + quarter * 32;
      if (rows == 0) {
        float z[kColsPerBox];
#pragma unroll
        for (int i = 0; i < kColsPerBox; ++i) z[i] = 0.f;
        for (int c = 0; c < BN; c += kColsPerBox) {
          if (nt * BN + c >= p.n || krow0 >= p.k) break;
          stage_row<kOutF32>(acquire_slice(), lane, z);
          release_slice(nt * BN + c, krow0, g);
        }
        continue;
      }
      if (!wait_bar(accf_bar(acc), acc_phase, abort_flag, p.err, p.wait_limit)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (uint32_t(quarter * 32) << 16) + acc * BN;
#pragma unroll 1
      for (int c = 0; c < BN; c += kColsPerBox) {
        float f[kColsPerBox];
#pragma unroll
        for (int h = 0; h < kColsPerBox / 32; ++h) {
          uint32_t v[32];
          tmem_ld_32cols(tbase + c + 32 * h, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) f[32 * h + i] = __uint_as_float(v[i]);
        }
        if (c + kColsPerBox == BN) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(acce_bar(acc), 0));
        }
        if (nt * BN + c < p.n && krow0 < p.k) {
          stage_row<kOutF32>(acquire_slice(), lane, f);
          release_slice(nt * BN + c, krow0, g);
        }
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (lane == 0) tma_store_wait_all<0>();
    __syncwarp();
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

template <bool kOutF32>
cudaError_t launch_impl(const TgmmLaunch& L, int max_ctas, cudaStream_t stream) {
  auto kern = tgmm_2sm_kernel<kOutF32>;
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
  Params p{L.group_sizes, L.num_total_groups, L.group_offset, L.num_local_groups, L.m, L.n, L.k, L.out, L.err,
           L.wait_limit > 0 ? (long long)L.wait_limit : kWaitLimitCycles, L.drop_stage};
  kern<<<grid, kThreads, SMEM_BYTES, stream>>>(L.tm_lhs, L.tm_dout, L.tm_out, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tgmm_2sm(const TgmmLaunch& p, bool out_f32, int max_ctas, cudaStream_t stream) {
  return out_f32 ? launch_impl<true>(p, max_ctas, stream) : launch_impl<false>(p, max_ctas, stream);
}

}  // namespace gmmk
