// Backward weight gradient per group: out[g] = lhs_g^T @ dout_g.
//
// For every local group g (page "Megablox: transposed-RHS gmm_v2 kernel for
// the backward dlhs", Context: the drhs of the grouped matmul; page
// "tpu-inference ...", gmm.py make_group_metadata: empty groups are still
// visited so that their output is zeroed, and start_group / num_nonzero_groups
// pick the slice of groups a shard computes):
//   out[g, kk, c] = sum_{r in group group_offset + g} lhs[r, kk] * dout[r, c].
// Group offsets run over all num_total_groups sizes, so rows of the groups
// before the slice are skipped.
// The contraction runs over the group's rows.  Both operands are read in
// place from their row-major [rows, features] layout as MN-major tcgen05
// operands (A = lhs_g^T: 128 lhs columns x 64 rows; B = dout_g: 256 dout
// columns x 64 rows).  The last row chunk of a group may run into the next
// group's rows; the MMA warp zeroes those rows in shared memory (both
// operands) before issuing, so no other group's data enters the sum.
//
// Same CTA shape as the forward kernel: warp 0 TMA, warp 1 TMEM + MMA,
// warps 2-5 epilogue.  The output (fp32 [G, k, n] by default) is the bulk of
// the bytes, so each epilogue warp stages its 32 rows x 128 bytes of the tile
// in a 128-byte-swizzled shared-memory slice (two per warp, alternating) and
// writes it with a TMA bulk tensor store; the TMA clips the k and n tails.
// Empty groups' tiles are written as zeros the same way, without TMEM.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "worklist.cuh"

namespace gmmk {
namespace {

constexpr int BM = 128;  // output rows (lhs columns)
constexpr int BN = 256;  // output columns (dout columns)
constexpr int BR = 64;   // contraction rows per stage
constexpr int STAGES = 3;
constexpr int kThreads = 192;
constexpr int kMaxGroups = 1024;
constexpr uint32_t BOX_BYTES = 64 * 64 * 2;  // one 64-feature x 64-row box
constexpr uint32_t A_BYTES = (BM / 64) * BOX_BYTES;
constexpr uint32_t B_BYTES = (BN / 64) * BOX_BYTES;
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
constexpr uint32_t OFF_OFFS = OFF_CTRL + 256;
constexpr uint32_t SMEM_USED = OFF_OFFS + 4 * (kMaxGroups + 4);
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

struct Params {
  const int32_t* group_sizes;
  int32_t num_total_groups, group_offset, num_local_groups;
  int32_t m, n, k;
  void* out;
  uint32_t* err;
  int32_t lhs_3d, dout_3d;  // tm_lhs / tm_dout are the [features / 64, rows, 64] views
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

template <bool kOutF32>
__global__ void __launch_bounds__(kThreads, 1)
    tgmm_kernel(const __grid_constant__ CUtensorMap tm_lhs, const __grid_constant__ CUtensorMap tm_dout,
                const __grid_constant__ CUtensorMap tm_out, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + OFF_ABORT);
  int32_t* offs = reinterpret_cast<int32_t*>(smem + OFF_OFFS);
  auto full_bar = [&](uint32_t s) { return sbase + OFF_FULL + 8 * s; };
  auto empty_bar = [&](uint32_t s) { return sbase + OFF_EMPTY + 8 * s; };
  auto accf_bar = [&](uint32_t b) { return sbase + OFF_ACCF + 8 * b; };
  auto acce_bar = [&](uint32_t b) { return sbase + OFF_ACCE + 8 * b; };
  const uint32_t done_bar = sbase + OFF_DONE;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), 128);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch(&tm_lhs);
    tma_prefetch(&tm_dout);
    tma_prefetch(&tm_out);
  }
  if (warp == 1) {
    tmem_alloc(sbase + OFF_TMEM, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 2) build_group_offsets(p.group_sizes, p.num_total_groups, p.m, offs, p.err);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + OFF_TMEM);

  const int32_t k_tiles = (p.k + BM - 1) / BM;
  const int32_t n_tiles = (p.n + BN - 1) / BN;
  const int32_t per_group = k_tiles * n_tiles;
  const int32_t total = p.num_local_groups * per_group;
  // Work item w covers local group g = w / per_group; its rows start at
  // loffs[g] (offsets run over all groups) and it writes out[g].
  const int32_t* loffs = offs + p.group_offset;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, pend_mask = 0;
      uint32_t pend_par[STAGES];
      bool ok = true;
      for (int32_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
        const int32_t g = w / per_group;
        const int32_t r = w - g * per_group;
        const int32_t kt = r / n_tiles, nt = r - kt * n_tiles;
        const int32_t row_begin = loffs[g], rows = loffs[g + 1] - loffs[g];
        for (int32_t c = 0; c * BR < rows; ++c) {
          if (!wait_bar(empty_bar(stage), phase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, STAGE_BYTES);
          const uint32_t a_dst = sbase + OFF_A + stage * A_BYTES;
          const uint32_t b_dst = sbase + OFF_B + stage * B_BYTES;
          const int32_t row = row_begin + c * BR;
          // one copy per operand where the shapes allow it: a thread's copy
          // issue, not the bytes, paced this loop with six boxes a chunk
          if (p.lhs_3d) {
            tma_load_3d(a_dst, &tm_lhs, fb, 0, row, kt * (BM / 64));
          } else {
#pragma unroll
            for (int j = 0; j < BM / 64; ++j) tma_load_2d(a_dst + j * BOX_BYTES, &tm_lhs, fb, kt * BM + 64 * j, row);
          }
          if (p.dout_3d) {
            tma_load_3d(b_dst, &tm_dout, fb, 0, row, nt * (BN / 64));
          } else {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j) tma_load_2d(b_dst + j * BOX_BYTES, &tm_dout, fb, nt * BN + 64 * j, row);
          }
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
    constexpr uint32_t kIdesc = idesc_bf16(BM, BN, true, true);
    uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
    bool ok = true;
    for (int32_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
      const int32_t g = w / per_group;
      const int32_t rows = loffs[g + 1] - loffs[g];
      if (rows == 0) continue;  // the epilogue writes zeros; no accumulator is used
      if (!wait_bar(acce_bar(acc), acc_phase ^ 1u, abort_flag, p.err)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      for (int32_t c = 0; c * BR < rows; ++c) {
        if (!wait_bar(full_bar(stage), phase, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = sbase + OFF_A + stage * A_BYTES;
        const uint32_t b0 = sbase + OFF_B + stage * B_BYTES;
        const int32_t valid = min(BR, rows - c * BR);
        const int32_t ksteps = (valid + 15) / 16, kfull = valid / 16;
        auto issue = [&](int32_t k0, int32_t k1) {
          for (int32_t kk = k0; kk < k1; ++kk) {
            const uint64_t ad = sw128_desc(a0 + kk * 2048, BOX_BYTES, 1024);
            const uint64_t bd = sw128_desc(b0 + kk * 2048, BOX_BYTES, 1024);
            mma_bf16_ss(d_tmem, ad, bd, kIdesc, (c | kk) != 0 ? 1u : 0u);
          }
        };
        // The 16-row blocks that hold only this group's rows go to the tensor
        // core first; the tail block is fixed up while they run.
        if (lane == 0) issue(0, kfull);
        if (kfull < ksteps) {
          // Rows [valid, 16 ksteps) belong to the next group (or lie past m):
          // zero them in all six boxes, lanes over (row, 16-byte chunk).  A row
          // is 128 contiguous bytes (the swizzle permutes chunks within a row).
          const int32_t zrows = 16 * ksteps - valid;
          const uint32_t chunk = uint32_t(lane & 7) * 16u;
#pragma unroll
          for (int box = 0; box < 6; ++box) {
            const uint32_t base = box < 2 ? a0 + box * BOX_BYTES : b0 + (box - 2) * BOX_BYTES;
            for (int32_t zr = lane >> 3; zr < zrows; zr += 4)
              st_shared_v4(base + uint32_t(valid + zr) * 128u + chunk, 0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) issue(kfull, ksteps);
        }
        if (lane == 0) mma_commit(empty_bar(stage));
        __syncwarp();
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (lane == 0) mma_commit(accf_bar(acc));
      __syncwarp();
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (lane == 0) {
      mma_commit(done_bar);
      drain_bar(done_bar, 0);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- epilogue
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
    for (int32_t w = blockIdx.x; w < total; w += gridDim.x) {
      const int32_t g = w / per_group;
      const int32_t r = w - g * per_group;
      const int32_t kt = r / n_tiles, nt = r - kt * n_tiles;
      const int32_t rows = loffs[g + 1] - loffs[g];
      const int32_t krow0 = kt * BM + quarter * 32;
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
      if (!wait_bar(accf_bar(acc), acc_phase, abort_flag, p.err)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (uint32_t(quarter * 32) << 16) + acc * BN;
      // The BN columns in 32-column pieces, two register buffers: the load of
      // piece q + 1 is in flight while piece q is staged and stored.
      constexpr int kPieces = BN / 32, kPerBox = kColsPerBox / 32;
      uint32_t buf[2][32];
      tmem_ld_32cols_async(tbase, buf[0]);
      tmem_wait_ld(buf[0]);
      float f[kColsPerBox];
#pragma unroll
      for (int q = 0; q < kPieces; ++q) {
        if (q + 1 < kPieces) tmem_ld_32cols_async(tbase + 32 * (q + 1), buf[(q + 1) & 1]);
#pragma unroll
        for (int i = 0; i < 32; ++i) f[32 * (q % kPerBox) + i] = __uint_as_float(buf[q & 1][i]);
        if ((q + 1) % kPerBox == 0) {
          const int c = (q + 1 - kPerBox) * 32;
          if (nt * BN + c < p.n && krow0 < p.k) {
            stage_row<kOutF32>(acquire_slice(), lane, f);
            release_slice(nt * BN + c, krow0, g);
          }
        }
        if (q + 1 < kPieces) tmem_wait_ld(buf[(q + 1) & 1]);
        if (q + 2 == kPieces) {
          // every column is in registers: the accumulator can take the next tile
          tc_fence_before();
          mbar_arrive(acce_bar(acc));
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
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

template <bool kOutF32>
cudaError_t launch_impl(const TgmmLaunch& L, int grid, cudaStream_t stream) {
  auto kern = tgmm_kernel<kOutF32>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(SMEM_BYTES));
  if (e != cudaSuccess) return e;
  Params p{L.group_sizes, L.num_total_groups, L.group_offset, L.num_local_groups, L.m, L.n, L.k, L.out, L.err,
           L.lhs_3d, L.dout_3d};
  kern<<<grid, kThreads, SMEM_BYTES, stream>>>(L.tm_lhs, L.tm_dout, L.tm_out, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tgmm(const TgmmLaunch& p, bool out_f32, int grid, cudaStream_t stream) {
  return out_f32 ? launch_impl<true>(p, grid, stream) : launch_impl<false>(p, grid, stream);
}

}  // namespace gmmk
