// Grouped matmul with FP8 E4M3 weights, per-(group, k-block, n) fp32 scale and
// bias, on the e4m3 tensor-core path:
//   out[r, c] = sum_b s[g, b, c] * sum_{kk in block b} lhs[r, kk] * W(g, c, kk) + bias[g, c]
// (page "tpu-inference 0.12.0.dev20251213 -> 0.13.2.dev20251230", gmm.py:
// _accum scales each quant block's partial sum by rhs_scale[g, b, 0, n] and adds
// rhs_bias once; rhs_scale [G, nb, 1, n], block width k // nb).
//
// The weights never leave e4m3: TMA copies each [128 n x 128 k] tile into shared
// memory, where tcgen05.mma.kind::f8f6f4 reads it as the A operand (M = 128
// weight rows, K = 32 per instruction).  The bf16 activations are brought to
// e4m3 without losing their value: for each token row and each 128-wide k step,
// with M the largest |x| of the step and E = floor(log2 M),
//   x = 2^(E-7) * (h + l / 16),   h = rne_e4m3(x / 2^(E-7)),
//                                 l = rne_e4m3(16 * (x / 2^(E-7) - h)).
// |x / 2^(E-7)| < 256, so h never saturates.  x has 8 significant bits and h the
// top 4 of them (rounded), so x / 2^(E-7) - h is a multiple of x's last place
// below half of h's last place: at most 4 significant bits, and 16 times it lies
// in e4m3's range.  The split is exact for every x with |x| >= M * 2^-14 (where
// x / 2^(E-7) is an e4m3 normal); below that, l is rounded to a multiple of 2^-9,
// an error of at most M * 2^-21 in x.  (Here "step" is the 256-wide k step.)  h and l are B operand rows (a token's
// h in row i, its l in row T8 + i) and the products with e4m3 weights are exact,
// summed in fp32 by the tensor core.  Each step accumulates into its own TMEM
// columns; the epilogue folds it as
//   acc[i] += s[g, b, c] * 2^(E_i-7) * (D[c, i] + D[c, T8 + i] / 16).
//
// A pipeline step covers 256 k (two 128-wide sub-tiles; the last step of an
// item holds one when k / 128 is odd).  Roles (320 threads, one CTA per SM,
// persistent over items):
//   warp 0      TMA: the step's two weight boxes [128 n x 128 k] (32 KB, 4-deep
//               ring) and its bf16 token rows ({64 k, 16 rows} boxes, 2-deep
//               ring), ahead of the MMA
//   warps 6-9   split the bf16 token rows into e4m3 h / l operand rows (2-deep
//               ring; all 128 threads share any chunk size) and write each
//               row's step scale (8-deep ring)
//   warp 1      TMEM owner; per step 8 MMAs 128 x (2 T8) x 32, one accumulator
//               per sub-tile, and one commit
//   warps 2-5   per sub-tile: TMEM -> registers, fold with the token scale and
//               the sub-tile's weight-block scale into fp32 registers; per item
//               add the bias, round, store
// Items are (local group, chunk of up to 32 of its rows, 128-wide n tile); a
// chunk of t rows uses T8 = 8, 16 or 32 operand rows per half (t rounded up).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "internal.h"
#include "ptx.cuh"
#include "worklist.cuh"

namespace gmmk {
namespace {

constexpr int BMW = 128;  // weight rows (n) per item = MMA M
constexpr int BT = 32;    // token rows per item at most
constexpr int KQ = 128;   // k per weight box / operand sub-tile (128 e4m3 bytes per row)
constexpr int QPS = 2;    // sub-tiles per pipeline step
constexpr int KS = KQ * QPS;  // k per step
constexpr int AST = 4;    // weight stages in flight (2 boxes each)
constexpr int RTS = 2;    // bf16 token stages
constexpr int BST = 2;    // e4m3 token operand stages
constexpr int NSC = 8;    // token-scale slots (outlive the operand until the epilogue reads them)
constexpr int NACC = 4;   // TMEM accumulator slots, one per step
// Slot columns: sub-tile h of a step accumulates into [128 slot + 64 h, + 2 T8).
constexpr int SLOT_COLS = QPS * 2 * BT;
constexpr uint32_t TMEM_COLS = 512;
static_assert(NACC * SLOT_COLS <= int(TMEM_COLS), "TMEM map");
// One barrier per step records that the step's MMAs have completed (a single
// tcgen05.commit): it frees the step's weight stage and operand stage and
// hands its accumulator slot to the epilogue.  The weight ring, the slots and
// this ring have the same depth, so step j uses index j % NDONE in all three.
constexpr int NDONE = 4;
static_assert(AST == NDONE && NACC == NDONE && BST <= NDONE, "step-done ring indexing");
constexpr int kConvWarps = 4;
constexpr int kThreads = 192 + 32 * kConvWarps;
constexpr int kMaxGroups = 1024;

constexpr uint32_t A_BOX = BMW * KQ;         // one e4m3 weight box, 128 rows x 128 bytes
constexpr uint32_t A_BYTES = QPS * A_BOX;
constexpr uint32_t RT_STRIP = BT * 128;      // 64 k of bf16 for 32 token rows
constexpr uint32_t RT_BYTES = (KS / 64) * RT_STRIP;
constexpr uint32_t RT_BOX = 16 * 128;        // one {64 k, 16 rows} box
constexpr uint32_t B_SUB = 2 * BT * KQ;      // e4m3 operand sub-tile: 64 rows x 128 bytes
constexpr uint32_t B_BYTES = QPS * B_SUB;

constexpr uint32_t OFF_A = 0;
constexpr uint32_t OFF_RT = OFF_A + AST * A_BYTES;
constexpr uint32_t OFF_B = OFF_RT + RTS * RT_BYTES;
constexpr uint32_t OFF_SC = OFF_B + BST * B_BYTES;
constexpr uint32_t OFF_CTRL = OFF_SC + NSC * BT * 4;
constexpr uint32_t OFF_AFULL = OFF_CTRL;
constexpr uint32_t OFF_DONEB = OFF_AFULL + 8 * AST;
constexpr uint32_t OFF_RFULL = OFF_DONEB + 8 * NDONE;
constexpr uint32_t OFF_REMPTY = OFF_RFULL + 8 * RTS;
constexpr uint32_t OFF_BFULL = OFF_REMPTY + 8 * RTS;
constexpr uint32_t OFF_SFULL = OFF_BFULL + 8 * BST;
constexpr uint32_t OFF_SEMPTY = OFF_SFULL + 8 * NSC;
constexpr uint32_t OFF_ACCE = OFF_SEMPTY + 8 * NSC;
constexpr uint32_t OFF_DONE = OFF_ACCE + 8 * NACC;
constexpr uint32_t OFF_TMEM = OFF_DONE + 8;
constexpr uint32_t OFF_ABORT = OFF_TMEM + 4;
constexpr uint32_t OFF_OFFS = OFF_CTRL + 1024;
constexpr uint32_t OFF_TILES = OFF_OFFS + 4 * (kMaxGroups + 4);
constexpr uint32_t SMEM_USED = OFF_TILES + 4 * (kMaxGroups + 4);
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;
static_assert(OFF_ABORT + 4 <= OFF_OFFS, "control block overlaps the tables");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(OFF_RT % 1024 == 0 && OFF_B % 1024 == 0 && RT_BOX % 1024 == 0 && B_SUB % 1024 == 0,
              "swizzle atoms are 1024-byte aligned");

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
  int32_t zero_rest;  // zero the rows outside the local groups (gmm) or leave them (gmm_into)
};

// Operand rows per half for a chunk of t token rows.
__device__ __forceinline__ int t8_of(int32_t t) { return t <= 8 ? 8 : (t <= 16 ? 16 : 32); }

// Two fp32 -> two e4m3fn, round to nearest even; `lo` goes to the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// The two e4m3fn values in the low 16 bits of v (low byte first), exactly.
__device__ __forceinline__ float2 e4m3x2_value(uint32_t v) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(uint16_t(v)));
  return __half22float2(*reinterpret_cast<__half2*>(&h));
}

// Splits N scaled values y[0..N-1] (k order, N a multiple of 4) into their e4m3
// h and l codes, N bytes each (k order, lowest k in the lowest byte).
template <int N>
__device__ __forceinline__ void split_e4m3(const float (&y)[N], uint32_t (&hw)[N / 4], uint32_t (&lw)[N / 4]) {
#pragma unroll
  for (int j = 0; j < N / 4; ++j) {
    const uint32_t h01 = e4m3x2(y[4 * j], y[4 * j + 1]);
    const uint32_t h23 = e4m3x2(y[4 * j + 2], y[4 * j + 3]);
    const float2 v01 = e4m3x2_value(h01), v23 = e4m3x2_value(h23);
    const uint32_t l01 = e4m3x2((y[4 * j] - v01.x) * 16.f, (y[4 * j + 1] - v01.y) * 16.f);
    const uint32_t l23 = e4m3x2((y[4 * j + 2] - v23.x) * 16.f, (y[4 * j + 3] - v23.y) * 16.f);
    hw[j] = h01 | (h23 << 16);
    lw[j] = l01 | (l23 << 16);
  }
}

template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&f)[N]) {
  static_assert(N == 16 || N == 32 || N == 64, "column count");
  if constexpr (N == 16) {
    uint32_t v[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) f[i] = __uint_as_float(v[i]);
  } else {
#pragma unroll
    for (int h = 0; h < N / 32; ++h) {
      uint32_t v[32];
      tmem_ld_32cols(taddr + 32u * h, v);
#pragma unroll
      for (int i = 0; i < 32; ++i) f[32 * h + i] = __uint_as_float(v[i]);
    }
  }
}

template <bool kOutF32>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_fp8_kernel(const __grid_constant__ CUtensorMap tm_lhs, const __grid_constant__ CUtensorMap tm_rhs,
                    const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + OFF_ABORT);
  int32_t* offs = reinterpret_cast<int32_t*>(smem + OFF_OFFS);
  int32_t* tiles = reinterpret_cast<int32_t*>(smem + OFF_TILES);
  float* tscale = reinterpret_cast<float*>(smem + OFF_SC);
  auto afull_bar = [&](uint32_t s) { return sbase + OFF_AFULL + 8 * s; };
  auto stepdone_bar = [&](uint32_t s) { return sbase + OFF_DONEB + 8 * s; };
  auto rfull_bar = [&](uint32_t s) { return sbase + OFF_RFULL + 8 * s; };
  auto rempty_bar = [&](uint32_t s) { return sbase + OFF_REMPTY + 8 * s; };
  auto bfull_bar = [&](uint32_t s) { return sbase + OFF_BFULL + 8 * s; };
  auto sfull_bar = [&](uint32_t s) { return sbase + OFF_SFULL + 8 * s; };
  auto sempty_bar = [&](uint32_t s) { return sbase + OFF_SEMPTY + 8 * s; };
  auto acce_bar = [&](uint32_t s) { return sbase + OFF_ACCE + 8 * s; };
  const uint32_t done_bar = sbase + OFF_DONE;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < AST; ++s) mbar_init(afull_bar(s), 1);
    for (int s = 0; s < NDONE; ++s) mbar_init(stepdone_bar(s), 1);
    for (int s = 0; s < RTS; ++s) {
      mbar_init(rfull_bar(s), 1);
      mbar_init(rempty_bar(s), kConvWarps);
    }
    for (int s = 0; s < BST; ++s) mbar_init(bfull_bar(s), kConvWarps);
    for (int s = 0; s < NSC; ++s) {
      mbar_init(sfull_bar(s), kConvWarps);
      mbar_init(sempty_bar(s), 4);
    }
    for (int s = 0; s < NACC; ++s) mbar_init(acce_bar(s), 4);
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

  const int32_t t_tiles = tiles[p.num_local_groups];  // row chunks over all local groups
  const int32_t n_tiles = (p.n + BMW - 1) / BMW;
  const int32_t nq = p.k / KQ;                         // 128-wide sub-tiles (k % 128 == 0 on this path)
  const int32_t ksteps = (nq + QPS - 1) / QPS;         // the last step may hold one sub-tile
  const int32_t nb = p.scale != nullptr ? p.num_blocks : 1;
  const int32_t q_per_block = nq / nb;                 // (k / nb) % 128 == 0 on this path
  const int32_t total = t_tiles * n_tiles;
  // Items: row chunks outer, the weight tiles of the chunk's group inner.
  auto item_of = [&](int32_t w) {
    return decode_gemm_tile(w, t_tiles, n_tiles, n_tiles, tiles, offs, p.group_offset, p.num_local_groups, BT);
  };
  auto halves = [&](int32_t ks) { return min(QPS, nq - QPS * ks); };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      uint32_t as = 0, aph = 0, rs = 0, rph = 0, apend = 0, rpend = 0;
      uint32_t apar[AST], rpar[RTS];
      bool ok = true;
      for (int32_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
        const GemmTile t = item_of(w);
        const int32_t rboxes = t.row_end - t.row0 > 16 ? 2 : 1;
        for (int32_t ks = 0; ks < ksteps; ++ks) {
          const int32_t hq = halves(ks);
          // weight stage `as` was last read by the step NDONE before: index as, previous phase
          if (!wait_bar(stepdone_bar(as), aph ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(afull_bar(as), uint32_t(hq) * A_BOX);
          for (int h = 0; h < hq; ++h)
            tma_load_3d(sbase + OFF_A + as * A_BYTES + h * A_BOX, &tm_rhs, afull_bar(as), (QPS * ks + h) * KQ,
                        t.n_tile * BMW, t.local_group);
          apar[as] = aph;
          apend |= 1u << as;
          if (++as == AST) {
            as = 0;
            aph ^= 1u;
          }
          if (!wait_bar(rempty_bar(rs), rph ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(rfull_bar(rs), uint32_t(rboxes * 2 * hq) * RT_BOX);
          for (int st = 0; st < 2 * hq; ++st)
            for (int rb = 0; rb < rboxes; ++rb)
              tma_load_2d(sbase + OFF_RT + rs * RT_BYTES + st * RT_STRIP + rb * RT_BOX, &tm_lhs, rfull_bar(rs),
                          ks * KS + 64 * st, t.row0 + 16 * rb);
          rpar[rs] = rph;
          rpend |= 1u << rs;
          if (++rs == RTS) {
            rs = 0;
            rph ^= 1u;
          }
        }
      }
      if (!ok) {
        for (int s = 0; s < AST; ++s)
          if (apend >> s & 1u) drain_bar(afull_bar(s), apar[s]);
        for (int s = 0; s < RTS; ++s)
          if (rpend >> s & 1u) drain_bar(rfull_bar(s), rpar[s]);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    // Step j of the CTA accumulates sub-tile h into TMEM columns
    // [128 slot + 64 h, + 2 T8) of slot j % NACC; the epilogue frees the slot
    // after reading it.  as == slot == j % NDONE throughout.
    uint32_t as = 0, aph = 0, bs = 0, bph = 0, slot = 0, sph = 0;
    bool ok = true;
    for (int32_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
      const GemmTile t = item_of(w);
      const int t8 = t8_of(t.row_end - t.row0);
      const uint32_t idesc = idesc_e4m3(BMW, 2 * t8);
      for (int32_t ks = 0; ks < ksteps; ++ks) {
        const int32_t hq = halves(ks);
        if (!wait_bar(acce_bar(slot), sph ^ 1u, abort_flag, p.err) ||
            !wait_bar(afull_bar(as), aph, abort_flag, p.err) || !wait_bar(bfull_bar(bs), bph, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          for (int h = 0; h < hq; ++h) {
            const uint32_t a0 = sbase + OFF_A + as * A_BYTES + h * A_BOX;
            const uint32_t b0 = sbase + OFF_B + bs * B_BYTES + h * B_SUB;
            const uint32_t d = tmem_base + slot * SLOT_COLS + uint32_t(h) * (2 * BT);
#pragma unroll
            for (int kk = 0; kk < KQ / 32; ++kk)
              mma_e4m3_ss(d, sw128_desc(a0 + 32 * kk, 16, 1024), sw128_desc(b0 + 32 * kk, 16, 1024), idesc,
                          kk != 0 ? 1u : 0u);
          }
          mma_commit(stepdone_bar(slot));
        }
        __syncwarp();
        if (++as == AST) {
          as = 0;
          aph ^= 1u;
        }
        if (++bs == BST) {
          bs = 0;
          bph ^= 1u;
        }
        if (++slot == NACC) {
          slot = 0;
          sph ^= 1u;
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
    // Per sub-tile q of the item (block q / q_per_block): read its 2 T8
    // accumulator columns and fold them with the block's weight scale for this
    // lane's column and the step's token scales.
    const int quarter = warp & 3;
    const int wrow = quarter * 32 + lane;  // weight row in the tile = output column
    const uint32_t lane_base = uint32_t(quarter * 32) << 16;
    uint32_t slot = 0, sph = 0, sc = 0, scph = 0;
    bool ok = true;
    constexpr int kPre = 8;  // weight scales are first-touch DRAM reads: fetched 8 blocks ahead
    for (int32_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
      const GemmTile t = item_of(w);
      const int32_t col = t.n_tile * BMW + wrow;
      const bool col_ok = col < p.n;
      const float* srow = p.scale != nullptr ? p.scale + int64_t(t.local_group) * nb * p.n + col : nullptr;
      auto load_scales = [&](int32_t b0, float (&dst)[kPre]) {
#pragma unroll
        for (int j = 0; j < kPre; ++j)
          dst[j] = (srow != nullptr && col_ok && b0 + j < nb) ? __ldg(srow + int64_t(b0 + j) * p.n) : 1.f;
      };
      float bias = 0.f;
      if (p.bias != nullptr && col_ok) {
        const int64_t bi = int64_t(t.local_group) * p.n + col;
        bias = p.bias_f32 ? __ldg(static_cast<const float*>(p.bias) + bi)
                          : __bfloat162float(static_cast<const __nv_bfloat16*>(p.bias)[bi]);
      }
      auto run = [&](auto t8c) {
        constexpr int T8 = decltype(t8c)::value;
        float acc[T8];
#pragma unroll
        for (int i = 0; i < T8; ++i) acc[i] = 0.f;
        float s_cur[kPre], s_next[kPre];
        load_scales(0, s_cur);
        int32_t q = 0;
        for (int32_t c0 = 0; c0 < nb && ok; c0 += kPre) {
          load_scales(c0 + kPre, s_next);
#pragma unroll
          for (int bi = 0; bi < kPre; ++bi) {
            if (c0 + bi >= nb || !ok) break;
            const float sw = s_cur[bi];
            for (int32_t qq = 0; qq < q_per_block; ++qq) {
              const int h = q % QPS;
              if (h == 0) {
                if (!wait_bar(stepdone_bar(slot), sph, abort_flag, p.err) ||
                    !wait_bar(sfull_bar(sc), scph, abort_flag, p.err)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
              }
              float d[2 * T8];
              tmem_ld_cols<2 * T8>(tmem_base + lane_base + slot * SLOT_COLS + uint32_t(h) * (2 * BT), d);
              const float* ts = tscale + sc * BT;
#pragma unroll
              for (int i = 0; i < T8; ++i) acc[i] = fmaf(sw * ts[i], fmaf(d[T8 + i], 0.0625f, d[i]), acc[i]);
              ++q;
              if (h == QPS - 1 || q == nq) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                  mbar_arrive(acce_bar(slot));
                  mbar_arrive(sempty_bar(sc));
                }
                if (++slot == NACC) {
                  slot = 0;
                  sph ^= 1u;
                }
                if (++sc == NSC) {
                  sc = 0;
                  scph ^= 1u;
                }
              }
            }
          }
#pragma unroll
          for (int j = 0; j < kPre; ++j) s_cur[j] = s_next[j];
        }
        if (!ok || !col_ok) return;
#pragma unroll
        for (int i = 0; i < T8; ++i) {
          const int32_t row = t.row0 + i;
          if (row < t.row_end) {
            const float r = acc[i] + bias;
            if constexpr (kOutF32)
              static_cast<float*>(p.out)[int64_t(row) * p.n + col] = r;
            else
              static_cast<__nv_bfloat16*>(p.out)[int64_t(row) * p.n + col] = __float2bfloat16_rn(r);
          }
        }
      };
      const int t8 = t8_of(t.row_end - t.row0);
      if (t8 == 8)
        run(std::integral_constant<int, 8>{});
      else if (t8 == 16)
        run(std::integral_constant<int, 16>{});
      else
        run(std::integral_constant<int, 32>{});
    }
    // Rows outside [offs[first local], offs[last local + 1]) are zero, unless the
    // caller keeps them (gmm_into).
    if (p.zero_rest) {
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
    }
  } else {
    // ---------------------------------------------------------------- token split
    // The 128 threads share a step's T8 rows evenly: 128 / T8 adjacent lanes per
    // token row r, each taking the same T8 consecutive k of every sub-tile h of
    // the step (T8 / 8 bf16 chunks of 16 bytes per sub-tile from the token tile;
    // T8 bytes of e4m3 into rows r (h part) and T8 + r (l part) of operand
    // sub-tile h).  The lanes of a row agree on the row's step maximum by
    // shuffles.  All tiles are 128-byte swizzled: 16-byte chunk j of row r sits
    // at position j ^ (r % 8).
    const int ct = int(threadIdx.x) - 192;
    uint32_t rs = 0, rph = 0, bs = 0, sc = 0, scph = 0;
    uint32_t j = 0;  // steps converted so far; operand stage bs was last read by step j - BST
    bool ok = true;
    for (int32_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
      const GemmTile t = item_of(w);
      auto run = [&](auto t8c) {
        constexpr int T8 = decltype(t8c)::value;
        constexpr int TPR = 128 / T8;  // threads per token row: 16, 8 or 4
        const int r = ct / TPR, seg = ct % TPR;
        for (int32_t ks = 0; ks < ksteps; ++ks) {
          const int32_t hq = halves(ks);
          if (!wait_bar(rfull_bar(rs), rph, abort_flag, p.err) ||
              (j >= uint32_t(BST) &&
               !wait_bar(stepdone_bar((j - BST) % NDONE), ((j - BST) / NDONE) & 1u, abort_flag, p.err)) ||
              !wait_bar(sempty_bar(sc), scph ^ 1u, abort_flag, p.err)) {
            ok = false;
            return;
          }
          // Sub-tile h, k [T8 seg, T8 seg + T8): bf16 chunks c = T8 seg / 8 + i of
          // the sub-tile, in strip 2 h + c / 8 of the token tile at position c % 8.
          uint32_t xw[QPS][T8 / 2];
          uint32_t amax = 0;
          const uint32_t src = sbase + OFF_RT + rs * RT_BYTES + uint32_t(r) * 128u;
#pragma unroll
          for (int h = 0; h < QPS; ++h) {
            if (h < hq) {
#pragma unroll
              for (int i = 0; i < T8 / 8; ++i) {
                const int c = seg * (T8 / 8) + i;
                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(xw[h][4 * i]), "=r"(xw[h][4 * i + 1]), "=r"(xw[h][4 * i + 2]),
                               "=r"(xw[h][4 * i + 3])
                             : "r"(src + uint32_t(2 * h + (c >> 3)) * RT_STRIP +
                                   (uint32_t((c & 7) ^ (r & 7)) << 4)));
              }
#pragma unroll
              for (int i = 0; i < T8 / 2; ++i)
                amax = max(amax, max((xw[h][i] << 16) & 0x7FFFFFFFu, xw[h][i] & 0x7FFF0000u));
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(rempty_bar(rs));  // the values are in registers
#pragma unroll
          for (int dd = 1; dd < TPR; dd <<= 1) amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, dd));
          // E + 127 of the step maximum, kept in [8, 254] so that both 2^(E-7)
          // and 2^(7-E) are fp32 normals; a NaN or infinity gives a NaN scale.
          const uint32_t e = min(max(amax >> 23, 8u), 254u);
          const float inv_s = __uint_as_float((261u - e) << 23);
#pragma unroll
          for (int h = 0; h < QPS; ++h) {
            if (h < hq) {
              float y[T8];
#pragma unroll
              for (int i = 0; i < T8 / 2; ++i) {
                y[2 * i] = __uint_as_float(xw[h][i] << 16) * inv_s;
                y[2 * i + 1] = __uint_as_float(xw[h][i] & 0xFFFF0000u) * inv_s;
              }
              uint32_t hw[T8 / 4], lw[T8 / 4];
              split_e4m3<T8>(y, hw, lw);
              // e4m3 bytes [T8 seg, T8 seg + T8) of the row: 16-byte chunk
              // (T8 seg) / 16, at byte (T8 seg) % 16 within it.
              const uint32_t sub = sbase + OFF_B + bs * B_BYTES + uint32_t(h) * B_SUB;
              const uint32_t hrow = sub + uint32_t(r) * 128u, lrow = sub + uint32_t(T8 + r) * 128u;
              if constexpr (T8 == 8) {
                const uint32_t pos = (uint32_t((seg >> 1) ^ (r & 7)) << 4) + uint32_t(seg & 1) * 8u;
                asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(hrow + pos), "r"(hw[0]), "r"(hw[1]));
                asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(lrow + pos), "r"(lw[0]), "r"(lw[1]));
              } else {
#pragma unroll
                for (int cc = 0; cc < T8 / 16; ++cc) {
                  const uint32_t pos = uint32_t((seg * (T8 / 16) + cc) ^ (r & 7)) << 4;
                  st_shared_v4(hrow + pos, hw[4 * cc], hw[4 * cc + 1], hw[4 * cc + 2], hw[4 * cc + 3]);
                  st_shared_v4(lrow + pos, lw[4 * cc], lw[4 * cc + 1], lw[4 * cc + 2], lw[4 * cc + 3]);
                }
              }
            }
          }
          if (seg == 0)
            tscale[sc * BT + r] = amax < 0x7F800000u ? __uint_as_float((e - 7u) << 23) : __uint_as_float(0x7FC00000u);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(bfull_bar(bs));
            mbar_arrive(sfull_bar(sc));
          }
          if (++rs == RTS) {
            rs = 0;
            rph ^= 1u;
          }
          if (++bs == BST) bs = 0;
          if (++sc == NSC) {
            sc = 0;
            scph ^= 1u;
          }
          ++j;
        }
      };
      const int t8 = t8_of(t.row_end - t.row0);
      if (t8 == 8)
        run(std::integral_constant<int, 8>{});
      else if (t8 == 16)
        run(std::integral_constant<int, 16>{});
      else
        run(std::integral_constant<int, 32>{});
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

template <bool kOutF32>
cudaError_t launch_impl(const ScaledLaunch& L, int grid, cudaStream_t stream) {
  auto kern = gemm_fp8_kernel<kOutF32>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(SMEM_BYTES));
  if (e != cudaSuccess) return e;
  Params p{L.group_sizes, L.num_total_groups, L.group_offset, L.num_local_groups, L.m, L.n, L.k, L.scale,
           L.num_blocks, L.bias, L.bias_f32, L.out, L.err, L.zero_rest};
  kern<<<grid, kThreads, SMEM_BYTES, stream>>>(L.tm_lhs, L.tm_rhs, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fp8(const ScaledLaunch& p, bool out_f32, int grid, cudaStream_t stream) {
  return out_f32 ? launch_impl<true>(p, grid, stream) : launch_impl<false>(p, grid, stream);
}

}  // namespace gmmk
