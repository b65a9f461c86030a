// Grouped matmul with 8- and 4-bit weights (e4m3fn, e5m2, int8, int4, uint4,
// e2m1), per-(group, k-block, n) fp32 scale and bias, on the fp8 tensor cores:
//   out[r, c] = sum_b s[g, b, c] * sum_{kk in block b} lhs[r, kk] * W(g, c, kk) + bias[g, c]
// (page "tpu-inference 0.12.0.dev20251213 -> 0.13.2.dev20251230", gmm.py:
// _accum scales each quant block's partial sum by rhs_scale[g, b, 0, n] and adds
// rhs_bias once; rhs_scale [G, nb, 1, n], block width k // nb; common.py lists
// the operand formats).
//
// Weights.  tcgen05.mma.kind::f8f6f4 reads a [128 n x 128 k] weight tile from
// shared memory as its A operand (M = 128 weight rows, K = 32 per instruction).
// e4m3, e5m2 and e2m1 tiles are used as TMA copies them (e2m1 through a tensor
// map that spreads each 16 packed codes over 16 bytes, the 4-bit operand
// layout of kind::f8f6f4).  int4, uint4 and int8 are rewritten as e4m3 tiles
// by 4 weight-converter warps, exactly: every int4 and uint4 value is an e4m3
// value, and an int8 w is 16 h + l with h its signed high nibble and l its
// unsigned low nibble, where 16 h and l are e4m3 values, so an int8 tile
// becomes two A tiles whose MMAs add into one accumulator.  The 4-bit formats
// hold two values per byte, the even k in the low nibble.
//
// Activations.  The pages multiply bf16 activations by the weights with exact
// products and fp32 sums (gmm.py, _accum: dot_general with an f32 result).
// Here each bf16 row is brought to e4m3 without losing its value, per token row
// and pipeline step (split_step): with M1 the largest |x| of the row's step and
// E1 = floor(log2 M1),
//   x = 2^(E1-7) * (h + l / 16) + r,   h = rne_e4m3(x / 2^(E1-7)),
//                                      l = rne_e4m3(16 * (x / 2^(E1-7) - h)).
// |x / 2^(E1-7)| < 256, so h never saturates.  x has 8 significant bits and h the
// top 4 of them (rounded), so x / 2^(E1-7) - h is a multiple of x's last place
// below half of h's last place: at most 4 significant bits, and 16 times it lies
// in e4m3's range.  So r = 0 for every x with |x| >= 2^(E1-13), where
// x / 2^(E1-7) is an e4m3 normal: every x within 2^13 of M1.  Smaller values
// leave a rest r (|r| <= 2^(E1-21)), which a second level splits the same way
// with its own largest magnitude M2: r = 2^(E2-7) * (h2 + l2 / 16) + r2.  The two
// levels hold every step whose magnitudes lie within two such ranges (a few
// large values beside small ones, the case one level gets wrong); a step that
// leaves r2 != 0, or holds an infinity or a NaN, marks its row, and the last
// CTA to finish computes that row's outputs again from the stored values
// (fix_marked_rows).  h, l, h2 and l2 are B operand rows (chunk row 8 b + i in
// rows 32 b + i, + 8, + 16, + 24); their products with the weights are exact
// and the tensor core sums them in fp32.  Each 128-wide sub-tile accumulates
// into its own TMEM columns, and the epilogue folds it as
//   acc[i] += s[g, b, c] * (s1_i * (D_h + D_l / 16) + s2_i * (D_h2 + D_l2 / 16)),
// reading the h2 / l2 columns only in steps where some row has a second level.
//
// Pipeline (one CTA per SM, persistent over items).  A step covers QPS
// sub-tiles (2, i.e. 256 k; 1 for int8, whose tiles are twice the MMA work);
// the last step of an item may hold fewer.  Roles:
//   warp 0      TMA: the step's raw weight boxes (4-deep ring) and its bf16
//               token rows ({64 k, 16 rows} boxes, 2-deep ring); with e4m3
//               activations the e4m3 token rows ({128 k, 16 rows} boxes)
//               straight into a 4-deep operand ring; with split activations
//               (below) their h, l, h2 and l2 rows ({128 k, 8 rows, 4 planes}
//               boxes) likewise
//   warps 6-9   split the bf16 token rows into e4m3 h / l / h2 / l2 operand
//               rows (2-deep ring; all 128 threads share any chunk size) and
//               write each row's step scales (8-deep ring); with e4m3
//               activations warp 6 alone writes each sub-tile's token scales
//   next 4 or 8 (int8, int4, uint4) rewrite raw weight tiles as e4m3 A tiles
//               (2-deep ring): one weight row per thread, or half a row with
//               e4m3 activations (8 warps)
//   warp 1      TMEM owner; per step 4 MMAs 128 x N x 32 per A tile (N = 4 T8
//               split rows, or 16 / 32 e4m3 token rows), one accumulator per
//               sub-tile, and one commit into a step-done ring
//   warps 2-5   per sub-tile: TMEM -> registers, fold with the token scales and
//               the sub-tile's weight-block scale into fp32 registers; per item
//               add the bias, round, store
// Items are (local group, chunk of up to BT of its rows, 128-wide n tile), BT =
// 16 with bf16 activations and 32 with e4m3 ones; a chunk of t rows uses T8 =
// 8, 16 or 32 operand rows per term (t rounded up).
//
// Split activations (kPS).  The same split of the bf16 rows can be made once
// per row by act_split.cu, instead of once per row and n tile here: the h, l,
// h2 and l2 codes of every row in four e4m3 planes and each row's (s1, s2) per
// step.  The kernel then loads each 8 chunk rows' four terms with one box into
// the operand layout the token split writes, and takes the step scales through
// the token-scale warp; the MMAs and the fold are those of the bf16 path, so
// both give the same bits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "internal.h"
#include "ptx.cuh"
#include "worklist.cuh"

namespace gmmk {
namespace fp8 {

enum class WFmt : int { kE4M3 = 0, kE5M2 = 1, kInt8 = 2, kInt4 = 3, kUint4 = 4, kE2M1 = 5 };

constexpr int BMW = 128;  // weight rows (n) per item = MMA M
constexpr int KQ = 128;   // k per sub-tile (one e4m3 A tile row is 128 bytes)
constexpr uint32_t TMEM_COLS = 512;
constexpr int kMaxGroups = 1024;
constexpr uint32_t A_SUB = BMW * KQ;     // one e4m3 A tile: 128 rows x 128 bytes
constexpr uint32_t RAW_BOX = BMW * 128;  // one raw weight box: 128 rows x 128 bytes
constexpr uint32_t RT_BOX = 16 * 128;    // one {64 k, 16 rows} bf16 or {128 k, 16 rows} e4m3 box
constexpr int SUB_COLS = 64;             // TMEM columns of one sub-tile's accumulator

// kA8: the token operand comes by TMA (e4m3 activations, or with kPS the
// split activations) and warp 6 writes its scales.
template <WFmt F, bool kA8, bool kPS = false>
struct Cfg {
  static_assert(kA8 || !kPS, "split activations come by TMA");
  // bf16 activations, split in the kernel or by the split pass: each chunk row
  // becomes four e4m3 operand rows (h, l, h2, l2)
  static constexpr bool kSplit = !kA8 || kPS;
  static constexpr int BT = kSplit ? 16 : 32;  // token rows per item at most
  static constexpr uint32_t RT_STRIP = BT * 128;  // 64 k of bf16 for BT token rows
  static constexpr bool kNibble = F == WFmt::kInt4 || F == WFmt::kUint4;  // 4-bit codes rewritten as e4m3
  static constexpr bool kConv = kNibble || F == WFmt::kInt8;              // weights rewritten in shared memory
  static constexpr int QPS = F == WFmt::kInt8 ? 1 : 2;        // sub-tiles per step
  static constexpr int KS = KQ * QPS;                         // k per step
  static constexpr int PASSES = F == WFmt::kInt8 ? 2 : 1;     // A tiles per sub-tile
  // kind::f8f6f4 type of A: e4m3 0, e5m2 1, e2m1 5
  static constexpr uint32_t kAType = F == WFmt::kE5M2 ? 1u : (F == WFmt::kE2M1 ? 5u : 0u);
  // Bytes a raw box brings from global memory: e2m1 boxes hold 128 k of packed
  // codes (64 bytes a row) that the TMA spreads over 128-byte rows, each 8
  // bytes of codes followed by an 8-byte gap (the layout kind::f8f6f4 reads
  // 4-bit operands in); the transaction count is the packed bytes.
  static constexpr uint32_t RAW_TX = F == WFmt::kE2M1 ? RAW_BOX / 2 : RAW_BOX;
  // A raw box holds 128 bytes per row: 128 k of an 8-bit format, 256 k of a 4-bit one.
  static constexpr int RAW_BOXES = kNibble ? 1 : QPS;
  static constexpr uint32_t RAW_BYTES = RAW_BOXES * RAW_BOX;
  static constexpr int RAWST = 4;
  static constexpr int CST = kConv ? 2 : 0;
  static constexpr uint32_t CONV_BYTES = QPS * PASSES * A_SUB;
  static constexpr int NACC = QPS == 2 ? 4 : 8;  // TMEM accumulator slots, one per step
  // e4m3 activations (kA8) come by TMA straight into the operand ring, which is
  // then freed through the step-done ring; bf16 ones pass the token split.
  static constexpr int RTS = kA8 ? 0 : 2, BST = kA8 ? 4 : 2, NSC = 8;
  // token scales per step: (s1, s2) per row with split activations, then four
  // words that are non-zero when some row of the chunk has a second level in
  // the step (one per split warp; with split activations only the first);
  // one scale per sub-tile and row with e4m3 activations
  static constexpr int SC_TOK = kSplit ? 2 * BT + 4 : QPS * BT;
  // then the weight scales of the step's (at most two) quant blocks for the
  // item's 128 columns, as stored (f32, or E8M0 bytes), one 512-byte row per
  // block: the epilogue reads them from here, not from DRAM
  static constexpr int SC_PER = SC_TOK + 2 * BMW;
  static constexpr int SLOT_COLS = QPS * SUB_COLS;  // sub-tile h: [slot * SLOT_COLS + 64 h, + N)
  // One barrier per step records that the step's MMAs have completed (a single
  // tcgen05.commit): it frees the step's A stage (raw for e4m3 / e5m2,
  // converted otherwise) and operand stage and hands its accumulator slot to
  // the epilogue; step j uses index j % NDONE.
  static constexpr int NDONE = NACC;
  static constexpr uint32_t RT_BYTES = (KS / 64) * RT_STRIP;
  // operand sub-tile: 4 BT = 64 split rows (per 8 chunk rows: 8 h, 8 l, 8 h2, 8 l2
  // rows), or 32 e4m3 token rows
  static constexpr uint32_t B_SUBT = (kSplit ? 4 * BT : BT) * KQ;
  static constexpr uint32_t B_BYTES = QPS * B_SUBT;
  static constexpr int kConvWarps = kA8 ? 1 : 4;       // token split, or the token-scale warp
  // weight rewrite: 4 warps (one thread per weight row), or 8 (two threads per
  // row) with e4m3 activations, whose single token warp leaves room
  static constexpr int kWConvWarps = kConv ? (kA8 ? 8 : 4) : 0;
  static constexpr int kRowParts = kWConvWarps / 4;
  // MMA issuers: warp 1 and the warps from kMma2 on, each taking every
  // kIssuers-th step (one thread issues a tcgen05.mma only every ~44-80 cycles;
  // issuers on several warps add up)
  static constexpr int kIssuers = 2;
  static constexpr int kMma2 = 6 + kConvWarps + kWConvWarps;
  static constexpr int kThreads = 32 * (kMma2 + kIssuers - 1);

  static constexpr uint32_t OFF_RAW = 0;
  static constexpr uint32_t OFF_CONV = OFF_RAW + RAWST * RAW_BYTES;
  static constexpr uint32_t OFF_RT = OFF_CONV + CST * CONV_BYTES;
  static constexpr uint32_t OFF_B = OFF_RT + RTS * RT_BYTES;
  static constexpr uint32_t OFF_SC = OFF_B + BST * B_BYTES;
  static constexpr uint32_t OFF_CTRL = OFF_SC + NSC * SC_PER * 4;
  static constexpr uint32_t OFF_RAWFULL = OFF_CTRL;
  static constexpr uint32_t OFF_RAWEMPTY = OFF_RAWFULL + 8 * RAWST;
  static constexpr uint32_t OFF_CONVFULL = OFF_RAWEMPTY + 8 * RAWST;
  static constexpr uint32_t OFF_DONEB = OFF_CONVFULL + 8 * (CST > 0 ? CST : 1);
  static constexpr uint32_t OFF_RFULL = OFF_DONEB + 8 * NDONE;
  static constexpr uint32_t OFF_REMPTY = OFF_RFULL + 8 * RTS;
  static constexpr uint32_t OFF_BFULL = OFF_REMPTY + 8 * RTS;
  static constexpr uint32_t OFF_SFULL = OFF_BFULL + 8 * BST;
  static constexpr uint32_t OFF_SEMPTY = OFF_SFULL + 8 * NSC;
  static constexpr uint32_t OFF_ACCE = OFF_SEMPTY + 8 * NSC;
  static constexpr uint32_t OFF_DONE = OFF_ACCE + 8 * NACC;
  static constexpr uint32_t OFF_TMEM = OFF_DONE + 8 * kIssuers;
  static constexpr uint32_t OFF_ABORT = OFF_TMEM + 4;
  static constexpr uint32_t OFF_OFFS = OFF_CTRL + 1024;
  static constexpr uint32_t OFF_TILES = OFF_OFFS + 4 * (kMaxGroups + 4);
  static constexpr uint32_t SMEM_USED = OFF_TILES + 4 * (kMaxGroups + 4);
  static constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;

  static_assert(NACC * SLOT_COLS <= int(TMEM_COLS), "TMEM map");
  // the MMA's N (4 T8 split rows, or up to 32 token rows) fits a sub-tile's columns
  static_assert((kSplit ? 4 * BT : BT) <= SUB_COLS, "sub-tile accumulator width");
  static_assert(kConv || RAWST == NDONE, "raw stages are freed through the step-done ring");
  static_assert(BST <= NDONE && CST <= NDONE, "step-done ring indexing");
  // Issuer i takes the steps j with j % kIssuers == i: a ring the issuers wait on must be at
  // least kIssuers deep, or the issuer of step j + depth (another warp) could begin its parity
  // wait a phase early and pass it at once.
  static_assert(NACC >= kIssuers && BST >= kIssuers && (kConv ? CST : RAWST) >= kIssuers,
                "rings the MMA issuers wait on");
  static_assert(OFF_ABORT + 4 <= OFF_OFFS, "control block overlaps the tables");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
  static_assert(OFF_CONV % 1024 == 0 && OFF_RT % 1024 == 0 && OFF_B % 1024 == 0 && B_SUBT % 1024 == 0,
                "swizzle atoms are 1024-byte aligned");
};

struct Params {
  const int32_t* group_sizes;
  int32_t num_total_groups, group_offset, num_local_groups;
  int32_t m, n, k;
  const void* scale;  // f32, or E8M0 bytes when scale_e8m0
  int32_t num_blocks;
  const void* bias;
  int32_t bias_f32;
  void* out;
  uint32_t* err;  // [0] sticky error flags; [1] split marks pending; [2] CTAs done (fix_marked_rows)
  int32_t zero_rest;  // zero the rows outside the local groups (gmm) or leave them (gmm_into)
  const int32_t* group_offset_dev;  // NULL, or the device scalar that replaces group_offset
  int32_t scale_e8m0;
  const float* lhs_scale;  // e4m3 activations: NULL or f32 [m, num_lhs_blocks];
                           // split activations: (s1, s2) pairs [m, num_lhs_blocks = k steps, 2]
  int32_t num_lhs_blocks;
  // For the rows whose split needs the exact path: the bf16 lhs [m, k] and the
  // weights as stored, [L, n, w_row_bytes] (k bytes, or k / 2 for 4-bit formats).
  const uint16_t* x;
  const uint8_t* w;
  int64_t w_row_bytes;
  // NVFP4 on the fp16-weight kernel: e4m3 block scales [L, n, k / 16] of the e2m1
  // weights (applied again by the exact recompute); NULL otherwise.
  const uint8_t* w_block_scale;
};

// A 4-byte asynchronous copy global -> shared, and the arrive on an mbarrier
// that follows this thread's earlier such copies (the barrier's pending count
// is raised now and lowered when they land, so the phase waits for them).
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.shared.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// An E8M0 block scale as fp32 (page "gemm_quant.rs", widen_block_scale_f32):
// byte e is 2^(e - 127), the bits e << 23, except that 0 is 2^-127 and 255 is 0.
__device__ __forceinline__ float e8m0_value(uint32_t e) {
  return e == 255u ? 0.f : __uint_as_float(e == 0u ? 0x00400000u : e << 23);
}

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

// Largest value (max) or union (or) over the TPR lanes of a token row; a row's
// lanes are TPR consecutive lanes starting at a multiple of TPR.  Every lane of
// the warp must call these together.
template <int TPR>
__device__ __forceinline__ uint32_t row_max(uint32_t v) {
  if constexpr (TPR == 32) {
    return __reduce_max_sync(0xffffffffu, v);
  } else {
#pragma unroll
    for (int d = 1; d < TPR; d <<= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, d));
    return v;
  }
}
template <int TPR>
__device__ __forceinline__ uint32_t row_or(uint32_t v) {
  if constexpr (TPR == 32) {
    return __reduce_or_sync(0xffffffffu, v);
  } else {
#pragma unroll
    for (int d = 1; d < TPR; d <<= 1) v |= __shfl_xor_sync(0xffffffffu, v, d);
    return v;
  }
}

// Bits of the scale 2^(E-7) and of its inverse for a largest magnitude with
// fp32 bits `amax` (sign cleared): E + 127 = amax's exponent field, kept in
// [8, 254] so that both are fp32 normals.
__device__ __forceinline__ float split_scale(uint32_t amax) {
  return __uint_as_float((min(max(amax >> 23, 8u), 254u) - 7u) << 23);
}
__device__ __forceinline__ float split_inv_scale(uint32_t amax) {
  return __uint_as_float((261u - min(max(amax >> 23, 8u), 254u)) << 23);
}

// x - s (h + l / 16) for the e4m3 codes h, l of two values (low bytes of hw, lw
// first): what a split level leaves of x.  Exact: s (h + l / 16) is a multiple of
// s 2^-13 below 2^128 with at most 22 significant bits, and the difference,
// a multiple of x's last place smaller than x or zero, is an fp32 value.
__device__ __forceinline__ float2 split_rest(float x0, float x1, uint32_t hw, uint32_t lw, float s) {
  const float2 h = e4m3x2_value(hw), l = e4m3x2_value(lw);
  return make_float2(fmaf(-s, fmaf(l.x, 0.0625f, h.x), x0), fmaf(-s, fmaf(l.y, 0.0625f, h.y), x1));
}

// The two-level split of one token row's k step (a pipeline step of the fp8
// kernel), of which this lane holds N bf16 values, packed two per word (k order,
// low half first; lanes past k hold zeros).  With M1 the step's largest |x| and
// s1 = 2^(E1-7), E1 = floor(log2 M1) (clamped as in split_scale):
//   x = s1 (h + l / 16) + r,       h = e4m3(x / s1),  l = e4m3(16 (x / s1 - h)),
// exact (r = 0) for every |x| >= 2^(E1-13); the rest r, an fp32 value, is split
// the same way with its own largest magnitude M2 and s2 = 2^(E2-7):
//   r = s2 (h2 + l2 / 16) + r2.
// When r = 0 for the whole step, s2 = 0 and h2 = l2 = 0.  When r2 != 0 somewhere
// in the step (the step's magnitudes spread over more than two such ranges), or
// the step holds an infinity or a NaN, s2 carries a set sign bit (s2 = -|s2|, or
// -0): the row must then be computed another way, and s1 is NaN for a
// non-finite step.  Every lane of the warp calls this together.  The rest is
// only computed when some row of the warp has a non-zero value below 2^(E1-13)
// (biased exponent below e1 - 13; none can be rounded when e1 <= 14, as x's last
// place is then no finer than the split's), decided by a vote, so that warps
// whose rows need no second level skip that work.
template <int N, int TPR>
__device__ __forceinline__ void split_step(const uint32_t (&xw)[N / 2], uint32_t (&hw)[N / 4], uint32_t (&lw)[N / 4],
                                           uint32_t (&hw2)[N / 4], uint32_t (&lw2)[N / 4], float& s1, float& s2) {
  static_assert(N % 4 == 0, "values per lane");
  uint32_t amax = 0;
#pragma unroll
  for (int i = 0; i < N / 2; ++i) amax = max(amax, max((xw[i] << 16) & 0x7FFFFFFFu, xw[i] & 0x7FFF0000u));
  amax = row_max<TPR>(amax);
  s1 = split_scale(amax);
  {
    const float inv = split_inv_scale(amax);
    float y[N];
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      y[2 * i] = __uint_as_float(xw[i] << 16) * inv;
      y[2 * i + 1] = __uint_as_float(xw[i] & 0xFFFF0000u) * inv;
    }
    split_e4m3<N>(y, hw, lw);
  }
  const bool nonfinite = amax >= 0x7F800000u;
  const uint32_t e1 = min(max(amax >> 23, 8u), 254u);
  bool small = false;  // a value of this lane the first level may round
#pragma unroll
  for (int i = 0; i < N / 2; ++i) {
    const uint32_t a = (xw[i] << 16) & 0x7FFFFFFFu, b = xw[i] & 0x7FFF0000u;
    small |= (a != 0u && (a >> 23) + 13u < e1) || (b != 0u && (b >> 23) + 13u < e1);
  }
  bool rest = false;  // the row has values that neither level holds
  s2 = 0.f;
#pragma unroll
  for (int j = 0; j < N / 4; ++j) hw2[j] = lw2[j] = 0u;
  if (__any_sync(0xffffffffu, small && !nonfinite)) {
    // what level 1 leaves: r = x - s1 (h + l / 16)
    float r[N];
    uint32_t rmax = 0;
#pragma unroll
    for (int j = 0; j < N / 4; ++j) {
      const uint32_t x01 = xw[2 * j], x23 = xw[2 * j + 1];
      const float2 r01 =
          split_rest(__uint_as_float(x01 << 16), __uint_as_float(x01 & 0xFFFF0000u), hw[j], lw[j], s1);
      const float2 r23 =
          split_rest(__uint_as_float(x23 << 16), __uint_as_float(x23 & 0xFFFF0000u), hw[j] >> 16, lw[j] >> 16, s1);
      r[4 * j] = r01.x, r[4 * j + 1] = r01.y, r[4 * j + 2] = r23.x, r[4 * j + 3] = r23.y;
#pragma unroll
      for (int u = 0; u < 4; ++u) rmax = max(rmax, __float_as_uint(r[4 * j + u]) & 0x7FFFFFFFu);
    }
    rmax = row_max<TPR>(rmax);
    if (nonfinite) rmax = 0u;
    const float inv2 = split_inv_scale(rmax);
    float y2[N];
#pragma unroll
    for (int j = 0; j < N; ++j) y2[j] = r[j] * inv2;
    split_e4m3<N>(y2, hw2, lw2);
    const float t2 = rmax != 0u ? split_scale(rmax) : 0.f;
    uint32_t left = 0;  // this lane's values that neither level holds
#pragma unroll
    for (int j = 0; j < N / 4; ++j) {
      const float2 a = split_rest(r[4 * j], r[4 * j + 1], hw2[j], lw2[j], t2);
      const float2 b = split_rest(r[4 * j + 2], r[4 * j + 3], hw2[j] >> 16, lw2[j] >> 16, t2);
      left |= __float_as_uint(a.x) | __float_as_uint(a.y) | __float_as_uint(b.x) | __float_as_uint(b.y);
    }
    if (rmax == 0u) {  // no second level in this row: zero codes, as in warps that skip it
      left = 0u;
#pragma unroll
      for (int j = 0; j < N / 4; ++j) hw2[j] = lw2[j] = 0u;
    }
    rest = row_or<TPR>(left & 0x7FFFFFFFu) != 0u;
    s2 = t2;
  }
  const bool flag = rest || nonfinite;
  if (nonfinite) s1 = __uint_as_float(0x7FC00000u);
  if (flag) s2 = __uint_as_float(__float_as_uint(s2) | 0x80000000u);
}

// ------------------------------------------------------------------ weight rewrite
// 4-bit codes become e4m3 bytes through 16-entry byte tables held in four words
// (entries 0..7 in t0/t1, 8..15 in t2/t3, little-endian, bit 7 clear) and
// prmt.  In prmt's default mode a selector nibble with bit 3 set replicates the
// sign bit of the byte it selects, so prmt(0x80808080, 0x80808080, codes) gives
// 0x80 for codes 0..7 and 0xFF for codes 8..15: the mask that picks the upper
// half of the table, and (shifted left by one) the sign bit of negative values.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// Four 4-bit codes (bits 0..15 of `codes`, k order) -> four e4m3 bytes (k order).
template <uint32_t T0, uint32_t T1, uint32_t T2, uint32_t T3, bool kSigned>
__device__ __forceinline__ uint32_t lut4(uint32_t codes) {
  if constexpr (!kSigned) {
    // Every entry is below 0x80, so a selector nibble with bit 3 set gives 0
    // (the replicated sign bit): codes 8..15 read 0 from the low table, and
    // with bit 3 flipped, codes 0..7 read 0 from the high one.
    static_assert(((T0 | T1 | T2 | T3) & 0x80808080u) == 0u, "unsigned tables hold positive codes");
    return prmt(T0, T1, codes) | prmt(T2, T3, codes ^ 0x8888u);
  }
  // signed: magnitudes from the two tables, picked and signed by the mask
  const uint32_t idx = codes & 0x7777u;
  const uint32_t upper = prmt(0x80808080u, 0x80808080u, codes);
  const uint32_t r = (prmt(T2, T3, idx) & upper) | (prmt(T0, T1, idx) & ~upper);
  return r | ((upper << 1) & 0x80808080u);
}

// e4m3 bytes of 0..15 (the unsigned table, also the low half of int4's).
constexpr uint32_t kU0 = 0x44403800u, kU1 = 0x4E4C4A48u, kU2 = 0x53525150u, kU3 = 0x57565554u;
// int4 codes 8..15 are -8..-1: magnitudes 8, 7, ..., 1 (the sign comes from the mask).
constexpr uint32_t kI2 = 0x4A4C4E50u, kI3 = 0x38404448u;
// 16 times the int4 value: magnitudes 0, 16, ..., 112 and 128, 112, ..., 16.
constexpr uint32_t kH0 = 0x64605800u, kH1 = 0x6E6C6A68u, kH2 = 0x6A6C6E70u, kH3 = 0x58606468u;

template <WFmt F>
__device__ __forceinline__ uint32_t nibble4_to_e4m3(uint32_t codes) {
  if constexpr (F == WFmt::kUint4) return lut4<kU0, kU1, kU2, kU3, false>(codes);
  else return lut4<kU0, kU1, kI2, kI3, true>(codes);
}

// 8 packed 4-bit codes (one word, k order from the low nibble) -> 8 e4m3 bytes.
template <WFmt F>
__device__ __forceinline__ void nibble8_to_e4m3(uint32_t w, uint32_t& o0, uint32_t& o1) {
  o0 = nibble4_to_e4m3<F>(w);
  o1 = nibble4_to_e4m3<F>(w >> 16);
}

// 4 int8 values (one word, k order) -> e4m3 bytes of 16 h (hi) and l (lo),
// w = 16 h + l, h the signed high nibble, l the unsigned low nibble.  The four
// low (high) nibbles are first packed into bits 0..15 as table selectors.
__device__ __forceinline__ void int8x4_to_e4m3(uint32_t w, uint32_t& hi, uint32_t& lo) {
  const uint32_t l = w & 0x0F0F0F0Fu, h = (w >> 4) & 0x0F0F0F0Fu;
  lo = lut4<kU0, kU1, kU2, kU3, false>(prmt(l | (l >> 4), 0u, 0x0020u));
  hi = lut4<kH0, kH1, kH2, kH3, true>(prmt(h | (h >> 4), 0u, 0x0020u));
}

// ------------------------------------------------------------------ exact rows
// The value of a 4-bit code (low nibble of c) of format F.
template <WFmt F>
__device__ __forceinline__ float nibble_value(uint32_t c) {
  c &= 15u;
  if constexpr (F == WFmt::kUint4) return float(c);
  if constexpr (F == WFmt::kInt4) return float(int32_t(c << 28) >> 28);
  // e2m1: sign, 2-bit exponent (bias 1), 1-bit mantissa; exponent 0 is 0 or 0.5
  const uint32_t e = (c >> 1) & 3u, m = c & 1u;
  const float v = e == 0u ? 0.5f * float(m) : __uint_as_float(((e + 126u) << 23) | (m << 22));
  return (c & 8u) ? -v : v;
}

// Eight stored weights of one row (8 bytes of an 8-bit format, or 4 bytes of a
// 4-bit one holding 8 codes) as fp32 values, k order.
template <WFmt F>
__device__ __forceinline__ void weights8(uint2 raw, float (&v)[8]) {
  if constexpr (F == WFmt::kE4M3 || F == WFmt::kE5M2) {
    const uint32_t w[2] = {raw.x, raw.y};
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t hh;
        const uint16_t pair = uint16_t(w[h] >> (16 * q));
        if constexpr (F == WFmt::kE4M3)
          asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hh) : "h"(pair));
        else
          asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(hh) : "h"(pair));
        const float2 f = __half22float2(*reinterpret_cast<__half2*>(&hh));
        v[4 * h + 2 * q] = f.x;
        v[4 * h + 2 * q + 1] = f.y;
      }
  } else if constexpr (F == WFmt::kInt8) {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = float(int32_t((i < 4 ? raw.x : raw.y) << (24 - 8 * (i & 3))) >> 24);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = nibble_value<F>(raw.x >> (4 * i));
  }
}

// out[row, col] before the bias, summed over k from the stored bf16 activations
// x (the row, k values) and weights wrow (the column's weight row as stored),
// without the split: for each quant block b the exact products x * w summed in
// fp32 (four interleaved partial sums), times the block's scale (scale[s0 + b
// sn], f32 or E8M0; 1 without scale), added in fp32; IEEE arithmetic
// throughout, so infinities and NaNs come out as the definition gives them.
// Used for the rows whose split is not exact, which realistic activations
// almost never produce; one lane per output column, its weight row read from
// global memory (k % 128 == 0, and the block width a multiple of 128, on this
// path).
template <WFmt F>
__device__ __forceinline__ float exact_row_sum(const uint16_t* __restrict__ x, const uint8_t* __restrict__ wrow,
                                               const void* scale, bool scale_e8m0, int64_t s0, int64_t sn,
                                               int32_t k, int32_t nb, const uint8_t* __restrict__ bs_row = nullptr) {
  constexpr bool k4 = F == WFmt::kInt4 || F == WFmt::kUint4 || F == WFmt::kE2M1;
  const int32_t kb = k / nb;
  float total = 0.f;
  for (int32_t b = 0; b < nb; ++b) {
    float part[4] = {0.f, 0.f, 0.f, 0.f};
    for (int32_t k0 = b * kb; k0 < (b + 1) * kb; k0 += 8) {
      const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x + k0));
      const uint2 raw = k4 ? make_uint2(__ldg(reinterpret_cast<const uint32_t*>(wrow + k0 / 2)), 0u)
                           : __ldg(reinterpret_cast<const uint2*>(wrow + k0));
      float wv[8];
      weights8<F>(raw, wv);
      if (bs_row != nullptr) {
        // NVFP4: the 8 codes' e4m3 block scale (per 16 k); MXFP8: their E8M0 one (per
        // 32 k).  w * s is exact (in fp32's range, for MXFP8)
        float sb;
        if constexpr (F == WFmt::kE2M1)
          sb = e4m3x2_value(__ldg(bs_row + k0 / 16)).x;
        else
          sb = e8m0_value(__ldg(bs_row + k0 / 32));
#pragma unroll
        for (int i = 0; i < 8; ++i) wv[i] *= sb;
      }
      const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        part[i] = fmaf(__uint_as_float(xs[i] << 16), wv[2 * i], part[i]);
        part[i] = fmaf(__uint_as_float(xs[i] & 0xFFFF0000u), wv[2 * i + 1], part[i]);
      }
    }
    float s = 1.f;
    if (scale != nullptr) {
      const int64_t si = s0 + int64_t(b) * sn;
      s = scale_e8m0 ? e8m0_value(__ldg(static_cast<const uint8_t*>(scale) + si))
                     : __ldg(static_cast<const float*>(scale) + si);
    }
    total = fmaf((part[0] + part[1]) + (part[2] + part[3]), s, total);
  }
  return total;
}

// Rows whose split a step marked (a second level left a rest, or the step held
// an infinity or a NaN) are summed again here, from the stored bf16 values and
// weights (exact_row_sum), and their outputs overwritten.  Called by every
// thread of every CTA at the end of the kernel with split activations.  With the
// split pass, which has completed by then, nothing is done unless it marked a
// row (err[1]).  Otherwise each CTA counts itself in (err[2], wrapping at the
// grid size) after its stores; the last one sees every other CTA's stores, and
// if a split marked some row (err[1], set by the split pass or the token split
// and cleared here) it finds
// the marked rows of the local groups (from the step scales' sign bits, or by
// splitting the rows again when the kernel split them itself) and recomputes
// them, one output column per thread.  Realistic activations almost never mark
// a row, so the last CTA normally only reads err[1].  `scratch`: shared memory
// no longer in use, at least 1040 bytes.
template <WFmt F, bool kPS, bool kOutF32>
__device__ __noinline__ void fix_marked_rows(const Params& p, int32_t go, const int32_t* offs, uint8_t* scratch,
                                             int32_t step) {
  uint32_t* s_todo = reinterpret_cast<uint32_t*>(scratch);
  uint8_t* mark = scratch + 16;
  constexpr int32_t RB = 1024;  // rows per block of marks
  if (threadIdx.x == 0) {
    uint32_t todo = 1u;
    if constexpr (kPS) {
      griddep_wait();  // the split pass has completed: err[1] holds all its marks
      todo = *reinterpret_cast<volatile uint32_t*>(p.err + 1);
    }
    if (todo != 0u) {
      __threadfence();  // this CTA's outputs are visible before it counts itself in
      const uint32_t prior = atomicInc(p.err + 2, gridDim.x - 1u);
      todo = 0u;
      if (prior == gridDim.x - 1u) {
        __threadfence();
        todo = atomicExch(p.err + 1, 0u);
      }
    }
    *s_todo = todo;
  }
  __syncthreads();
  if (*s_todo == 0u) return;
  const int32_t nb = p.scale != nullptr ? p.num_blocks : 1;
  const int32_t ksteps = (p.k + step - 1) / step;
  const int32_t row_lo = offs[go], row_hi = offs[go + p.num_local_groups];
  const int warps = int(blockDim.x) >> 5, wid = int(threadIdx.x) >> 5, lane = int(threadIdx.x) & 31;
  for (int32_t r0 = row_lo; r0 < row_hi; r0 += RB) {
    const int32_t nr = min(RB, row_hi - r0);
    for (int32_t i = threadIdx.x; i < nr; i += blockDim.x) mark[i] = 0;
    __syncthreads();
    if constexpr (kPS) {
      for (int64_t i = threadIdx.x; i < int64_t(nr) * ksteps; i += blockDim.x) {
        const int64_t at = (int64_t(r0) * ksteps + i) * 2 + 1;  // s2 of (row, step)
        if (__float_as_uint(p.lhs_scale[at]) >> 31) mark[i / ksteps] = 1;
      }
    } else {
      // the token split's marks, found again with the split pass's lane layout:
      // one warp per (row, step), step / 32 values per lane
      for (int64_t u = wid; u < int64_t(nr) * ksteps; u += warps) {
        const int32_t rr = int32_t(u / ksteps), ks = int32_t(u % ksteps);
        const uint16_t* x = p.x + int64_t(r0 + rr) * p.k;
        float s1, s2;
        if (step == 256) {
          uint32_t xw[4] = {0u, 0u, 0u, 0u}, hw[2], lw[2], hw2[2], lw2[2];
          const int32_t kk = ks * 256 + lane * 8;
          if (kk < p.k) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + kk));
            xw[0] = v.x, xw[1] = v.y, xw[2] = v.z, xw[3] = v.w;
          }
          split_step<8, 32>(xw, hw, lw, hw2, lw2, s1, s2);
        } else {
          uint32_t xw[2] = {0u, 0u}, hw[1], lw[1], hw2[1], lw2[1];
          const int32_t kk = ks * 128 + lane * 4;
          if (kk < p.k) {
            const uint2 v = __ldg(reinterpret_cast<const uint2*>(x + kk));
            xw[0] = v.x, xw[1] = v.y;
          }
          split_step<4, 32>(xw, hw, lw, hw2, lw2, s1, s2);
        }
        if (lane == 0 && (__float_as_uint(s2) >> 31)) mark[rr] = 1;
      }
    }
    __syncthreads();
    for (int32_t rr = 0; rr < nr; ++rr) {
      if (!mark[rr]) continue;
      const int32_t row = r0 + rr;
      int32_t lo = go, hi = go + p.num_local_groups;  // the largest g with offs[g] <= row
      while (hi - lo > 1) {
        const int32_t mid = (lo + hi) >> 1;
        if (offs[mid] <= row)
          lo = mid;
        else
          hi = mid;
      }
      const int32_t lg = lo - go;
      const uint16_t* x = p.x + int64_t(row) * p.k;
      for (int32_t c = threadIdx.x; c < p.n; c += blockDim.x) {
        float v = exact_row_sum<F>(x, p.w + (int64_t(lg) * p.n + c) * p.w_row_bytes, p.scale, p.scale_e8m0 != 0,
                                   int64_t(lg) * nb * p.n + c, p.n, p.k, nb,
                                   p.w_block_scale != nullptr
                                       ? p.w_block_scale + (int64_t(lg) * p.n + c) * (p.k / (F == WFmt::kE2M1 ? 16 : 32))
                                       : nullptr);
        if (p.bias != nullptr) {
          const int64_t bi = int64_t(lg) * p.n + c;
          v += p.bias_f32 ? __ldg(static_cast<const float*>(p.bias) + bi)
                          : __bfloat162float(static_cast<const __nv_bfloat16*>(p.bias)[bi]);
        }
        if constexpr (kOutF32)
          static_cast<float*>(p.out)[int64_t(row) * p.n + c] = v;
        else
          static_cast<__nv_bfloat16*>(p.out)[int64_t(row) * p.n + c] = __float2bfloat16_rn(v);
      }
    }
    __syncthreads();
  }
}

template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&f)[N]) {
  static_assert(N == 8 || N == 16 || N == 32, "column count");
  if constexpr (N == 8) {
    uint32_t v[8];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(v[i]);
  } else if constexpr (N == 16) {
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
    uint32_t v[32];
    tmem_ld_32cols(taddr, v);
#pragma unroll
    for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
  }
}

template <WFmt F, bool kA8, bool kPS, bool kOutF32>
__global__ void __launch_bounds__(Cfg<F, kA8, kPS>::kThreads, 1)
    gemm_fp8_kernel(const __grid_constant__ CUtensorMap tm_lhs, const __grid_constant__ CUtensorMap tm_rhs,
                    const Params p) {
  using C = Cfg<F, kA8, kPS>;
  constexpr int QPS = C::QPS, NACC = C::NACC, NDONE = C::NDONE, NSC = C::NSC;
  int32_t go;
  if (!resolve_group_offset(p.group_offset_dev, p.group_offset, p.num_total_groups, p.num_local_groups, p.err, go))
    return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_ABORT);
  int32_t* offs = reinterpret_cast<int32_t*>(smem + C::OFF_OFFS);
  int32_t* tiles = reinterpret_cast<int32_t*>(smem + C::OFF_TILES);
  float* tscale = reinterpret_cast<float*>(smem + C::OFF_SC);
  auto rawfull_bar = [&](uint32_t s) { return sbase + C::OFF_RAWFULL + 8 * s; };
  auto rawempty_bar = [&](uint32_t s) { return sbase + C::OFF_RAWEMPTY + 8 * s; };
  auto convfull_bar = [&](uint32_t s) { return sbase + C::OFF_CONVFULL + 8 * s; };
  auto stepdone_bar = [&](uint32_t s) { return sbase + C::OFF_DONEB + 8 * s; };
  auto rfull_bar = [&](uint32_t s) { return sbase + C::OFF_RFULL + 8 * s; };
  auto rempty_bar = [&](uint32_t s) { return sbase + C::OFF_REMPTY + 8 * s; };
  auto bfull_bar = [&](uint32_t s) { return sbase + C::OFF_BFULL + 8 * s; };
  auto sfull_bar = [&](uint32_t s) { return sbase + C::OFF_SFULL + 8 * s; };
  auto sempty_bar = [&](uint32_t s) { return sbase + C::OFF_SEMPTY + 8 * s; };
  auto acce_bar = [&](uint32_t s) { return sbase + C::OFF_ACCE + 8 * s; };

  const uint32_t done_bar = sbase + C::OFF_DONE;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < C::RAWST; ++s) {
      mbar_init(rawfull_bar(s), 1);
      mbar_init(rawempty_bar(s), C::kWConvWarps > 0 ? C::kWConvWarps : 1);
    }
    for (int s = 0; s < C::CST; ++s) mbar_init(convfull_bar(s), C::kWConvWarps);
    for (int s = 0; s < NDONE; ++s) mbar_init(stepdone_bar(s), 1);
    for (int s = 0; s < C::RTS; ++s) {
      mbar_init(rfull_bar(s), 1);
      mbar_init(rempty_bar(s), C::kConvWarps);
    }
    for (int s = 0; s < C::BST; ++s) mbar_init(bfull_bar(s), kA8 ? 1 : C::kConvWarps);
    for (int s = 0; s < NSC; ++s) {
      mbar_init(sfull_bar(s), C::kConvWarps);
      mbar_init(sempty_bar(s), 4);
    }
    for (int s = 0; s < NACC; ++s) mbar_init(acce_bar(s), 4);
    for (int s = 0; s < C::kIssuers; ++s) mbar_init(done_bar + 8 * s, 1);
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch(&tm_lhs);
    tma_prefetch(&tm_rhs);
  }
  if (warp == 1) {
    tmem_alloc(sbase + C::OFF_TMEM, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 2) {
    build_group_offsets(p.group_sizes, p.num_total_groups, p.m, offs, p.err);
    build_tile_prefix(offs, go, p.num_local_groups, C::BT, tiles);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + C::OFF_TMEM);

  const int32_t t_tiles = tiles[p.num_local_groups];  // row chunks over all local groups
  const int32_t n_tiles = (p.n + BMW - 1) / BMW;
  const int32_t nq = p.k / KQ;                         // 128-wide sub-tiles (k % 128 == 0 on this path)
  const int32_t ksteps = (nq + QPS - 1) / QPS;         // the last step may hold fewer sub-tiles
  const int32_t nb = p.scale != nullptr ? p.num_blocks : 1;
  const int32_t q_per_block = nq / nb;                 // (k / nb) % 128 == 0 on this path
  const int32_t total = t_tiles * n_tiles;
  // Items: row chunks outer, the weight tiles of the chunk's group inner.
  auto item_of = [&](int32_t w) {
    return decode_gemm_tile(w, t_tiles, n_tiles, n_tiles, tiles, offs, go, p.num_local_groups, C::BT);
  };
  auto halves = [&](int32_t ks) { return min(QPS, nq - QPS * ks); };
  // Rows of an item's chunk: row_end is the end of the chunk's group, which can
  // lie past the chunk's BT rows.
  auto chunk_rows = [&](const GemmTile& t) { return min(t.row_end - t.row0, int32_t(C::BT)); };
  // Step j's operand / converted stage is reused by step j + depth once step j's MMAs are done.
  auto wait_step_done = [&](uint32_t j, int depth) {
    return j < uint32_t(depth) ||
           wait_bar(stepdone_bar((j - depth) % NDONE), ((j - depth) / NDONE) & 1u, abort_flag, p.err);
  };

  // The weight scales of step ks of item t, into scale slot sc: one row per
  // quant block the step touches (at most two), the item's 128 columns as
  // stored.  Bulk copies completing on the slot's full barrier; returns their
  // bytes, which the caller's arrive expects.  Rows whose pitch is not a
  // multiple of 16 bytes (E8M0 with n % 16 != 0) are loaded by this warp
  // instead (0 bytes).
  auto load_weight_scales = [&](uint32_t sc, const GemmTile& t, int32_t ks) -> uint32_t {
    if (p.scale == nullptr) return 0u;
    const int esz = p.scale_e8m0 ? 1 : 4;
    const int32_t b0 = ks * QPS / q_per_block, b1 = min(nb - 1, (ks * QPS + halves(ks) - 1) / q_per_block);
    const int32_t cols = min(BMW, p.n - t.n_tile * BMW);
    const uint32_t dst = smem_u32(tscale + sc * C::SC_PER + C::SC_TOK);
    const uint8_t* src = static_cast<const uint8_t*>(p.scale) +
                         ((int64_t(t.local_group) * nb + b0) * p.n + int64_t(t.n_tile) * BMW) * esz;
    if ((p.n * esz) % 16 == 0 && reinterpret_cast<uintptr_t>(p.scale) % 16 == 0) {
      const uint32_t bytes = uint32_t(cols * esz + 15) & ~15u;
      if (lane == 0)
        for (int32_t b = b0; b <= b1; ++b)
          bulk_load(dst + uint32_t(b - b0) * 512u, src + int64_t(b - b0) * p.n * esz, bytes, sfull_bar(sc));
      return uint32_t(b1 - b0 + 1) * bytes;
    }
    uint8_t* d8 = reinterpret_cast<uint8_t*>(tscale + sc * C::SC_PER + C::SC_TOK);
    for (int32_t b = b0; b <= b1; ++b)
      for (int c = lane; c < cols * esz; c += 32) d8[(b - b0) * 512 + c] = __ldg(src + int64_t(b - b0) * p.n * esz + c);
    return 0u;
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      // The token ring: bf16 rows for the split (RTS deep), or e4m3 operand rows (BST deep).
      constexpr int TR = kA8 ? C::BST : C::RTS;
      uint32_t as = 0, aph = 0, rs = 0, rph = 0, apend = 0, rpend = 0;
      uint32_t apar[C::RAWST], rpar[TR];
      uint32_t j = 0;  // steps loaded so far
      bool ok = true;
      bool split_ready = false;  // kPS: the split rows' kernel has completed
      for (int32_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
        const GemmTile t = item_of(w);
        const int32_t rboxes = chunk_rows(t) > 16 ? 2 : 1;
        for (int32_t ks = 0; ks < ksteps; ++ks) {
          const int32_t hq = halves(ks);
          // Raw stage `as` is free once its last reader is done: the MMAs of the
          // step RAWST before (index as, previous phase), or the weight rewrite.
          const uint32_t free_bar = C::kConv ? rawempty_bar(as) : stepdone_bar(as);
          if (!wait_bar(free_bar, aph ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const uint32_t dst = sbase + C::OFF_RAW + as * C::RAW_BYTES;
          if constexpr (C::kNibble) {
            // one box of 128 bytes per row = 256 k (a half-empty box past k is zero-filled)
            mbar_arrive_expect_tx(rawfull_bar(as), RAW_BOX);
            tma_load_3d(dst, &tm_rhs, rawfull_bar(as), ks * 128, t.n_tile * BMW, t.local_group);
          } else {
            mbar_arrive_expect_tx(rawfull_bar(as), uint32_t(hq) * C::RAW_TX);
            for (int h = 0; h < hq; ++h)
              tma_load_3d(dst + h * RAW_BOX, &tm_rhs, rawfull_bar(as), (QPS * ks + h) * KQ, t.n_tile * BMW,
                          t.local_group);
          }
          apar[as] = aph;
          apend |= 1u << as;
          if (++as == C::RAWST) {
            as = 0;
            aph ^= 1u;
          }
          if constexpr (kPS) {
            // per 8 chunk rows one {128 k, 8 rows, 4 planes} box: their h, l,
            // h2 and l2 rows, operand rows [32 b, 32 b + 32) of each sub-tile
            if (!wait_step_done(j, C::BST)) {
              ok = false;
              break;
            }
            const int t8 = t8_of(chunk_rows(t));
            if (!split_ready) {  // weights already stream; the split rows come from the kernel before
              griddep_wait();
              split_ready = true;
            }
            mbar_arrive_expect_tx(bfull_bar(rs), uint32_t(hq * 4 * t8) * 128u);
            for (int h = 0; h < hq; ++h)
              for (int r8 = 0; r8 < t8; r8 += 8)
                tma_load_3d(sbase + C::OFF_B + rs * C::B_BYTES + h * C::B_SUBT + uint32_t(4 * r8) * 128u, &tm_lhs,
                            bfull_bar(rs), (QPS * ks + h) * KQ, t.row0 + r8, 0);
          } else if constexpr (kA8) {
            // e4m3 token rows, one {128 k, 16 rows} box per sub-tile and 16 rows,
            // straight into operand stage rs once step j - BST's MMAs are done.
            if (!wait_step_done(j, C::BST)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(bfull_bar(rs), uint32_t(rboxes * hq) * RT_BOX);
            for (int h = 0; h < hq; ++h)
              for (int rb = 0; rb < rboxes; ++rb)
                tma_load_2d(sbase + C::OFF_B + rs * C::B_BYTES + h * C::B_SUBT + rb * RT_BOX, &tm_lhs,
                            bfull_bar(rs), (QPS * ks + h) * KQ, t.row0 + 16 * rb);
          } else {
            if (!wait_bar(rempty_bar(rs), rph ^ 1u, abort_flag, p.err)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(rfull_bar(rs), uint32_t(rboxes * 2 * hq) * RT_BOX);
            for (int st = 0; st < 2 * hq; ++st)
              for (int rb = 0; rb < rboxes; ++rb)
                tma_load_2d(sbase + C::OFF_RT + rs * C::RT_BYTES + st * C::RT_STRIP + rb * RT_BOX, &tm_lhs,
                            rfull_bar(rs), ks * C::KS + 64 * st, t.row0 + 16 * rb);
          }
          rpar[rs] = rph;
          rpend |= 1u << rs;
          if (++rs == TR) {
            rs = 0;
            rph ^= 1u;
          }
          ++j;
        }
      }
      if (!ok) {
        for (int s = 0; s < C::RAWST; ++s)
          if (apend >> s & 1u) drain_bar(rawfull_bar(s), apar[s]);
        for (int s = 0; s < TR; ++s)
          if (rpend >> s & 1u) drain_bar(kA8 ? bfull_bar(s) : rfull_bar(s), rpar[s]);
      }
    }
  } else if (warp == 1 || warp >= C::kMma2) {
    // ---------------------------------------------------------------- MMA issuers
    // Step j accumulates sub-tile h into TMEM columns [SLOT_COLS slot + 64 h,
    // + 2 T8) of slot j % NACC; the epilogue frees the slot after reading it.
    // Issuer `mine` takes the steps j with j % kIssuers == mine: each step has
    // its own A stage, operand stage, slot and commit, so they share nothing.
    const uint32_t mine = warp == 1 ? 0u : uint32_t(warp - C::kMma2 + 1);
    constexpr uint32_t kAst = C::kConv ? C::CST : C::RAWST;
    bool ok = true;
    uint32_t j = 0;  // the step's index over the CTA's items
    for (int32_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
      const GemmTile t = item_of(w);
      const int t8 = t8_of(chunk_rows(t));
      // N: the h, l, h2 and l2 rows of the split (4 T8), or the e4m3 token rows (16 or 32).
      const uint32_t idesc = idesc_e4m3(BMW, C::kSplit ? 4 * t8 : max(t8, 16)) | (C::kAType << 7);
      for (int32_t ks = 0; ks < ksteps; ++ks, ++j) {
        if (j % C::kIssuers != mine) continue;
        const uint32_t as = j % kAst, aph = (j / kAst) & 1u, bs = j % C::BST, bph = (j / C::BST) & 1u;
        const uint32_t slot = j % NACC, sph = (j / NACC) & 1u;
        const int32_t hq = halves(ks);
        const uint32_t afull = C::kConv ? convfull_bar(as) : rawfull_bar(as);
        if (!wait_bar(acce_bar(slot), sph ^ 1u, abort_flag, p.err) || !wait_bar(afull, aph, abort_flag, p.err) ||
            !wait_bar(bfull_bar(bs), bph, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          for (int h = 0; h < hq; ++h) {
            const uint32_t b0 = sbase + C::OFF_B + bs * C::B_BYTES + h * C::B_SUBT;
            const uint32_t d = tmem_base + slot * C::SLOT_COLS + uint32_t(h) * SUB_COLS;
#pragma unroll
            for (int pass = 0; pass < C::PASSES; ++pass) {
              const uint32_t a0 = C::kConv ? sbase + C::OFF_CONV + as * C::CONV_BYTES + (h * C::PASSES + pass) * A_SUB
                                           : sbase + C::OFF_RAW + as * C::RAW_BYTES + h * RAW_BOX;
#pragma unroll
              for (int kk = 0; kk < KQ / 32; ++kk)
                mma_e4m3_ss(d, sw128_desc(a0 + 32 * kk, 16, 1024), sw128_desc(b0 + 32 * kk, 16, 1024), idesc,
                            (pass | kk) != 0 ? 1u : 0u);
            }
          }
          mma_commit(stepdone_bar(slot));
        }
        __syncwarp();
      }
    }
    if (lane == 0) {
      mma_commit(done_bar + 8 * mine);
      drain_bar(done_bar + 8 * mine, 0);
    }
    __syncwarp();
  } else if (warp < 6) {
    // ---------------------------------------------------------------- epilogue
    // Per sub-tile q of the item (block q / q_per_block): read its h columns,
    // then its l columns, and fold them with the block's weight scale for this
    // lane's column and the step's token scales.
    const int quarter = warp & 3;
    const int wrow = quarter * 32 + lane;  // weight row in the tile = output column
    const uint32_t lane_base = uint32_t(quarter * 32) << 16;
    uint32_t slot = 0, sph = 0, sc = 0, scph = 0;
    bool ok = true;
    for (int32_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
      const GemmTile t = item_of(w);
      const int32_t col = t.n_tile * BMW + wrow;
      const bool col_ok = col < p.n;
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
        for (int32_t q = 0; q < nq && ok; ++q) {
          const int h = q % QPS;
          if (h == 0) {
            if (!wait_bar(stepdone_bar(slot), sph, abort_flag, p.err) ||
                !wait_bar(sfull_bar(sc), scph, abort_flag, p.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          // the weight scale of the sub-tile's block for this column, staged with
          // the step's token scales (row 0: the step's first block)
          const int srow = q / q_per_block - (q - h) / q_per_block;
          const uint8_t* wsc = reinterpret_cast<const uint8_t*>(tscale + sc * C::SC_PER + C::SC_TOK) + srow * 512;
          const float sw = p.scale == nullptr ? 1.f
                           : p.scale_e8m0   ? e8m0_value(wsc[wrow])
                                            : reinterpret_cast<const float*>(wsc)[wrow];
          const uint32_t col0 = tmem_base + lane_base + slot * C::SLOT_COLS + uint32_t(h) * SUB_COLS;
          if constexpr (!C::kSplit) {
            // one e4m3 product per token: its T8 columns, times the sub-tile's token scale
            const float* ts = tscale + sc * C::SC_PER + h * C::BT;
            float d[T8];
            tmem_ld_cols<T8>(col0, d);
#pragma unroll
            for (int i = 0; i < T8; ++i) acc[i] = fmaf(sw * ts[i], d[i], acc[i]);
          } else {
            // Chunk row 8 b + i has its h, l, h2, l2 products in columns 32 b + i,
            // + 8, + 16, + 24.  The h2 and l2 columns are read only in steps where
            // some row of the chunk has a second level (s2 != 0).
            const float2* ts = reinterpret_cast<const float2*>(tscale + sc * C::SC_PER);
            const uint4 lv2 = *reinterpret_cast<const uint4*>(tscale + sc * C::SC_PER + 2 * C::BT);
            const bool two = (lv2.x | lv2.y | lv2.z | lv2.w) != 0u;
#pragma unroll
            for (int b = 0; b < T8 / 8; ++b) {
              float d[16];
              tmem_ld_cols<16>(col0 + 32 * b, d);
#pragma unroll
              for (int i = 0; i < 8; ++i)
                acc[8 * b + i] = fmaf(sw * ts[8 * b + i].x, fmaf(d[8 + i], 0.0625f, d[i]), acc[8 * b + i]);
              if (two) {
                tmem_ld_cols<16>(col0 + 32 * b + 16, d);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  // a row without a second level keeps its sum (its h2 / l2 products
                  // are with zero codes, NaN against an infinite weight)
                  const float s2 = ts[8 * b + i].y;
                  if (s2 != 0.f) acc[8 * b + i] = fmaf(sw * s2, fmaf(d[8 + i], 0.0625f, d[i]), acc[8 * b + i]);
                }
              }
            }
          }
          if (h == QPS - 1 || q + 1 == nq) {
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
      const int t8 = t8_of(chunk_rows(t));
      if (t8 == 8)
        run(std::integral_constant<int, 8>{});
      else if (C::kSplit || t8 == 16)
        run(std::integral_constant<int, 16>{});
      else
        run(std::integral_constant<int, C::kSplit ? 16 : 32>{});
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
  } else if (kA8 && warp == 6) {
    // ---------------------------------------------------------------- token scales
    // e4m3 activations: per step, the token scale of each of its sub-tiles for
    // the item's rows (lhs_scale[row, lhs block of the sub-tile], 1 without
    // lhs_scale, 0 for operand rows past the chunk).  Split activations: the
    // row's (s1, s2) for the step (lhs_scale[row, step, 0..1]) for both
    // sub-tiles, (0, 0) past the chunk.
    if constexpr (kPS) griddep_wait();  // the step scales come from the kernel before
    const int32_t nlb = p.lhs_scale != nullptr ? p.num_lhs_blocks : 1;
    const int32_t q_per_lblock = nq / nlb;  // (k / nlb) % 128 == 0 on this path
    uint32_t sc = 0, scph = 0;
    uint32_t wpend = 0, wpar = 0;  // slots with weight-scale copies issued, and their phases
    bool ok = true;
    for (int32_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
      const GemmTile t = item_of(w);
      const int32_t rows = chunk_rows(t);
      for (int32_t ks = 0; ks < ksteps; ++ks) {
        const int32_t hq = halves(ks);
        if (!wait_bar(sempty_bar(sc), scph ^ 1u, abort_flag, p.err)) {
          ok = false;
          break;
        }
        if constexpr (kPS) {
          uint32_t two = 0;  // some row of the chunk has a second level in this step
          for (int idx = lane; idx < 2 * C::BT; idx += 32) {
            const int r = idx >> 1;
            const float v = r < rows ? __ldg(p.lhs_scale + (int64_t(t.row0 + r) * nlb + ks) * 2 + (idx & 1)) : 0.f;
            tscale[sc * C::SC_PER + idx] = v;
            two |= (idx & 1) ? __float_as_uint(v) : 0u;
          }
          two = __any_sync(0xffffffffu, two != 0u) ? 1u : 0u;
          if (lane < 4) reinterpret_cast<uint32_t*>(tscale)[sc * C::SC_PER + 2 * C::BT + lane] = lane == 0 ? two : 0u;
        } else {
          for (int idx = lane; idx < QPS * C::BT; idx += 32) {
            const int h = idx / C::BT, r = idx % C::BT;
            float v = 0.f;
            if (h < hq && r < rows)
              v = p.lhs_scale != nullptr ? __ldg(p.lhs_scale + int64_t(t.row0 + r) * nlb + (QPS * ks + h) / q_per_lblock)
                                         : 1.f;
            tscale[sc * C::SC_PER + idx] = v;
          }
        }
        const uint32_t wbytes = load_weight_scales(sc, t, ks);
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(sfull_bar(sc), wbytes);
        if (wbytes != 0u) {
          wpend |= 1u << sc;
          wpar = (wpar & ~(1u << sc)) | (scph << sc);
        }
        if (++sc == NSC) {
          sc = 0;
          scph ^= 1u;
        }
      }
    }
    // a wait gave up: the weight-scale copies still in flight land before exit
    if (!ok && lane == 0)
      for (int s2 = 0; s2 < NSC; ++s2)
        if (wpend >> s2 & 1u) drain_bar(sfull_bar(s2), wpar >> s2 & 1u);
  } else if (!kA8 && warp < 10) {
    // ---------------------------------------------------------------- token split
    // The 128 threads share a step's T8 rows evenly: 128 / T8 adjacent lanes per
    // token row r, each taking the same T8 consecutive k of every sub-tile h of
    // the step (T8 / 8 bf16 chunks of 16 bytes per sub-tile from the token tile).
    // split_step turns them into T8 bytes of each of h, l, h2 and l2, written to
    // rows 32 (r / 8) + 8 p + r % 8 (p = 0, 1, 2, 3) of operand sub-tile h; the
    // lanes of a row agree on its maxima by shuffles.  All tiles are 128-byte
    // swizzled: 16-byte chunk j of row R sits at position j ^ (R % 8), and
    // R % 8 = r % 8.
    const int ct = int(threadIdx.x) - 192;
    uint32_t rs = 0, rph = 0, bs = 0, sc = 0, scph = 0;
    uint32_t wpend = 0, wpar = 0;  // warp 6: slots with weight-scale copies issued, and their phases
    uint32_t j = 0;  // steps split so far
    bool ok = true;
    for (int32_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
      const GemmTile t = item_of(w);
      const int32_t rows = chunk_rows(t);
      auto run = [&](auto t8c) {
        constexpr int T8 = decltype(t8c)::value;
        constexpr int TPR = 128 / T8;  // threads per token row: 16 or 8
        constexpr int NV = QPS * T8;   // values per lane and step
        const int r = ct / TPR, seg = ct % TPR;
        for (int32_t ks = 0; ks < ksteps; ++ks) {
          const int32_t hq = halves(ks);
          if (!wait_bar(rfull_bar(rs), rph, abort_flag, p.err) || !wait_step_done(j, C::BST) ||
              !wait_bar(sempty_bar(sc), scph ^ 1u, abort_flag, p.err)) {
            ok = false;
            return;
          }
          // Sub-tile h, k [T8 seg, T8 seg + T8): bf16 chunks c = T8 seg / 8 + i of
          // the sub-tile, in strip 2 h + c / 8 of the token tile at position c % 8.
          uint32_t xw[NV / 2];
          const uint32_t src = sbase + C::OFF_RT + rs * C::RT_BYTES + uint32_t(r) * 128u;
#pragma unroll
          for (int h = 0; h < QPS; ++h) {
#pragma unroll
            for (int i = 0; i < T8 / 8; ++i) {
              uint32_t* v = xw + h * (T8 / 2) + 4 * i;
              v[0] = v[1] = v[2] = v[3] = 0u;
              if (h < hq) {
                const int c = seg * (T8 / 8) + i;
                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
                             : "r"(src + uint32_t(2 * h + (c >> 3)) * C::RT_STRIP +
                                   (uint32_t((c & 7) ^ (r & 7)) << 4)));
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(rempty_bar(rs));  // the values are in registers
          uint32_t code[4][NV / 4];
          float s1, s2;
          split_step<NV, TPR>(xw, code[0], code[1], code[2], code[3], s1, s2);
#pragma unroll
          for (int h = 0; h < QPS; ++h) {
            if (h < hq) {
              // e4m3 bytes [T8 seg, T8 seg + T8) of each of the row's four operand
              // rows: 16-byte chunk (T8 seg) / 16, at byte (T8 seg) % 16 within it.
              const uint32_t sub = sbase + C::OFF_B + bs * C::B_BYTES + uint32_t(h) * C::B_SUBT;
#pragma unroll
              for (int pl = 0; pl < 4; ++pl) {
                const uint32_t prow = sub + uint32_t(32 * (r >> 3) + 8 * pl + (r & 7)) * 128u;
                const uint32_t* cw = code[pl] + h * (T8 / 4);
                if constexpr (T8 == 8) {
                  const uint32_t pos = (uint32_t((seg >> 1) ^ (r & 7)) << 4) + uint32_t(seg & 1) * 8u;
                  asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(prow + pos), "r"(cw[0]), "r"(cw[1]));
                } else {
                  st_shared_v4(prow + (uint32_t(seg ^ (r & 7)) << 4), cw[0], cw[1], cw[2], cw[3]);
                }
              }
            }
          }
          const bool live = r < rows;
          if (seg == 0) {
            tscale[sc * C::SC_PER + 2 * r] = live ? s1 : 0.f;
            tscale[sc * C::SC_PER + 2 * r + 1] = live ? s2 : 0.f;
            // a marked row: the last CTA sums it again (see fix_marked_rows)
            if (live && (__float_as_uint(s2) >> 31)) atomicOr(p.err + 1, 1u);
          }
          // warp 6 brings the step's weight scales (its arrive expects their bytes)
          const uint32_t wbytes = warp == 6 ? load_weight_scales(sc, t, ks) : 0u;
          // this warp's rows: any second level in the step (read by the epilogue)
          const bool two = __any_sync(0xffffffffu, seg == 0 && live && __float_as_uint(s2) != 0u);
          if (lane == 0)
            reinterpret_cast<uint32_t*>(tscale)[sc * C::SC_PER + 2 * C::BT + (warp - 6)] = two ? 1u : 0u;
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(bfull_bar(bs));
            mbar_arrive_expect_tx(sfull_bar(sc), wbytes);
          }
          if (wbytes != 0u) {
            wpend |= 1u << sc;
            wpar = (wpar & ~(1u << sc)) | (scph << sc);
          }
          if (++rs == C::RTS) {
            rs = 0;
            rph ^= 1u;
          }
          if (++bs == C::BST) bs = 0;
          if (++sc == NSC) {
            sc = 0;
            scph ^= 1u;
          }
          ++j;
        }
      };
      if (t8_of(rows) == 8)
        run(std::integral_constant<int, 8>{});
      else
        run(std::integral_constant<int, 16>{});
    }
    // a wait gave up: the weight-scale copies still in flight land before exit
    if (!ok && warp == 6 && lane == 0)
      for (int s2 = 0; s2 < NSC; ++s2)
        if (wpend >> s2 & 1u) drain_bar(sfull_bar(s2), wpar >> s2 & 1u);
  } else if constexpr (C::kConv) {
    // ---------------------------------------------------------------- weight rewrite
    // Thread t rewrites part t / 128 (of kRowParts) of weight row r = t % 128 of
    // every sub-tile of the step.  Raw rows and A-tile rows are 128 bytes,
    // 128-byte swizzled (chunk j of row r at position j ^ (r % 8)), so the 8
    // rows of a quarter-warp hit 8 different positions.  4-bit: raw chunk 4 h + i
    // (32 codes) of the row becomes A chunks 2 i and 2 i + 1 of sub-tile h.
    // int8: raw chunk c (16 values) becomes chunk c of the 16 h tile (pass 0)
    // and of the l tile (pass 1).
    constexpr int kParts = C::kRowParts;
    const int tw = int(threadIdx.x) - 32 * (6 + C::kConvWarps);
    const int r = tw & 127, part = tw >> 7;
    uint32_t rs = 0, rph = 0, cs = 0;
    uint32_t j = 0;  // steps rewritten so far
    bool ok = true;
    for (int32_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
      for (int32_t ks = 0; ks < ksteps; ++ks) {
        const int32_t hq = halves(ks);
        if (!wait_bar(rawfull_bar(rs), rph, abort_flag, p.err) || !wait_step_done(j, C::CST)) {
          ok = false;
          break;
        }
        const uint32_t src = sbase + C::OFF_RAW + rs * C::RAW_BYTES + uint32_t(r) * 128u;
        const uint32_t dst = sbase + C::OFF_CONV + cs * C::CONV_BYTES + uint32_t(r) * 128u;
        if constexpr (C::kNibble) {
          for (int h = 0; h < hq; ++h) {
#pragma unroll
            for (int ii = 0; ii < 4 / kParts; ++ii) {
              const int i = part * (4 / kParts) + ii;
              uint32_t x[4];
              asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                           : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3])
                           : "r"(src + (uint32_t((4 * h + i) ^ (r & 7)) << 4)));
              uint32_t o[8];
#pragma unroll
              for (int u = 0; u < 4; ++u) nibble8_to_e4m3<F>(x[u], o[2 * u], o[2 * u + 1]);
              const uint32_t sub = dst + uint32_t(h) * A_SUB;
              st_shared_v4(sub + (uint32_t((2 * i) ^ (r & 7)) << 4), o[0], o[1], o[2], o[3]);
              st_shared_v4(sub + (uint32_t((2 * i + 1) ^ (r & 7)) << 4), o[4], o[5], o[6], o[7]);
            }
          }
        } else {
          // int8: this thread's raw chunks of the row are loaded first, so that
          // their latencies overlap
          constexpr int kChunks = 8 / kParts;
          uint32_t x[kChunks][4];
#pragma unroll
          for (int cc = 0; cc < kChunks; ++cc) {
            const int c = part * kChunks + cc;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(x[cc][0]), "=r"(x[cc][1]), "=r"(x[cc][2]), "=r"(x[cc][3])
                         : "r"(src + (uint32_t(c ^ (r & 7)) << 4)));
          }
#pragma unroll
          for (int cc = 0; cc < kChunks; ++cc) {
            const int c = part * kChunks + cc;
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) int8x4_to_e4m3(x[cc][u], hi[u], lo[u]);
            const uint32_t pos = uint32_t(c ^ (r & 7)) << 4;
            st_shared_v4(dst + pos, hi[0], hi[1], hi[2], hi[3]);
            st_shared_v4(dst + A_SUB + pos, lo[0], lo[1], lo[2], lo[3]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(rawempty_bar(rs));
          mbar_arrive(convfull_bar(cs));
        }
        if (++rs == C::RAWST) {
          rs = 0;
          rph ^= 1u;
        }
        if (++cs == C::CST) cs = 0;
        ++j;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
  if constexpr (C::kSplit) fix_marked_rows<F, kPS, kOutF32>(p, go, offs, smem + C::OFF_B, C::KS);
}

template <WFmt F, bool kA8, bool kPS, bool kOutF32>
cudaError_t launch_format(const ScaledLaunch& L, int grid, cudaStream_t stream) {
  using C = Cfg<F, kA8, kPS>;
  auto kern = gemm_fp8_kernel<F, kA8, kPS, kOutF32>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(C::SMEM_BYTES));
  if (e != cudaSuccess) return e;
  constexpr bool k4 = F == WFmt::kInt4 || F == WFmt::kUint4 || F == WFmt::kE2M1;
  Params p{L.group_sizes, L.num_total_groups, L.group_offset, L.num_local_groups, L.m, L.n, L.k, L.scale,
           L.num_blocks, L.bias, L.bias_f32, L.out, L.err, L.zero_rest, L.group_offset_dev, L.scale_e8m0,
           L.lhs_scale, L.num_lhs_blocks, static_cast<const uint16_t*>(L.lhs_raw),
           static_cast<const uint8_t*>(L.rhs_raw), k4 ? int64_t(L.k) / 2 : int64_t(L.k),
           /*w_block_scale=*/nullptr};  // block-scaled weights run on the other kernels
  if constexpr (kPS) {
    // Launched as the programmatic dependent of the split-rows kernel just
    // before it in the stream: the prologue and the weight stream overlap that
    // kernel's end; only the split rows and their scales wait for it.  Every
    // other input was written before that kernel started.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(unsigned(C::kThreads));
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, L.tm_lhs, L.tm_rhs, p);
  }
  kern<<<grid, C::kThreads, C::SMEM_BYTES, stream>>>(L.tm_lhs, L.tm_rhs, p);
  return cudaGetLastError();
}

// bf16 activations (kA8 false: the exact two-term split), e4m3 ones (kA8
// true) or split ones (kA8 and kPS).
template <WFmt F, bool kA8, bool kPS = false>
cudaError_t launch_format(const ScaledLaunch& L, bool out_f32, int grid, cudaStream_t stream) {
  return out_f32 ? launch_format<F, kA8, kPS, true>(L, grid, stream)
                 : launch_format<F, kA8, kPS, false>(L, grid, stream);
}

}  // namespace fp8
}  // namespace gmmk
