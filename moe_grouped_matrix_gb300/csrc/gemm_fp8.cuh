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
// Activations.  The bf16 lhs rows are brought to e4m3 without losing their
// value: for each token row and each pipeline step, with M the largest |x| of
// the row's step and E = floor(log2 M),
//   x = 2^(E-7) * (h + l / 16),   h = rne_e4m3(x / 2^(E-7)),
//                                 l = rne_e4m3(16 * (x / 2^(E-7) - h)).
// |x / 2^(E-7)| < 256, so h never saturates.  x has 8 significant bits and h the
// top 4 of them (rounded), so x / 2^(E-7) - h is a multiple of x's last place
// below half of h's last place: at most 4 significant bits, and 16 times it lies
// in e4m3's range.  The split is exact for every x with |x| >= 2^(E-13), where
// x / 2^(E-7) is an e4m3 normal: so for every x within 2^13 of M.  Below that,
// l is rounded to a multiple of 2^-9, an error of at most M * 2^-21 in x.  h and l are B operand rows (a token's h
// in row i, its l in row T8 + i); their products with the weights are exact and
// the tensor core sums them in fp32.  Each 128-wide sub-tile accumulates into
// its own TMEM columns, and the epilogue folds it as
//   acc[i] += s[g, b, c] * 2^(E_i-7) * (D[c, i] + D[c, T8 + i] / 16).
//
// Pipeline (one CTA per SM, persistent over items).  A step covers QPS
// sub-tiles (2, i.e. 256 k; 1 for int8, whose tiles are twice the MMA work);
// the last step of an item may hold fewer.  Roles:
//   warp 0      TMA: the step's raw weight boxes (4-deep ring) and its bf16
//               token rows ({64 k, 16 rows} boxes, 2-deep ring); with e4m3
//               activations the e4m3 token rows ({128 k, 16 rows} boxes)
//               straight into a 4-deep operand ring; with split activations
//               (below) their h and l rows ({128 k, 8 rows} boxes) likewise
//   warps 6-9   split the bf16 token rows into e4m3 h / l operand rows (2-deep
//               ring; all 128 threads share any chunk size) and write each
//               row's step scale (8-deep ring); with e4m3 activations warp 6
//               alone writes each sub-tile's token scales
//   next 4 or 8 (int8, int4, uint4) rewrite raw weight tiles as e4m3 A tiles
//               (2-deep ring): one weight row per thread, or half a row with
//               e4m3 activations (8 warps)
//   warp 1      TMEM owner; per step 4 MMAs 128 x N x 32 per A tile (N = 2 T8,
//               or 16 / 32 e4m3 token rows), one accumulator per sub-tile,
//               and one commit into a step-done ring
//   warps 2-5   per sub-tile: TMEM -> registers, fold with the token scale and
//               the sub-tile's weight-block scale into fp32 registers; per item
//               add the bias, round, store
// Items are (local group, chunk of up to 32 of its rows, 128-wide n tile); a
// chunk of t rows uses T8 = 8, 16 or 32 operand rows per half (t rounded up).
//
// Split activations (kPS).  The same two-term split of the bf16 rows can be
// made once per row by act_split.cu, instead of once per row and n tile here:
// h and l codes of every row in two e4m3 planes and each row's 2^(E-7) per
// step.  The kernel then loads the chunk's h rows into operand rows [0, T8)
// and its l rows into [T8, 2 T8), the layout the token split writes, and takes
// the step scales through the token-scale warp; the MMAs and the fold are
// those of the bf16 path, so both give the same bits.
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
constexpr int BT = 32;    // token rows per item at most
constexpr int KQ = 128;   // k per sub-tile (one e4m3 A tile row is 128 bytes)
constexpr uint32_t TMEM_COLS = 512;
constexpr int kMaxGroups = 1024;
constexpr uint32_t A_SUB = BMW * KQ;     // one e4m3 A tile: 128 rows x 128 bytes
constexpr uint32_t RAW_BOX = BMW * 128;  // one raw weight box: 128 rows x 128 bytes
constexpr uint32_t RT_STRIP = BT * 128;  // 64 k of bf16 for 32 token rows
constexpr uint32_t RT_BOX = 16 * 128;    // one {64 k, 16 rows} box
constexpr uint32_t B_SUB = 2 * BT * KQ;  // e4m3 operand sub-tile: 64 rows x 128 bytes

// kA8: the token operand comes by TMA (e4m3 activations, or with kPS the
// split activations) and warp 6 writes its scales.
template <WFmt F, bool kA8, bool kPS = false>
struct Cfg {
  static_assert(kA8 || !kPS, "split activations come by TMA");
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
  static constexpr int SC_PER = kA8 ? QPS * BT : BT;  // token scales per step: per sub-tile with kA8
  static constexpr int SLOT_COLS = QPS * 2 * BT;  // sub-tile h: [slot * SLOT_COLS + 64 h, + 2 T8)
  // One barrier per step records that the step's MMAs have completed (a single
  // tcgen05.commit): it frees the step's A stage (raw for e4m3 / e5m2,
  // converted otherwise) and operand stage and hands its accumulator slot to
  // the epilogue; step j uses index j % NDONE.
  static constexpr int NDONE = NACC;
  static constexpr uint32_t RT_BYTES = (KS / 64) * RT_STRIP;
  static constexpr uint32_t B_SUBT = kA8 && !kPS ? BT * KQ : B_SUB;  // operand sub-tile: 32 or 64 rows
  static constexpr uint32_t B_BYTES = QPS * B_SUBT;
  static constexpr int kConvWarps = kA8 ? 1 : 4;       // token split, or the token-scale warp
  // weight rewrite: 4 warps (one thread per weight row), or 8 (two threads per
  // row) with e4m3 activations, whose single token warp leaves room
  static constexpr int kWConvWarps = kConv ? (kA8 ? 8 : 4) : 0;
  static constexpr int kRowParts = kWConvWarps / 4;
  static constexpr int kThreads = 192 + 32 * (kConvWarps + kWConvWarps);

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
  static constexpr uint32_t OFF_TMEM = OFF_DONE + 8;
  static constexpr uint32_t OFF_ABORT = OFF_TMEM + 4;
  static constexpr uint32_t OFF_OFFS = OFF_CTRL + 1024;
  static constexpr uint32_t OFF_TILES = OFF_OFFS + 4 * (kMaxGroups + 4);
  static constexpr uint32_t SMEM_USED = OFF_TILES + 4 * (kMaxGroups + 4);
  static constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;

  static_assert(NACC * SLOT_COLS <= int(TMEM_COLS), "TMEM map");
  static_assert(kConv || RAWST == NDONE, "raw stages are freed through the step-done ring");
  static_assert(BST <= NDONE && CST <= NDONE, "step-done ring indexing");
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
  uint32_t* err;
  int32_t zero_rest;  // zero the rows outside the local groups (gmm) or leave them (gmm_into)
  const int32_t* group_offset_dev;  // NULL, or the device scalar that replaces group_offset
  int32_t scale_e8m0;
  const float* lhs_scale;  // e4m3 activations: NULL or f32 [m, num_lhs_blocks]
  int32_t num_lhs_blocks;
};

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
    mbar_init(done_bar, 1);
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
    build_tile_prefix(offs, go, p.num_local_groups, BT, tiles);
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
    return decode_gemm_tile(w, t_tiles, n_tiles, n_tiles, tiles, offs, go, p.num_local_groups, BT);
  };
  auto halves = [&](int32_t ks) { return min(QPS, nq - QPS * ks); };
  // Step j's operand / converted stage is reused by step j + depth once step j's MMAs are done.
  auto wait_step_done = [&](uint32_t j, int depth) {
    return j < uint32_t(depth) ||
           wait_bar(stepdone_bar((j - depth) % NDONE), ((j - depth) / NDONE) & 1u, abort_flag, p.err);
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
        const int32_t rboxes = t.row_end - t.row0 > 16 ? 2 : 1;
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
            // h and l rows, {128 k, 8 rows} boxes from planes 0 and 1, into
            // operand rows [0, T8) and [T8, 2 T8) of each sub-tile
            if (!wait_step_done(j, C::BST)) {
              ok = false;
              break;
            }
            const int t8 = t8_of(t.row_end - t.row0);
            if (!split_ready) {  // weights already stream; the split rows come from the kernel before
              griddep_wait();
              split_ready = true;
            }
            mbar_arrive_expect_tx(bfull_bar(rs), uint32_t(hq * 2 * t8) * 128u);
            for (int h = 0; h < hq; ++h)
              for (int z = 0; z < 2; ++z)
                for (int r8 = 0; r8 < t8; r8 += 8)
                  tma_load_3d(sbase + C::OFF_B + rs * C::B_BYTES + h * C::B_SUBT + uint32_t(z * t8 + r8) * 128u,
                              &tm_lhs, bfull_bar(rs), (QPS * ks + h) * KQ, t.row0 + r8, z);
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
                tma_load_2d(sbase + C::OFF_RT + rs * C::RT_BYTES + st * RT_STRIP + rb * RT_BOX, &tm_lhs,
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
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    // Step j accumulates sub-tile h into TMEM columns [SLOT_COLS slot + 64 h,
    // + 2 T8) of slot j % NACC; the epilogue frees the slot after reading it.
    uint32_t as = 0, aph = 0, bs = 0, bph = 0, slot = 0, sph = 0;
    bool ok = true;
    for (int32_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
      const GemmTile t = item_of(w);
      const int t8 = t8_of(t.row_end - t.row0);
      // N: the h and l rows of the split (2 T8), or the e4m3 token rows (16 or 32).
      const uint32_t idesc = idesc_e4m3(BMW, kA8 && !kPS ? max(t8, 16) : 2 * t8) | (C::kAType << 7);
      for (int32_t ks = 0; ks < ksteps; ++ks) {
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
            const uint32_t d = tmem_base + slot * C::SLOT_COLS + uint32_t(h) * (2 * BT);
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
        if (++as == (C::kConv ? C::CST : C::RAWST)) {
          as = 0;
          aph ^= 1u;
        }
        if (++bs == C::BST) {
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
    // Per sub-tile q of the item (block q / q_per_block): read its h columns,
    // then its l columns, and fold them with the block's weight scale for this
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
      const int64_t sidx = int64_t(t.local_group) * nb * p.n + col;  // scale of block 0 for this column
      // Prefetched as stored (f32 bits or an E8M0 byte), widened only when used, so
      // that no instruction waits for the loads before then.
      auto load_scales = [&](int32_t b0, uint32_t (&dst)[kPre]) {
#pragma unroll
        for (int j = 0; j < kPre; ++j) {
          dst[j] = p.scale_e8m0 ? 127u : 0x3F800000u;  // 1
          if (p.scale != nullptr && col_ok && b0 + j < nb) {
            const int64_t i = sidx + int64_t(b0 + j) * p.n;
            dst[j] = p.scale_e8m0 ? uint32_t(__ldg(static_cast<const uint8_t*>(p.scale) + i))
                                  : __float_as_uint(__ldg(static_cast<const float*>(p.scale) + i));
          }
        }
      };
      auto widen = [&](uint32_t v) { return p.scale_e8m0 ? e8m0_value(v) : __uint_as_float(v); };
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
        uint32_t s_cur[kPre], s_next[kPre];
        load_scales(0, s_cur);
        int32_t q = 0;
        for (int32_t c0 = 0; c0 < nb && ok; c0 += kPre) {
          load_scales(c0 + kPre, s_next);
#pragma unroll
          for (int bi = 0; bi < kPre; ++bi) {
            if (c0 + bi >= nb || !ok) break;
            const float sw = widen(s_cur[bi]);
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
              const float* ts = tscale + sc * C::SC_PER + (kA8 ? h * BT : 0);
              const uint32_t col0 = tmem_base + lane_base + slot * C::SLOT_COLS + uint32_t(h) * (2 * BT);
              if constexpr (kA8 && !kPS) {
                // one e4m3 product per token: its T8 columns, times the sub-tile's token scale
                float d[T8];
                tmem_ld_cols<T8>(col0, d);
#pragma unroll
                for (int i = 0; i < T8; ++i) acc[i] = fmaf(sw * ts[i], d[i], acc[i]);
              } else if constexpr (T8 < 32) {
                // h and l columns in one load
                float d[2 * T8];
                tmem_ld_cols<2 * T8>(col0, d);
#pragma unroll
                for (int i = 0; i < T8; ++i) acc[i] = fmaf(sw * ts[i], fmaf(d[T8 + i], 0.0625f, d[i]), acc[i]);
              } else {
                // 32 h columns, then 32 l columns (fewer live registers)
                float d[T8];
                tmem_ld_cols<T8>(col0, d);
#pragma unroll
                for (int i = 0; i < T8; ++i) acc[i] = fmaf(sw * ts[i], d[i], acc[i]);
                tmem_ld_cols<T8>(col0 + T8, d);
#pragma unroll
                for (int i = 0; i < T8; ++i) acc[i] = fmaf(sw * ts[i] * 0.0625f, d[i], acc[i]);
              }
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
    // row's 2^(E-7) for the step (lhs_scale[row, step]) for both sub-tiles.
    if constexpr (kPS) griddep_wait();  // the step scales come from the kernel before
    const int32_t nlb = p.lhs_scale != nullptr ? p.num_lhs_blocks : 1;
    const int32_t q_per_lblock = nq / nlb;  // (k / nlb) % 128 == 0 on this path
    uint32_t sc = 0, scph = 0;
    bool ok = true;
    for (int32_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
      const GemmTile t = item_of(w);
      const int32_t rows = t.row_end - t.row0;
      for (int32_t ks = 0; ks < ksteps; ++ks) {
        const int32_t hq = halves(ks);
        if (!wait_bar(sempty_bar(sc), scph ^ 1u, abort_flag, p.err)) {
          ok = false;
          break;
        }
        for (int idx = lane; idx < QPS * BT; idx += 32) {
          const int h = idx / BT, r = idx % BT;
          float v = 0.f;
          if (h < hq && r < rows)
            v = p.lhs_scale != nullptr
                    ? __ldg(p.lhs_scale + int64_t(t.row0 + r) * nlb + (kPS ? ks : (QPS * ks + h) / q_per_lblock))
                    : 1.f;
          tscale[sc * C::SC_PER + idx] = v;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(sfull_bar(sc));
        if (++sc == NSC) {
          sc = 0;
          scph ^= 1u;
        }
      }
    }
  } else if (!kA8 && warp < 10) {
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
    uint32_t j = 0;  // steps split so far
    bool ok = true;
    for (int32_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
      const GemmTile t = item_of(w);
      auto run = [&](auto t8c) {
        constexpr int T8 = decltype(t8c)::value;
        constexpr int TPR = 128 / T8;  // threads per token row: 16, 8 or 4
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
          uint32_t xw[QPS][T8 / 2];
          uint32_t amax = 0;
          const uint32_t src = sbase + C::OFF_RT + rs * C::RT_BYTES + uint32_t(r) * 128u;
#pragma unroll
          for (int h = 0; h < QPS; ++h) {
            if (h < hq) {
#pragma unroll
              for (int i = 0; i < T8 / 8; ++i) {
                const int c = seg * (T8 / 8) + i;
                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(xw[h][4 * i]), "=r"(xw[h][4 * i + 1]), "=r"(xw[h][4 * i + 2]),
                               "=r"(xw[h][4 * i + 3])
                             : "r"(src + uint32_t(2 * h + (c >> 3)) * RT_STRIP + (uint32_t((c & 7) ^ (r & 7)) << 4)));
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
              const uint32_t sub = sbase + C::OFF_B + bs * C::B_BYTES + uint32_t(h) * B_SUB;
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
      const int t8 = t8_of(t.row_end - t.row0);
      if (t8 == 8)
        run(std::integral_constant<int, 8>{});
      else if (t8 == 16)
        run(std::integral_constant<int, 16>{});
      else
        run(std::integral_constant<int, 32>{});
    }
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
}

template <WFmt F, bool kA8, bool kPS, bool kOutF32>
cudaError_t launch_format(const ScaledLaunch& L, int grid, cudaStream_t stream) {
  using C = Cfg<F, kA8, kPS>;
  auto kern = gemm_fp8_kernel<F, kA8, kPS, kOutF32>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(C::SMEM_BYTES));
  if (e != cudaSuccess) return e;
  Params p{L.group_sizes, L.num_total_groups, L.group_offset, L.num_local_groups, L.m, L.n, L.k, L.scale,
           L.num_blocks, L.bias, L.bias_f32, L.out, L.err, L.zero_rest, L.group_offset_dev, L.scale_e8m0,
           L.lhs_scale, L.num_lhs_blocks};
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
