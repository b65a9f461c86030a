// Grouped matmul with int8, int4, uint4, NVFP4 or MXFP8 weights on the fp16 tensor cores:
//   out[r, c] = sum_b s[g, b, c] * sum_{kk in block b} lhs[r, kk] * W(g, c, kk) + bias[g, c]
// (page "tpu-inference 0.12.0.dev20251213 -> 0.13.2.dev20251230", gmm.py:
// _accum scales each quant block's partial sum by rhs_scale[g, b, 0, n] and adds
// rhs_bias once; common.py lists int8, int4 and uint4 among the weight formats).
//
// Every int8, int4 and uint4 value is an fp16 value, and an fp16 value is
// reached from its code by placing it in the mantissa of 1024 (0x6400) and
// subtracting the bias, two values per instruction: int8 codes are moved next
// to 0x64 bytes by prmt, 4-bit codes masked into the low nibble of each half
// (or the second nibble, taken back by a multiply-add with 1/16).  That is
// about one integer instruction per weight, where the e4m3 rewrite of the same
// codes (gemm_fp8.cuh) needs table lookups and held the integer pipe.  The
// 4-bit rewrite produces each 8 k in the order 0, 4, 1, 5, 2, 6, 3, 7; the
// activation rows are stored in the same order, so the products pair up.
// NVFP4 (e2m1 codes with an e4m3 scale per 16 k; microscaling, the scope's
// next formats) is a 4-bit format whose rewrite also multiplies each code by
// its block scale, which fp16 holds exactly (e2m1x8_to_f16); the block scales
// come with each raw box.
// MXFP8 (e4m3 codes with an E8M0 scale per 32 k): every e4m3 value is an fp16
// value (one cvt per two codes), but a power of two from 2^-127 to 2^127 is
// not always one, so the block scales are not folded into the weights: each
// 32-k block of a step accumulates into its own 16 columns (a step's slot is
// 64 columns, 4 slots), and the epilogue scales the four partial sums by their
// blocks' powers of two.  The E8M0 bytes come with the step's scales (4 bytes
// of each weight row a step).
//
// Activations: bf16 rows split once per row and 128-wide step by
// act_split_f16_kernel (act_split.cu) into fp16 values x / sc with sc a power
// of two per (row, step): exact for every x within 2^28 of the step's largest
// and for smaller ones down to fp16's subnormal grid.  A step the split does
// not hold exactly (or with an infinity or a NaN) marks its row, and the last
// CTA sums that row again from the stored values (fix_marked_rows in
// gemm_fp8.cuh).  fp16 x fp16 products are exact and the tensor core sums
// them in fp32, as the pages' dot_general with an f32 result.
//
// Pipeline (one CTA per SM, persistent over items of (local group, chunk of
// up to 16 of its rows, 128-wide n tile)); a step is 128 k:
//   warp 0      TMA: raw weight boxes {128 bytes, 128 rows} (128 k of int8,
//               256 k of a 4-bit format: two steps; NVFP4 adds the box's
//               {16 bytes, 128 rows} of block scales) into a 6-deep ring
//   warp 17     TMA: the chunk's fp16 activation rows, one {64 k, 16 rows,
//               2 atoms} box a step, into an 8-deep ring
//   warps 8-15  rewrite a step's raw codes as an fp16 A tile in tensor memory
//               (weight row r in TMEM lane r, 64 columns of two fp16 in k
//               order), half a weight row per thread, 4-deep
//   warps 1, 7, 18, 19
//               MMA issuers, each every fourth step: 8 tcgen05.mma.kind::f16
//               128 x 16 x 16 with A read from tensor memory, into the step's
//               32-column accumulator slot (8 slots), one commit; warp 1 owns
//               the tensor memory
//   warps 6, 16 per step (even / odd): the chunk rows' split scales, and the
//               weight scales of the step's quant block for the item's 128
//               columns (bulk copies on the slot's barrier)
//   warps 2-5   per step: acc[i] += s_w * sc_i * D[i]; per item the bias,
//               rounding and the store, lane = output column
// Why so many control warps: measured on GB300, one thread issues a
// tcgen05.mma about every 44-53 cycles whatever the shape (M = 128, N = 16 to
// 32), while issuers on several warps add up (two reach ~27 cycles per MMA
// between them, four ~13); an mbarrier check costs such a thread ~170 cycles
// inside this kernel.  With one issuer a step took ~1350 cycles, of which ~700
// issuing its 8 MMAs; with four, and the scale work split in two, the kernel
// runs a step in ~880 cycles (int8: 0.62 of the HBM roofline).  The A tiles
// live in tensor memory because shared memory could not carry them beside the
// raw boxes (writing and reading 32 KB of fp16 a step).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gemm_fp8.cuh"

namespace gmmk {
namespace f16w {
namespace {

using fp8::cp_async_4;
using fp8::cp_async_mbar_arrive;
using fp8::cp_async_wait_all;
using fp8::Params;
using fp8::WFmt;

constexpr int BMW = 128;                   // weight rows (n) per item = MMA M
constexpr int BT = 16;                     // token rows per item at most = MMA N
constexpr int KS = 128;                    // k per step
constexpr uint32_t RAW_BYTES = 128 * 128;  // one raw box
constexpr uint32_t SCALE_BOX = 16 * 128;   // NVFP4: the box's e4m3 block scales, 16 a weight row (256 k)
constexpr uint32_t RAW_STAGE = RAW_BYTES + SCALE_BOX;
constexpr int RAWST = 6;
constexpr int A_COLS = KS / 2;             // TMEM columns of one A tile (two fp16 per column)
constexpr int CST = 4;
constexpr uint32_t B_ATOM = BT * 128;      // 16 rows x 64 fp16
constexpr uint32_t B_BYTES = 2 * B_ATOM;
constexpr int BST = 8;
constexpr int NACC = 8;                    // accumulator slots
constexpr int NDONE = 8;                   // step-done barriers: step j commits to j % NDONE
constexpr int SLOT_COLS = 32;
constexpr uint32_t A_COL0 = NACC * SLOT_COLS;  // the A tiles follow the accumulator slots
constexpr uint32_t TMEM_COLS = 512;
constexpr int NSC = 8;
constexpr int SC_TOK = BT;                 // the chunk rows' split scales
constexpr int SC_MX = SC_TOK + BMW;        // MXFP8: the step's 4 E8M0 bytes of each weight row
constexpr int SC_PER = SC_MX + BMW;        // after one 512-byte weight-scale row
constexpr int MX_SLOT_COLS = 4 * BT;       // MXFP8: a step's four 32-k blocks, 16 columns each
constexpr int MX_NACC = A_COL0 / MX_SLOT_COLS;
constexpr int kMaxGroups = 1024;
constexpr int kConvWarps = 8;             // the weight rewrite: two threads per weight row
constexpr int kParts = kConvWarps / 4;
constexpr int kMma2 = 7;                   // the second MMA issuer
constexpr int kConvWarp0 = 8;              // a multiple of 4: warp w reaches TMEM lanes 32 (w % 4) ..
constexpr int kScale2 = kConvWarp0 + kConvWarps;  // the second scale warp
constexpr int kBWarp = kScale2 + 1;        // the activation-row copies
constexpr int kMma3 = kBWarp + 1;          // MMA issuers 3 and 4
constexpr int kIssuers = 4;
constexpr int kThreads = 32 * (kMma3 + 2);

constexpr uint32_t OFF_RAW = 0;
constexpr uint32_t OFF_B = OFF_RAW + RAWST * RAW_STAGE;
constexpr uint32_t OFF_SC = OFF_B + BST * B_BYTES;
constexpr uint32_t OFF_CTRL = OFF_SC + NSC * SC_PER * 4;
constexpr uint32_t OFF_RAWFULL = OFF_CTRL;
constexpr uint32_t OFF_RAWEMPTY = OFF_RAWFULL + 8 * RAWST;
constexpr uint32_t OFF_CONVFULL = OFF_RAWEMPTY + 8 * RAWST;
constexpr uint32_t OFF_DONEB = OFF_CONVFULL + 8 * CST;
constexpr uint32_t OFF_BFULL = OFF_DONEB + 8 * NDONE;
constexpr uint32_t OFF_SFULL = OFF_BFULL + 8 * BST;
constexpr uint32_t OFF_SEMPTY = OFF_SFULL + 8 * NSC;
constexpr uint32_t OFF_ACCE = OFF_SEMPTY + 8 * NSC;
constexpr uint32_t OFF_DONE = OFF_ACCE + 8 * NACC;
constexpr uint32_t OFF_TMEM = OFF_DONE + 8 * kIssuers;
constexpr uint32_t OFF_ABORT = OFF_TMEM + 4;
constexpr uint32_t OFF_OFFS = OFF_CTRL + 1024;
constexpr uint32_t OFF_TILES = OFF_OFFS + 4 * (kMaxGroups + 4);
constexpr uint32_t SMEM_USED = OFF_TILES + 4 * (kMaxGroups + 4);
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;
static_assert(OFF_ABORT + 4 <= OFF_OFFS, "control block overlaps the tables");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(OFF_B % 1024 == 0 && B_ATOM % 1024 == 0 && RAW_STAGE % 1024 == 0, "swizzle atoms are 1024-byte aligned");
static_assert(CST <= NDONE && BST <= NDONE && NACC <= NDONE, "step-done ring indexing");
static_assert(NACC * SLOT_COLS <= int(A_COL0) && A_COL0 + CST * A_COLS <= TMEM_COLS, "TMEM map");
static_assert(MX_NACC * MX_SLOT_COLS <= int(A_COL0) && MX_NACC <= NACC, "TMEM map (MXFP8)");
// Issuer i takes the steps j with j % kIssuers == i.  A ring an issuer waits on must be at
// least kIssuers deep: the issuer of step j has issued step j - kIssuers, so the ring's
// producer is then past step j - depth, and the wait cannot see that step's phase parity as
// its own.  A shallower ring lets the issuer of step j + depth, another warp, begin its wait a
// phase early and pass it at once (tests/test_f16w_pipeline_cpu.py models the protocol).
static_assert(CST >= kIssuers && BST >= kIssuers && NACC >= kIssuers && MX_NACC >= kIssuers,
              "rings the MMA issuers wait on");

// kind::f16 with fp16 A and B (type code 0), both K-major, f32 D.
__host__ __device__ constexpr uint32_t idesc_f16(int m, int n) { return (1u << 4) | (uint32_t(n >> 3) << 17) | (uint32_t(m >> 4) << 24); }

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// Four int8 values (k order, lowest in the low byte) -> two fp16x2 words: with
// u = v + 128 (the sign bit flipped), 0x64uu is the fp16 1024 + u, and 1024 +
// u - 1152 = v exactly.
__device__ __forceinline__ void int8x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  lo = hsub2(prmt(u, 0x64646464u, 0x4140u), 0x64806480u);
  hi = hsub2(prmt(u, 0x64646464u, 0x4342u), 0x64806480u);
}

// Four e4m3 codes (k order, lowest in the low byte) -> two fp16x2 words, the
// lower byte of each pair in the lower half: exact, every e4m3fn value being an
// fp16 value (the NaN codes become NaN).
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(lo) : "h"(uint16_t(w)));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hi) : "h"(uint16_t(w >> 16)));
}

// Eight 4-bit codes (k order from the low nibble) -> four fp16x2 words holding
// k (0, 4), (1, 5), (2, 6), (3, 7).  A code c in the low nibble of a half
// under 0x6400 is 1024 + c; in its second nibble 1024 + 16 c, which times 1/16
// minus 64 is c.  Signed codes are biased by 8 first (c ^ 8 = c + 8 mod 16).
template <bool kSigned>
__device__ __forceinline__ void nib8_to_f16(uint32_t w, uint32_t (&o)[4]) {
  const uint32_t u = kSigned ? w ^ 0x88888888u : w;
  const uint32_t sub = kSigned ? 0x64086408u : 0x64006400u;  // 1032 or 1024
  const uint32_t add = kSigned ? 0xD480D480u : 0xD400D400u;  // -72 or -64
  const uint32_t u8 = u >> 8;
  o[0] = hsub2((u & 0x000F000Fu) | 0x64006400u, sub);
  o[1] = hfma2((u & 0x00F000F0u) | 0x64006400u, 0x2C002C00u, add);
  o[2] = hsub2((u8 & 0x000F000Fu) | 0x64006400u, sub);
  o[3] = hfma2((u8 & 0x00F000F0u) | 0x64006400u, 0x2C002C00u, add);
}

// NVFP4: eight e2m1 codes (k order from the low nibble) times their block's
// e4m3 scale -> four fp16x2 words holding k (0, 4), (1, 5), (2, 6), (3, 7), as
// nib8_to_f16 orders them.  A code's sign and three magnitude bits placed at
// fp16 bits 15 and 11..9 are the fp16 number 2^-14 times its value (magnitude
// 1 lands on fp16's subnormal 2^-15 = 0.5 * 2^-14), so times 2^14 it is the
// value; times the scale (`s2`, the scale in both halves) it stays exact: an
// e2m1 value times an e4m3 one has at most 6 significant bits, lies within
// 6 * 448 = 2688 and, being a multiple of 2^-10, on fp16's normal grid.
__device__ __forceinline__ void e2m1x8_to_f16(uint32_t w, uint32_t s2, uint32_t (&o)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t v = w >> (4 * i);  // code i in bits 0..3, code i + 4 in bits 16..19
    const uint32_t bits = ((v & 0x00070007u) << 9) | ((v & 0x00080008u) << 12);
    o[i] = hmul2(hmul2(bits, 0x74007400u), s2);  // 2^14, then the block scale
  }
}

// D[tmem] (+)= A[tmem] * B[smem]^T, fp16 inputs, fp32 accumulator; A (M = 128)
// one row per TMEM lane, two fp16 per 32-bit column in k order.
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st_32cols(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

template <WFmt F, bool kOutF32>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_f16w_kernel(const __grid_constant__ CUtensorMap tm_lhs, const __grid_constant__ CUtensorMap tm_rhs,
                     const __grid_constant__ CUtensorMap tm_bs,
                     const Params p) {
  constexpr bool kNv = F == WFmt::kE2M1;  // NVFP4: e2m1 codes with an e4m3 scale per 16 k
  constexpr bool k4 = F == WFmt::kInt4 || F == WFmt::kUint4 || kNv;
  constexpr int STEPS_PER_RAW = k4 ? 2 : 1;  // a raw box holds 256 k of a 4-bit format
  constexpr bool kMx = F == WFmt::kE4M3;     // MXFP8: e4m3 codes with an E8M0 scale per 32 k
  constexpr int kSlotCols = kMx ? MX_SLOT_COLS : SLOT_COLS;
  constexpr int kNacc = kMx ? MX_NACC : NACC;
  int32_t go;
  if (!resolve_group_offset(p.group_offset_dev, p.group_offset, p.num_total_groups, p.num_local_groups, p.err, go))
    return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + OFF_ABORT);
  int32_t* offs = reinterpret_cast<int32_t*>(smem + OFF_OFFS);
  int32_t* tiles = reinterpret_cast<int32_t*>(smem + OFF_TILES);
  float* tscale = reinterpret_cast<float*>(smem + OFF_SC);
  auto rawfull_bar = [&](uint32_t s) { return sbase + OFF_RAWFULL + 8 * s; };
  auto rawempty_bar = [&](uint32_t s) { return sbase + OFF_RAWEMPTY + 8 * s; };
  auto convfull_bar = [&](uint32_t s) { return sbase + OFF_CONVFULL + 8 * s; };
  auto stepdone_bar = [&](uint32_t s) { return sbase + OFF_DONEB + 8 * s; };
  auto bfull_bar = [&](uint32_t s) { return sbase + OFF_BFULL + 8 * s; };
  auto sfull_bar = [&](uint32_t s) { return sbase + OFF_SFULL + 8 * s; };
  auto sempty_bar = [&](uint32_t s) { return sbase + OFF_SEMPTY + 8 * s; };
  auto acce_bar = [&](uint32_t s) { return sbase + OFF_ACCE + 8 * s; };
  const uint32_t done_bar = sbase + OFF_DONE;  // one per MMA issuer

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < RAWST; ++s) {
      mbar_init(rawfull_bar(s), 1);
      mbar_init(rawempty_bar(s), kConvWarps);  // the rewrite warps, after the raw box's last step
    }
    for (int s = 0; s < CST; ++s) mbar_init(convfull_bar(s), kConvWarps);
    for (int s = 0; s < NDONE; ++s) mbar_init(stepdone_bar(s), 1);
    for (int s = 0; s < NACC; ++s) mbar_init(acce_bar(s), 4);
    for (int s = 0; s < BST; ++s) mbar_init(bfull_bar(s), 1);
    for (int s = 0; s < NSC; ++s) {
      mbar_init(sfull_bar(s), 1);
      mbar_init(sempty_bar(s), 4);
    }
    for (int s = 0; s < kIssuers; ++s) mbar_init(done_bar + 8 * s, 1);
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch(&tm_lhs);
    tma_prefetch(&tm_rhs);
    if constexpr (kNv) tma_prefetch(&tm_bs);
  }
  if (warp == 1) {
    tmem_alloc(sbase + OFF_TMEM, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 2) {
    build_group_offsets(p.group_sizes, p.num_total_groups, p.m, offs, p.err);
    build_tile_prefix(offs, go, p.num_local_groups, BT, tiles);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + OFF_TMEM);

  const int32_t t_tiles = tiles[p.num_local_groups];  // row chunks over all local groups
  const int32_t n_tiles = (p.n + BMW - 1) / BMW;
  const int32_t ksteps = p.k / KS;                     // k % 128 == 0 on this path (k % 256 for 4-bit)
  const int32_t nb = p.scale != nullptr ? p.num_blocks : 1;
  const int32_t s_per_block = ksteps / nb;             // (k / nb) % 128 == 0 on this path
  const int32_t total = t_tiles * n_tiles;
  auto item_of = [&](int32_t w) {
    return decode_gemm_tile(w, t_tiles, n_tiles, n_tiles, tiles, offs, go, p.num_local_groups, BT);
  };
  auto chunk_rows = [&](const GemmTile& t) { return min(t.row_end - t.row0, int32_t(BT)); };
  // Step j's converted / operand stage is reused by step j + depth once step j's MMAs are done.
  auto wait_step_done = [&](uint32_t j, int depth) {
    return j < uint32_t(depth) ||
           wait_bar(stepdone_bar((j - depth) % NDONE), ((j - depth) / NDONE) & 1u, abort_flag, p.err);
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producers
    // Weight boxes: one per step (per two steps of 4-bit codes).
    if (lane == 0) {
      uint32_t apend = 0, apar = 0;  // slots with a copy in flight, and their phases
      uint32_t bx = 0;               // boxes over the CTA's items
      bool ok = true;
      for (int32_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
        const GemmTile t = item_of(w);
        for (int32_t ks = 0; ks < ksteps; ks += STEPS_PER_RAW, ++bx) {
          const uint32_t as = bx % RAWST, aph = (bx / RAWST) & 1u;
          if (!wait_bar(rawempty_bar(as), aph ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(rawfull_bar(as), kNv ? RAW_STAGE : RAW_BYTES);
          tma_load_3d(sbase + OFF_RAW + as * RAW_STAGE, &tm_rhs, rawfull_bar(as), (ks / STEPS_PER_RAW) * 128,
                      t.n_tile * BMW, t.local_group);
          if constexpr (kNv)  // the box's block scales: 16 bytes of each of its 128 weight rows
            tma_load_3d(sbase + OFF_RAW + as * RAW_STAGE + RAW_BYTES, &tm_bs, rawfull_bar(as),
                        (ks / STEPS_PER_RAW) * 16, t.n_tile * BMW, t.local_group);
          apend |= 1u << as;
          apar = (apar & ~(1u << as)) | (aph << as);
        }
      }
      if (!ok)
        for (int s = 0; s < RAWST; ++s)
          if (apend >> s & 1u) drain_bar(rawfull_bar(s), apar >> s & 1u);
    }
  } else if (warp == kBWarp) {
    // ---------------------------------------------------------------- TMA activation rows
    // Per step the chunk's fp16 rows for 128 k, both 64-wide atoms in one box
    // ({64 k, 16 rows, 2 atoms} over the plane viewed as [k / 64, m, 64]), once
    // the MMAs of step j - BST are done.
    if (lane == 0) {
      uint32_t bpend = 0, bpar = 0;
      uint32_t j = 0;  // the step's index over the CTA's items
      bool ok = true;
      griddep_wait();  // the rows come from the split pass
      for (int32_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
        const GemmTile t = item_of(w);
        for (int32_t ks = 0; ks < ksteps; ++ks, ++j) {
          if (!wait_step_done(j, BST)) {
            ok = false;
            break;
          }
          const uint32_t bs = j % BST, bph = (j / BST) & 1u;
          mbar_arrive_expect_tx(bfull_bar(bs), B_BYTES);
          tma_load_3d(sbase + OFF_B + bs * B_BYTES, &tm_lhs, bfull_bar(bs), 0, t.row0, 2 * ks);
          bpend |= 1u << bs;
          bpar = (bpar & ~(1u << bs)) | (bph << bs);
        }
      }
      if (!ok)
        for (int s = 0; s < BST; ++s)
          if (bpend >> s & 1u) drain_bar(bfull_bar(s), bpar >> s & 1u);
    }
  } else if (warp == 1 || warp == kMma2 || warp == kMma3 || warp == kMma3 + 1) {
    // ---------------------------------------------------------------- MMA issuers
    // Four warps issue MMAs, each every fourth step: in this kernel one
    // thread's waits and issue for a step take far longer than the tensor
    // core needs for the step's MMAs (about 50 cycles of issue per tcgen05.mma
    // per thread, and ~170 per mbarrier check).  Each step has its own
    // operand stage, accumulator slot and commit, so the issuers share nothing.
    constexpr uint32_t kIdesc = idesc_f16(BMW, BT);
    const uint32_t mine = warp == 1 ? 0u : (warp == kMma2 ? 1u : uint32_t(warp - kMma3 + 2));
    bool ok = true;
    uint32_t j = 0;  // the step's index over the CTA's items
    for (int32_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
      for (int32_t ks = 0; ks < ksteps; ++ks, ++j) {
        if ((j & uint32_t(kIssuers - 1)) != mine) continue;
        const uint32_t cs = j % CST, bs = j % BST, slot = j % kNacc;
        if (!wait_bar(acce_bar(slot), ((j / kNacc) & 1u) ^ 1u, abort_flag, p.err) ||
            !wait_bar(convfull_bar(cs), (j / CST) & 1u, abort_flag, p.err) ||
            !wait_bar(bfull_bar(bs), (j / BST) & 1u, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a0 = tmem_base + A_COL0 + cs * A_COLS;
          const uint32_t b0 = sbase + OFF_B + bs * B_BYTES;
          const uint32_t d = tmem_base + slot * kSlotCols;
#pragma unroll
          for (int kk = 0; kk < KS / 16; ++kk) {
            const uint32_t atom = uint32_t(kk >> 2), off = uint32_t(kk & 3) * 32u;
            const uint64_t bd = sw128_desc(b0 + atom * B_ATOM + off, 16, 1024);
            if constexpr (kMx)  // 32-k block kk / 2 into its own 16 columns
              mma_f16_ts(d + uint32_t(BT) * uint32_t(kk >> 1), a0 + 8u * kk, bd, kIdesc, uint32_t(kk & 1));
            else
              mma_f16_ts(d, a0 + 8u * kk, bd, kIdesc, kk != 0 ? 1u : 0u);
          }
          mma_commit(stepdone_bar(j % NDONE));
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
    const int quarter = warp & 3;
    const int wrow = quarter * 32 + lane;  // weight row in the tile = output column
    const uint32_t lane_base = uint32_t(quarter * 32) << 16;
    uint32_t slot = 0, ds = 0, dph = 0, sc = 0, scph = 0;
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
        for (int32_t ks = 0; ks < ksteps && ok; ++ks) {
          if (!wait_bar(stepdone_bar(ds), dph, abort_flag, p.err) || !wait_bar(sfull_bar(sc), scph, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float* ts = tscale + sc * SC_PER;
          const uint8_t* wsc = reinterpret_cast<const uint8_t*>(ts + SC_TOK);
          const float sw = p.scale == nullptr ? 1.f
                           : p.scale_e8m0   ? fp8::e8m0_value(wsc[wrow])
                                            : reinterpret_cast<const float*>(wsc)[wrow];
          if constexpr (kMx) {
            // the four 32-k blocks' sums, two per load: D_q * sc_i is the block's partial
            // sum, times its power of two (and the quant block's weight scale)
            const uint32_t e4 = reinterpret_cast<const uint32_t*>(ts + SC_MX)[wrow];
            const uint32_t col0 = tmem_base + lane_base + slot * kSlotCols;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const float u0 = sw * fp8::e8m0_value((e4 >> (16 * h)) & 255u);
              const float u1 = sw * fp8::e8m0_value((e4 >> (16 * h + 8)) & 255u);
              float d[2 * BT];
              fp8::tmem_ld_cols<2 * BT>(col0 + uint32_t(2 * BT * h), d);
#pragma unroll
              for (int i = 0; i < T8; ++i) acc[i] = fmaf(u1, ts[i] * d[BT + i], fmaf(u0, ts[i] * d[i], acc[i]));
            }
          } else {
            float d[T8];
            fp8::tmem_ld_cols<T8>(tmem_base + lane_base + slot * SLOT_COLS, d);
#pragma unroll
            for (int i = 0; i < T8; ++i) acc[i] = fmaf(sw * ts[i], d[i], acc[i]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(acce_bar(slot));
            mbar_arrive(sempty_bar(sc));
          }
          if (++slot == uint32_t(kNacc)) slot = 0;
          if (++ds == NDONE) {
            ds = 0;
            dph ^= 1u;
          }
          if (++sc == NSC) {
            sc = 0;
            scph ^= 1u;
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
      if (fp8::t8_of(chunk_rows(t)) == 8)
        run(std::integral_constant<int, 8>{});
      else
        run(std::integral_constant<int, 16>{});
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
  } else if (warp == 6 || warp == kScale2) {
    // ---------------------------------------------------------------- scales
    // Per step: the chunk rows' split scales (lhs_scale[row, step, 0]; 0 past
    // the chunk), one 4-byte asynchronous copy per row, and the weight scales
    // of the step's quant block for the item's 128 columns, as stored (a bulk
    // copy; E8M0 rows of n % 16 != 0 bytes loaded by this warp), all landing on
    // the slot's full barrier.  The warp waits for no load.  Warp 6 serves the
    // even steps, warp kScale2 the odd ones.
    griddep_wait();  // the split scales come from the kernel before
    const uint32_t mine = warp == 6 ? 0u : 1u;
    uint32_t wpend = 0, wpar = 0;
    bool ok = true;
    const int esz = p.scale_e8m0 ? 1 : 4;
    const bool bulk = (p.n * esz) % 16 == 0 && reinterpret_cast<uintptr_t>(p.scale) % 16 == 0;
    int32_t w = blockIdx.x, ks = 0;
    uint32_t j = 0;  // the step's index over the CTA's items
    GemmTile t = w < total ? item_of(w) : GemmTile{};
    // the item's weight-scale row of the current quant block, and the step's place in that block
    const int64_t block_pitch = int64_t(p.n) * esz;
    int64_t wrow = 0;  // byte offset into p.scale
    int32_t kb = 0;
    auto item_start = [&]() {
      wrow = (int64_t(t.local_group) * nb * p.n + int64_t(t.n_tile) * BMW) * esz;
      kb = 0;
    };
    auto step_fwd = [&]() {
      ++j;
      if (++kb == s_per_block) {
        kb = 0;
        wrow += block_pitch;
      }
      if (++ks == ksteps) {
        ks = 0;
        w += gridDim.x;
        if (w < total) {
          t = item_of(w);
          item_start();
        }
      }
    };
    if (w < total) item_start();
    if (mine == 1u && w < total) step_fwd();
    while (w < total) {
      const uint32_t sc = j % NSC, scph = (j / NSC) & 1u;
      if (!wait_bar(sempty_bar(sc), scph ^ 1u, abort_flag, p.err)) {
        ok = false;
        break;
      }
      if (lane < BT) {
        if (lane < chunk_rows(t))
          cp_async_4(smem_u32(tscale + sc * SC_PER + lane), p.lhs_scale + (int64_t(t.row0 + lane) * ksteps + ks) * 2);
        else
          tscale[sc * SC_PER + lane] = 0.f;
      }
      if constexpr (kMx) {
        // the step's 4 E8M0 bytes of each of the item's weight rows (rows of k / 32
        // bytes; k % 128 == 0, so each copy is 4-byte aligned)
        const int32_t cols = min(BMW, p.n - t.n_tile * BMW);
        const int64_t pitch = p.k / 32;
        const uint8_t* src = p.w_block_scale + (int64_t(t.local_group) * p.n + int64_t(t.n_tile) * BMW) * pitch + 4 * ks;
        uint32_t* dst = reinterpret_cast<uint32_t*>(tscale + sc * SC_PER + SC_MX);
#pragma unroll
        for (int q = 0; q < BMW / 32; ++q) {
          const int c = lane + 32 * q;
          if (c < cols)
            cp_async_4(smem_u32(dst + c), src + c * pitch);
          else
            dst[c] = 0u;
        }
      }
      cp_async_mbar_arrive(sfull_bar(sc));
      uint32_t wbytes = 0;
      if (p.scale != nullptr) {
        const int32_t cols = min(BMW, p.n - t.n_tile * BMW);
        const uint8_t* src = static_cast<const uint8_t*>(p.scale) + wrow;
        const uint32_t dst = smem_u32(tscale + sc * SC_PER + SC_TOK);
        if (bulk) {
          wbytes = uint32_t(cols * esz);  // a multiple of 16: n % 8 == 0 (f32) or n % 16 == 0 (E8M0)
          if (lane == 0) bulk_load(dst, src, wbytes, sfull_bar(sc));
        } else {
          uint8_t* d8 = reinterpret_cast<uint8_t*>(tscale + sc * SC_PER + SC_TOK);
          for (int c = lane; c < cols * esz; c += 32) d8[c] = __ldg(src + c);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(sfull_bar(sc), wbytes);
      if (wbytes != 0u) {
        wpend |= 1u << sc;
        wpar = (wpar & ~(1u << sc)) | (scph << sc);
      }
      step_fwd();
      if (w < total) step_fwd();
    }
    cp_async_wait_all();  // this thread's scale copies have landed
    // a wait gave up: the weight-scale copies still in flight land before exit
    if (!ok && lane == 0)
      for (int s2 = 0; s2 < NSC; ++s2)
        if (wpend >> s2 & 1u) drain_bar(sfull_bar(s2), wpar >> s2 & 1u);
  } else if (warp >= kConvWarp0 && warp < kConvWarp0 + kConvWarps) {
    // ---------------------------------------------------------------- weight rewrite
    // Thread t rewrites part t / 128 of weight row r = t % 128 of each step's
    // raw codes as fp16 into TMEM lane r (two threads per row, so that each SM
    // sub-partition has two rewrite warps to interleave).  Raw rows are 128
    // bytes, 128-byte swizzled (16-byte chunk j of row r at position j ^ (r % 8));
    // A column 4 q + i holds word i of the row's 16-byte fp16 chunk q (8 k).
    // int8 and e4m3: raw chunk c (16 codes) becomes A chunks 2c and 2c + 1.
    // 4-bit: raw chunk 4 h + c of the box (step h of its two) becomes A chunks
    // 4c .. 4c + 3.  Either way part p writes columns 32 p .. 32 p + 31.
    const int r = (warp & 3) * 32 + lane, part = (warp - kConvWarp0) >> 2;
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    uint32_t rs = 0, rph = 0, cs = 0;
    uint32_t j = 0;  // steps rewritten so far
    bool ok = true;
    for (int32_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
      for (int32_t ks = 0; ks < ksteps; ++ks) {
        const int h = ks % STEPS_PER_RAW;
        if ((h == 0 && !wait_bar(rawfull_bar(rs), rph, abort_flag, p.err)) || !wait_step_done(j, CST)) {
          ok = false;
          break;
        }
        tc_fence_after();  // the MMAs that read this A stage are complete
        const uint32_t src = sbase + OFF_RAW + rs * RAW_STAGE + uint32_t(r) * 128u;
        const uint32_t sw = uint32_t(r & 7);
        uint32_t o[32];
        if constexpr (k4) {
          constexpr int kC = 4 / kParts;
          uint32_t x[kC][4];
#pragma unroll
          for (int cc = 0; cc < kC; ++cc)
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(x[cc][0]), "=r"(x[cc][1]), "=r"(x[cc][2]), "=r"(x[cc][3])
                         : "r"(src + ((uint32_t(4 * h + part * kC + cc) ^ sw) << 4)));
          // NVFP4: the scales of the thread's four 16-k blocks (bytes 8 h + 4 part .. + 3
          // of its row in the box's scale rows), each as an fp16 pair
          uint32_t sp[4] = {0u, 0u, 0u, 0u};
          if constexpr (kNv) {
            uint32_t sb, lo, hi;
            asm volatile("ld.shared.b32 %0, [%1];"
                         : "=r"(sb)
                         : "r"(sbase + OFF_RAW + rs * RAW_STAGE + RAW_BYTES + uint32_t(r) * 16u +
                               uint32_t(8 * h + 4 * part)));
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(lo) : "h"(uint16_t(sb)));
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hi) : "h"(uint16_t(sb >> 16)));
            sp[0] = prmt(lo, lo, 0x1010u);
            sp[1] = prmt(lo, lo, 0x3232u);
            sp[2] = prmt(hi, hi, 0x1010u);
            sp[3] = prmt(hi, hi, 0x3232u);
          }
#pragma unroll
          for (int cc = 0; cc < kC; ++cc)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              uint32_t q[4];
              if constexpr (kNv)
                e2m1x8_to_f16(x[cc][u], sp[2 * cc + (u >> 1)], q);  // codes 32 cc + 8 u ..: block 2 cc + u / 2
              else
                nib8_to_f16<F == WFmt::kInt4>(x[cc][u], q);
#pragma unroll
              for (int i = 0; i < 4; ++i) o[16 * cc + 4 * u + i] = q[i];
            }
        } else {
          constexpr int kC = 8 / kParts;
          uint32_t x[kC][4];
#pragma unroll
          for (int cc = 0; cc < kC; ++cc)
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(x[cc][0]), "=r"(x[cc][1]), "=r"(x[cc][2]), "=r"(x[cc][3])
                         : "r"(src + ((uint32_t(part * kC + cc) ^ sw) << 4)));
#pragma unroll
          for (int cc = 0; cc < kC; ++cc)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              if constexpr (kMx)
                e4m3x4_to_f16(x[cc][u], o[8 * cc + 2 * u], o[8 * cc + 2 * u + 1]);
              else
                int8x4_to_f16(x[cc][u], o[8 * cc + 2 * u], o[8 * cc + 2 * u + 1]);
            }
        }
        tmem_st_32cols(tmem_base + lane_base + A_COL0 + cs * A_COLS + 32u * part, o);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        // the raw box is done after its last step (or the item's last, k % 256 == 128)
        const bool box_done = h == STEPS_PER_RAW - 1 || ks + 1 == ksteps;
        if (lane == 0) {
          if (box_done) mbar_arrive(rawempty_bar(rs));
          mbar_arrive(convfull_bar(cs));
        }
        if (box_done && ++rs == RAWST) {
          rs = 0;
          rph ^= 1u;
        }
        if (++cs == CST) cs = 0;
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
  // marked rows: summed again by the last CTA (the split pass marked them)
  fp8::fix_marked_rows<F, true, kOutF32>(p, go, offs, smem + OFF_RAW, KS);
}

template <WFmt F, bool kOutF32>
cudaError_t launch_impl(const ScaledLaunch& L, int grid, cudaStream_t stream) {
  auto kern = gemm_f16w_kernel<F, kOutF32>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(SMEM_BYTES));
  if (e != cudaSuccess) return e;
  constexpr bool k4 = F == WFmt::kInt4 || F == WFmt::kUint4 || F == WFmt::kE2M1;
  Params p{L.group_sizes, L.num_total_groups, L.group_offset, L.num_local_groups, L.m, L.n, L.k, L.scale,
           L.num_blocks, L.bias, L.bias_f32, L.out, L.err, L.zero_rest, L.group_offset_dev, L.scale_e8m0,
           L.lhs_scale, L.num_lhs_blocks, static_cast<const uint16_t*>(L.lhs_raw),
           static_cast<const uint8_t*>(L.rhs_raw), k4 ? int64_t(L.k) / 2 : int64_t(L.k),
           F == WFmt::kE2M1 || F == WFmt::kE4M3 ? L.mx_scale : nullptr};
  // Launched as the programmatic dependent of the split pass just before it in
  // the stream: the prologue and the weight stream overlap that kernel's end.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(unsigned(kThreads));
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, L.tm_lhs, L.tm_rhs, L.tm_bs, p);
}

template <WFmt F>
cudaError_t launch_fmt(const ScaledLaunch& L, bool out_f32, int grid, cudaStream_t stream) {
  return out_f32 ? launch_impl<F, true>(L, grid, stream) : launch_impl<F, false>(L, grid, stream);
}

}  // namespace
}  // namespace f16w

cudaError_t launch_f16w(const ScaledLaunch& p, int weight_format, bool out_f32, int grid, cudaStream_t stream) {
  switch (weight_format) {
    case kWeightInt8: return f16w::launch_fmt<fp8::WFmt::kInt8>(p, out_f32, grid, stream);
    case kWeightInt4: return f16w::launch_fmt<fp8::WFmt::kInt4>(p, out_f32, grid, stream);
    case kWeightUint4: return f16w::launch_fmt<fp8::WFmt::kUint4>(p, out_f32, grid, stream);
    case kWeightE2M1: return f16w::launch_fmt<fp8::WFmt::kE2M1>(p, out_f32, grid, stream);  // NVFP4 (tm_bs)
    case kWeightE4M3:  // MXFP8 only: the E8M0 block scales are required
      if (p.mx_scale == nullptr || reinterpret_cast<uintptr_t>(p.mx_scale) % 4 != 0 || p.k % 128 != 0)
        return cudaErrorInvalidValue;
      return f16w::launch_fmt<fp8::WFmt::kE4M3>(p, out_f32, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gmmk
