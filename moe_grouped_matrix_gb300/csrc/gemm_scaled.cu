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
//   warp 0      TMA: the weight tile and the step's token tile [16 rows x 128 k]
//               (6-deep token ring), well ahead of the MMA.  e4m3: the raw
//               tile [128 n x 128 k] (16 KB) into an 8-deep raw ring; bf16:
//               the tile straight into a shared-memory operand ring.
//   warps 6-21  (e4m3 only) decode the raw tile to bf16 and write it into
//               TMEM with tcgen05.st (lane = weight row), where the MMA reads
//               its A operand; the raw stage is freed as soon as it is read.
//               With A in TMEM the MMA reads only the 512-byte token tile from
//               shared memory, instead of 4 KB of weights per instruction.
//   warp 1      TMEM owner; issues 8 tcgen05.mma 128x16x16 per step into the
//               16 columns of the current quant block; 4 consecutive blocks
//               share one TMEM slot, handed to the epilogue with one commit
//   warps 2-5   per slot: TMEM -> registers, multiply each block's 16 columns by
//               that block's scale for this lane's n, add into fp32 registers;
//               at the end of the item add the bias, round and store
// TMEM columns: accumulator slots [0, 256) (4 slots x 4 blocks x 16); e4m3
// weight stages [256, 512) (2 stages x 128; a 128-wide k step of bf16 fills 64).
//
// e4m3fn -> bf16 is exact: every e4m3fn value is a bf16 value.  The decoder
// places the 7 exponent/mantissa bits of the code at bf16 bits 4..10 (giving
// the bf16 number 2^-120 times the code's value, subnormals included) and
// multiplies by 2^120; the two NaN codes (0x7F, 0xFF) are mapped to NaN.
//
// Microscaling (MXFP8): with an E8M0 scale per 32 consecutive k of a weight
// row, each decoder thread's 32 values of a step are one scale block, and the
// decoded bf16 values are multiplied by the block's power of two, exactly
// while the product stays within bf16's normal range (|w| 2^(e-127) between
// 2^-126 and 2^128).
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "worklist.cuh"

namespace gmmk {
namespace {

constexpr int BMW = 128;  // weight rows (n) per item = MMA M
constexpr int BT = 16;    // tokens per item = MMA N
constexpr int KS = 128;   // k per pipeline step
constexpr int RSTAGES = 8;  // raw e4m3 weight tiles in flight (freed as soon as decoded)
constexpr int BSTAGES = 6;  // token tiles in flight (loaded ahead by the producer)
constexpr int SB = 4;       // quant blocks per TMEM slot (one commit / wait / release per slot)
constexpr int NACC = 4;     // TMEM accumulator slots of SB x 16 columns
constexpr int kConvWarps = 16;
constexpr int kConvThreads = kConvWarps * 32;
constexpr int kMaxGroups = 1024;
constexpr uint32_t A_BYTES = BMW * KS * 2;  // bf16 weight operand in shared memory (bf16 path)
constexpr uint32_t RAW_BYTES = BMW * KS;    // e4m3 tile
constexpr uint32_t B_BYTES = BT * KS * 2;   // token tile: two 64-wide k atoms
constexpr uint32_t SLOT_COLS = SB * BT;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TMEM_A_BASE = NACC * SLOT_COLS;  // 256: e4m3 weight stages start here
constexpr uint32_t TMEM_A_STAGE_COLS = 128;
static_assert(TMEM_A_BASE + 2 * TMEM_A_STAGE_COLS <= TMEM_COLS, "TMEM map");

// Shared-memory layout; the e4m3 path keeps its weight operand in TMEM.
template <bool kE4M3>
struct Layout {
  static constexpr int kOStages = kE4M3 ? 2 : 3;  // weight operand stages (TMEM or shared memory)
  static constexpr uint32_t OFF_A = 0;
  static constexpr uint32_t OFF_B = OFF_A + (kE4M3 ? 0u : uint32_t(kOStages) * A_BYTES);
  static constexpr uint32_t OFF_RAW = OFF_B + BSTAGES * B_BYTES;
  static constexpr uint32_t OFF_CTRL = OFF_RAW + (kE4M3 ? uint32_t(RSTAGES) * RAW_BYTES : 0u);
  static constexpr uint32_t OFF_RFULL = OFF_CTRL;
  static constexpr uint32_t OFF_REMPTY = OFF_RFULL + 8 * RSTAGES;
  static constexpr uint32_t OFF_OFULL = OFF_REMPTY + 8 * RSTAGES;
  static constexpr uint32_t OFF_OEMPTY = OFF_OFULL + 8 * kOStages;
  static constexpr uint32_t OFF_BFULL = OFF_OEMPTY + 8 * kOStages;
  static constexpr uint32_t OFF_BEMPTY = OFF_BFULL + 8 * BSTAGES;
  static constexpr uint32_t OFF_ACCF = OFF_BEMPTY + 8 * BSTAGES;
  static constexpr uint32_t OFF_ACCE = OFF_ACCF + 8 * NACC;
  static constexpr uint32_t OFF_DONE = OFF_ACCE + 8 * NACC;
  static constexpr uint32_t OFF_TMEM = OFF_DONE + 8;
  static constexpr uint32_t OFF_ABORT = OFF_TMEM + 4;
  static constexpr uint32_t OFF_OFFS = OFF_CTRL + 1024;
  static constexpr uint32_t OFF_TILES = OFF_OFFS + 4 * (kMaxGroups + 4);
  static constexpr uint32_t SMEM_USED = OFF_TILES + 4 * (kMaxGroups + 4);
  static constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
  static_assert(OFF_ABORT + 4 <= OFF_OFFS, "control block overlaps the tables");
};

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
  const int32_t* group_offset_dev;  // NULL, or the device scalar that replaces group_offset
  // Microscaling block scales [L, n, k / block] of the weights: MXFP8 (e4m3
  // weights) E8M0 per 32 k, or NULL; NVFP4 (e2m1 weights) e4m3 per 16 k.
  const uint8_t* mx_scale;
};

// bf16x2 holding 2^(e - 127) twice, the value of an E8M0 byte (page
// "gemm_quant.rs", widen_block_scale_f32: e = 0 is 2^-127, e = 255 is 0).
__device__ __forceinline__ uint32_t e8m0_bf16x2(uint32_t e) {
  const uint32_t b = e == 255u ? 0u : (e == 0u ? 0x0040u : e << 7);
  return b | (b << 16);
}

// bf16x2 holding an e4m3fn value twice (exact: every e4m3fn value is a bf16 value).
__device__ __forceinline__ uint32_t e4m3_bf16x2(uint32_t code) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(uint16_t(code)));
  const float f = __half2float(__ushort_as_half(uint16_t(h)));
  const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(f));
  return b | (b << 16);
}

// 32 e2m1 codes (16 bytes, the even k in the low nibble) -> 32 bf16 (16 words,
// k order: words 0..7 in lo, 8..15 in hi), the first 16 times s_lo and the
// last 16 times s_hi (bf16x2 scale factors).  Per 4 codes (16 bits, k order):
// two byte permutes look the high and low bytes of each code's bf16 value up
// in 8-entry tables indexed by the code's magnitude bits, a third replicates
// each code's sign into a mask whose bit 7 per byte is the sign, and two more
// interleave low and high bytes into two bf16x2 words.  The bf16x2 fma by the
// block scale is exact (an e2m1 value times an e4m3 value has at most 6
// significant bits).
__device__ __forceinline__ void decode_fp4_32(const uint4 raw, uint32_t s_lo, uint32_t s_hi, uint32_t (&lo)[8],
                                              uint32_t (&hi)[8]) {
  // bf16 of the magnitudes 0, 0.5, 1, 1.5 | 2, 3, 4, 6: high bytes, low bytes
  constexpr uint32_t kH0 = 0x3F3F3F00u, kH1 = 0x40404040u;
  constexpr uint32_t kL0 = 0xC0800000u, kL1 = 0xC0804000u;
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const uint32_t codes = half == 0 ? w[i] : (w[i] >> 16);
      const uint32_t idx = codes & 0x7777u;
      // prmt's default mode: a selector nibble with bit 3 set replicates the
      // selected byte's sign, giving 0xFF for negative codes and 0x80 otherwise
      uint32_t rep;
      asm("prmt.b32 %0, %1, %2, %3;" : "=r"(rep) : "r"(0x80808080u), "r"(0x80808080u), "r"(codes));
      const uint32_t sign = (rep << 1) & 0x80808080u;
      const uint32_t hb = __byte_perm(kH0, kH1, idx) | sign;
      const uint32_t lb = __byte_perm(kL0, kL1, idx);
      const uint32_t s2 = i < 2 ? s_lo : s_hi;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        uint32_t y = __byte_perm(lb, hb, j == 0 ? 0x5140u : 0x7362u);
        asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(y) : "r"(y), "r"(s2), "r"(0x80008000u));
        const int word = 4 * i + 2 * half + j;  // values 2 word, 2 word + 1
        if (word < 8)
          lo[word] = y;
        else
          hi[word - 8] = y;
      }
    }
  }
}

// 16 e4m3fn codes (one 16-byte chunk, lowest k first) -> 16 bf16 (8 words).
// Per 4 codes, magnitudes (low 7 bits) and signs are split once; per pair of
// codes two byte permutes put the magnitudes at bits 0..6 / 16..22 and the
// signs at bits 15 / 31, and one integer multiply-add (x16) moves the
// magnitudes to bf16 bits 4..10 under their signs: a bf16 number equal to
// 2^-120 times the code's value, subnormal codes included.  A bf16x2 fma then
// multiplies by 2^120 exactly (adding -0 keeps the sign of zero).  The two NaN
// codes (magnitude 0x7F) would come out as +-480: magnitude + 1 carries into
// bit 7 only for them, so one add per 4 codes finds a chunk holding one, which
// is fixed on a separate, rarely taken path.
__device__ __forceinline__ void decode16(const uint4 raw, uint32_t (&o)[8]) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  uint32_t nan_any = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t mag = w[i] & 0x7F7F7F7Fu;
    const uint32_t sgn = w[i] & 0x80808080u;
    nan_any |= (mag + 0x01010101u) & 0x80808080u;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t mp = __byte_perm(mag, 0u, h == 0 ? 0x4140u : 0x4342u);
      const uint32_t sp = __byte_perm(sgn, 0u, h == 0 ? 0x1404u : 0x3424u);
      const uint32_t x = mp * 16u + sp;
      uint32_t y;
      asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(y) : "r"(x), "r"(0x7B807B80u), "r"(0x80008000u));
      o[2 * i + h] = y;
    }
  }
  if (nan_any != 0u) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t lo = (w[i] >> (16 * h)) & 0x7Fu, hi = (w[i] >> (16 * h + 8)) & 0x7Fu;
        if (lo == 0x7Fu) o[2 * i + h] = (o[2 * i + h] & 0xFFFF0000u) | 0x7FC0u;
        if (hi == 0x7Fu) o[2 * i + h] = (o[2 * i + h] & 0x0000FFFFu) | 0x7FC00000u;
      }
    }
  }
}

// kE4M3: weights decoded to bf16 by the decoder warps, e4m3 codes, or (kFp4)
// e2m1 codes two per byte with an e4m3 scale per 16 k (NVFP4).
template <bool kE4M3, bool kFp4, bool kOutF32>
__global__ void __launch_bounds__(kE4M3 ? 192 + kConvThreads : 192, 1)
    gemm_scaled_kernel(const __grid_constant__ CUtensorMap tm_lhs, const __grid_constant__ CUtensorMap tm_rhs,
                       const Params p) {
  static_assert(kE4M3 || !kFp4, "4-bit weights are decoded");
  using L = Layout<kE4M3>;
  constexpr int OSTAGES = L::kOStages;
  int32_t go;
  if (!resolve_group_offset(p.group_offset_dev, p.group_offset, p.num_total_groups, p.num_local_groups, p.err, go))
    return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::OFF_ABORT);
  int32_t* offs = reinterpret_cast<int32_t*>(smem + L::OFF_OFFS);
  int32_t* tiles = reinterpret_cast<int32_t*>(smem + L::OFF_TILES);
  auto rfull_bar = [&](uint32_t s) { return sbase + L::OFF_RFULL + 8 * s; };
  auto rempty_bar = [&](uint32_t s) { return sbase + L::OFF_REMPTY + 8 * s; };
  auto ofull_bar = [&](uint32_t s) { return sbase + L::OFF_OFULL + 8 * s; };
  auto oempty_bar = [&](uint32_t s) { return sbase + L::OFF_OEMPTY + 8 * s; };
  auto bfull_bar = [&](uint32_t s) { return sbase + L::OFF_BFULL + 8 * s; };
  auto bempty_bar = [&](uint32_t s) { return sbase + L::OFF_BEMPTY + 8 * s; };
  auto accf_bar = [&](uint32_t b) { return sbase + L::OFF_ACCF + 8 * b; };
  auto acce_bar = [&](uint32_t b) { return sbase + L::OFF_ACCE + 8 * b; };
  const uint32_t done_bar = sbase + L::OFF_DONE;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < RSTAGES; ++s) {
      mbar_init(rfull_bar(s), 1);
      mbar_init(rempty_bar(s), kConvWarps);
    }
    for (int s = 0; s < OSTAGES; ++s) {
      // e4m3: one arrive per decoder warp; bf16: the producer's expect_tx.
      mbar_init(ofull_bar(s), kE4M3 ? kConvWarps : 1);
      mbar_init(oempty_bar(s), 1);
    }
    for (int s = 0; s < BSTAGES; ++s) {
      mbar_init(bfull_bar(s), 1);
      mbar_init(bempty_bar(s), 1);
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
    tmem_alloc(sbase + L::OFF_TMEM, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 2) {
    build_group_offsets(p.group_sizes, p.num_total_groups, p.m, offs, p.err);
    build_tile_prefix(offs, go, p.num_local_groups, BT, tiles);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + L::OFF_TMEM);

  const int32_t t_tiles = tiles[p.num_local_groups];  // token chunks over all local groups
  const int32_t n_tiles = (p.n + BMW - 1) / BMW;
  const int32_t ksteps = p.k / KS;                     // k % 128 == 0 on this path
  const int32_t nb = p.scale != nullptr ? p.num_blocks : 1;
  const int32_t steps_per_block = ksteps / nb;         // (k / nb) % 128 == 0 on this path
  const int32_t total = t_tiles * n_tiles;
  // Items: token chunks outer, the weight tiles of the chunk's group inner.
  auto item_of = [&](int32_t w) {
    return decode_gemm_tile(w, t_tiles, n_tiles, n_tiles, tiles, offs, go, p.num_local_groups, BT);
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    // Per k step: the weight tile (e4m3: raw, into the 6-deep raw ring for the
    // decoders; bf16: straight into the operand ring) and the token tile (into
    // the 6-deep token ring), both well ahead of the MMA.
    if (lane == 0) {
      constexpr int WS = kE4M3 ? RSTAGES : OSTAGES;
      uint32_t ws = 0, wphase = 0, bs = 0, bphase = 0, wpend = 0, bpend = 0;
      uint32_t wpar[WS], bpar[BSTAGES];
      bool ok = true;
      for (int32_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
        const GemmTile t = item_of(w);
        for (int32_t ks = 0; ks < ksteps; ++ks) {
          const uint32_t wempty = kE4M3 ? rempty_bar(ws) : oempty_bar(ws);
          if (!wait_bar(wempty, wphase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          if constexpr (kE4M3) {
            // e2m1: 64 bytes a row ({64 bytes, 128 rows} box, rows 64 bytes apart)
            const uint32_t fb = rfull_bar(ws);
            mbar_arrive_expect_tx(fb, kFp4 ? RAW_BYTES / 2 : RAW_BYTES);
            tma_load_3d(sbase + L::OFF_RAW + ws * RAW_BYTES, &tm_rhs, fb, kFp4 ? ks * (KS / 2) : ks * KS,
                        t.n_tile * BMW, t.local_group);
          } else {
            const uint32_t fb = ofull_bar(ws);
            mbar_arrive_expect_tx(fb, A_BYTES);
#pragma unroll
            for (int h = 0; h < 2; ++h)
              tma_load_3d(sbase + L::OFF_A + ws * A_BYTES + h * (A_BYTES / 2), &tm_rhs, fb, ks * KS + 64 * h,
                          t.n_tile * BMW, t.local_group);
          }
          wpar[ws] = wphase;
          wpend |= 1u << ws;
          if (++ws == WS) {
            ws = 0;
            wphase ^= 1u;
          }
          if (!wait_bar(bempty_bar(bs), bphase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const uint32_t bb = bfull_bar(bs);
          mbar_arrive_expect_tx(bb, B_BYTES);
#pragma unroll
          for (int h = 0; h < 2; ++h)
            tma_load_2d(sbase + L::OFF_B + bs * B_BYTES + h * (B_BYTES / 2), &tm_lhs, bb, ks * KS + 64 * h, t.row0);
          bpar[bs] = bphase;
          bpend |= 1u << bs;
          if (++bs == BSTAGES) {
            bs = 0;
            bphase ^= 1u;
          }
        }
      }
      if (!ok) {
        for (int s = 0; s < WS; ++s)
          if (wpend >> s & 1u) drain_bar(kE4M3 ? rfull_bar(s) : ofull_bar(s), wpar[s]);
        for (int s = 0; s < BSTAGES; ++s)
          if (bpend >> s & 1u) drain_bar(bfull_bar(s), bpar[s]);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    // Quant block b of an item accumulates into columns [16 (b % SB), +16) of
    // TMEM slot (b / SB); a slot is committed to the epilogue once its SB
    // blocks (or the item's last ones) are done.
    constexpr uint32_t kIdesc = idesc_bf16(BMW, BT, false, false);
    uint32_t stage = 0, phase = 0, bs = 0, bphase = 0, slot = 0, slot_phase = 0;
    bool ok = true;
    for (int32_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
      for (int32_t b0 = 0; b0 < nb && ok; b0 += SB) {
        if (!wait_bar(acce_bar(slot), slot_phase ^ 1u, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int32_t nblk = min(SB, nb - b0);
        for (int32_t bi = 0; bi < nblk && ok; ++bi) {
          const uint32_t d_tmem = tmem_base + slot * SLOT_COLS + uint32_t(bi) * BT;
          for (int32_t st = 0; st < steps_per_block; ++st) {
            if (!wait_bar(ofull_bar(stage), phase, abort_flag, p.err) ||
                !wait_bar(bfull_bar(bs), bphase, abort_flag, p.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            if (lane == 0) {
              const uint32_t a0 = sbase + L::OFF_A + stage * A_BYTES;
              const uint32_t a_tmem = tmem_base + TMEM_A_BASE + stage * TMEM_A_STAGE_COLS;
              const uint32_t b0s = sbase + L::OFF_B + bs * B_BYTES;
#pragma unroll
              for (int kk = 0; kk < KS / 16; ++kk) {
                const int h = kk >> 2;
                const uint64_t bd = sw128_desc(b0s + h * (B_BYTES / 2) + (kk & 3) * 32, 16, 1024);
                if constexpr (kE4M3) {
                  // k [16 kk, 16 kk + 16) of the 128 weight rows: 8 TMEM columns
                  mma_bf16_ts(d_tmem, a_tmem + uint32_t(kk) * 8u, bd, kIdesc, (st | kk) != 0 ? 1u : 0u);
                } else {
                  const uint64_t ad = sw128_desc(a0 + h * (A_BYTES / 2) + (kk & 3) * 32, 16, 1024);
                  mma_bf16_ss(d_tmem, ad, bd, kIdesc, (st | kk) != 0 ? 1u : 0u);
                }
              }
              mma_commit(oempty_bar(stage));
              mma_commit(bempty_bar(bs));
            }
            __syncwarp();
            if (++stage == OSTAGES) {
              stage = 0;
              phase ^= 1u;
            }
            if (++bs == BSTAGES) {
              bs = 0;
              bphase ^= 1u;
            }
          }
        }
        if (!ok) break;
        if (lane == 0) mma_commit(accf_bar(slot));
        __syncwarp();
        if (++slot == NACC) {
          slot = 0;
          slot_phase ^= 1u;
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
      // The item's scales (one per quant block for this lane's column) and its
      // bias are first-touch DRAM reads: issue them kPre blocks ahead so their
      // latency is paid once per kPre blocks, not once per block.
      constexpr int kPre = 8;
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
      static_assert(kPre % SB == 0, "a prefetch chunk holds whole slots");
      float s_cur[kPre], s_next[kPre];
      load_scales(0, s_cur);
      for (int32_t c0 = 0; c0 < nb && ok; c0 += kPre) {
        load_scales(c0 + kPre, s_next);
#pragma unroll
        for (int sb = 0; sb < kPre / SB; ++sb) {
          const int32_t b0 = c0 + sb * SB;
          if (b0 >= nb) break;
          if (!wait_bar(accf_bar(slot), slot_phase, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int bi = 0; bi < SB; ++bi) {
            if (b0 + bi >= nb) break;
            uint32_t v[BT];
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
                "tcgen05.wait::ld.sync.aligned;"
                : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                  "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
                  "=r"(v[15])
                : "r"(tmem_base + (uint32_t(quarter * 32) << 16) + slot * SLOT_COLS + uint32_t(bi) * BT)
                : "memory");
#pragma unroll
            for (int i = 0; i < BT; ++i) acc[i] = fmaf(s_cur[sb * SB + bi], __uint_as_float(v[i]), acc[i]);
          }
          tc_fence_before();
          mbar_arrive(acce_bar(slot));
          if (++slot == NACC) {
            slot = 0;
            slot_phase ^= 1u;
          }
        }
#pragma unroll
        for (int j = 0; j < kPre; ++j) s_cur[j] = s_next[j];
      }
      if (!ok) break;
      if (!col_ok) continue;
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
  } else if constexpr (kE4M3) {
    // ---------------------------------------------------------------- e4m3 -> bf16 decoders
    // Decoder warp dw (0..15) may only touch the TMEM lanes of its quarter
    // q = warp % 4; its thread owns weight row r = 32 q + lane and decodes the
    // two 16-byte raw chunks c = 2 (dw / 4) and c + 1 of that row (k [16 c, 16 c
    // + 16)).  Raw row r holds its 8 chunks at positions c ^ (r % 8), so the 8
    // lanes of each quarter-warp hit 8 different positions.  The 16 decoded bf16
    // of chunk c (two per 32-bit column, k order) go to TMEM columns
    // [8 c, 8 c + 8) of the operand stage, on the thread's own lane.  A raw
    // stage goes back to the TMA producer as soon as every decoder warp holds
    // its part in registers.
    const int dw = warp - 6;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int c0 = 2 * (dw >> 2);
    const uint32_t lane_base = uint32_t(quarter * 32) << 16;
    const int32_t mx_per_row = p.k / (kFp4 ? 16 : 32);
    uint32_t rs = 0, rphase = 0, os = 0, ophase = 0;
    bool ok = true;
    for (int32_t w = blockIdx.x; w < total && ok; w += gridDim.x) {
      // this thread's weight row in the group's rhs, for its MX scales
      const uint8_t* mx_row = nullptr;
      if (p.mx_scale != nullptr) {
        const GemmTile t = item_of(w);
        const int32_t wr = t.n_tile * BMW + row;
        // MXFP8: block 4 ks + c0 / 2 holds this thread's 32 values of step ks;
        // NVFP4: blocks 8 ks + c0 and + 1 hold them
        if (wr < p.n) mx_row = p.mx_scale + (int64_t(t.local_group) * p.n + wr) * mx_per_row + (kFp4 ? c0 : c0 / 2);
      }
      for (int32_t ks = 0; ks < ksteps; ++ks) {
        uint32_t mx = 127u, s_lo = 0x3F803F80u, s_hi = 0x3F803F80u;  // scales of 1
        if constexpr (kFp4) {
          if (mx_row != nullptr) {
            s_lo = e4m3_bf16x2(__ldg(mx_row + 8 * ks));
            s_hi = e4m3_bf16x2(__ldg(mx_row + 8 * ks + 1));
          }
        } else {
          if (mx_row != nullptr) mx = uint32_t(__ldg(mx_row + 4 * ks));
        }
        if (!wait_bar(rfull_bar(rs), rphase, abort_flag, p.err) ||
            !wait_bar(oempty_bar(os), ophase ^ 1u, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tcol = tmem_base + lane_base + TMEM_A_BASE + os * TMEM_A_STAGE_COLS;
        if constexpr (kFp4) {
          // the row's 16-byte chunk c0 / 2 (k [16 c0, 16 c0 + 32)), unswizzled 64-byte rows
          uint4 raw;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(raw.x), "=r"(raw.y), "=r"(raw.z), "=r"(raw.w)
                       : "r"(sbase + L::OFF_RAW + rs * RAW_BYTES + uint32_t(row) * 64u + uint32_t(c0 / 2) * 16u));
          uint32_t lo[8], hi[8];
          decode_fp4_32(raw, s_lo, s_hi, lo, hi);
          tmem_st_8cols(tcol + uint32_t(c0) * 8u, lo);
          tmem_st_8cols(tcol + uint32_t(c0 + 1) * 8u, hi);
        } else {
        const uint32_t raw0 = sbase + L::OFF_RAW + rs * RAW_BYTES + uint32_t(row) * 128u;
        uint4 raw[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int c = c0 + i;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(raw[i].x), "=r"(raw[i].y), "=r"(raw[i].z), "=r"(raw[i].w)
                       : "r"(raw0 + (uint32_t(c ^ (row & 7)) << 4)));
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          uint32_t o[8];
          decode16(raw[i], o);
          if (p.mx_scale != nullptr) {
            const uint32_t s2 = e8m0_bf16x2(mx);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(o[j]) : "r"(o[j]), "r"(s2), "r"(0x80008000u));
          }
          tmem_st_8cols(tcol + uint32_t(c0 + i) * 8u, o);
        }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(rempty_bar(rs));
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(ofull_bar(os));
        if (++rs == RSTAGES) {
          rs = 0;
          rphase ^= 1u;
        }
        if (++os == OSTAGES) {
          os = 0;
          ophase ^= 1u;
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

template <bool kE4M3, bool kFp4, bool kOutF32>
cudaError_t launch_impl(const ScaledLaunch& L, int grid, cudaStream_t stream) {
  auto kern = gemm_scaled_kernel<kE4M3, kFp4, kOutF32>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(Layout<kE4M3>::SMEM_BYTES));
  if (e != cudaSuccess) return e;
  const auto* scale = static_cast<const float*>(L.scale);
  Params p{L.group_sizes, L.num_total_groups, L.group_offset, L.num_local_groups, L.m, L.n, L.k, scale,
           L.num_blocks, L.bias, L.bias_f32, L.out, L.err, L.zero_rest, L.group_offset_dev, L.mx_scale};
  kern<<<grid, kE4M3 ? 192 + kConvThreads : 192, Layout<kE4M3>::SMEM_BYTES, stream>>>(L.tm_lhs, L.tm_rhs, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_scaled(const ScaledLaunch& p, bool rhs_e4m3, bool out_f32, int grid, cudaStream_t stream) {
  if (rhs_e4m3)
    return out_f32 ? launch_impl<true, false, true>(p, grid, stream) : launch_impl<true, false, false>(p, grid, stream);
  return out_f32 ? launch_impl<false, false, true>(p, grid, stream) : launch_impl<false, false, false>(p, grid, stream);
}

cudaError_t launch_scaled_nvfp4(const ScaledLaunch& p, bool out_f32, int grid, cudaStream_t stream) {
  return out_f32 ? launch_impl<true, true, true>(p, grid, stream) : launch_impl<true, true, false>(p, grid, stream);
}

}  // namespace gmmk
