// Grouped matrix multiplication oracle: TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, fp64 CPU statement of what the grouped matmul computes.  It is
// used by the tests, by __graft_entry__.smoke() and by the CPU-baseline leg of
// bench.py to check and time the CUDA library; nothing in the product path may
// link or call it.  It shares no code, header, table or helper with the CUDA
// library.
//
// Sources (page "tpu-inference 0.12.0.dev20251213 -> 0.13.2.dev20251230",
// files tpu_inference/kernels/megablox/gmm.py and common.py; common.py's
// assert_is_supported_dtype lists the operand formats bf16, f32, e4m3fn, e5m2,
// int8, int4, e2m1fn and uint4):
//   * gmm docstring: row block of group i of lhs [m,k] times the group's rhs;
//     rhs is [num_groups, n, k] and the contraction is over the last dim of both
//     operands (the dot_general in the kernel body contracts dim 1 with dim 1).
//   * make_group_metadata: group offsets are the exclusive cumulative sum of
//     group_sizes (CSR-style row offsets).
//   * kernel body (_accum): fp32 accumulation; on the last k tile of quant block
//     b the block's partial sum is multiplied by rhs_scale[g, b, 0, n]; the bias
//     rhs_bias[g, 0, n] is added once (with the first block).
//   * rhs index is group_id - group_offset (rhs_transform_indices), and rows
//     outside the groups [group_offset, group_offset + num_local_groups) are
//     zero (_zero_uninitialized_memory).
// Readings where the pages are silent (all of them listed in the design notes):
//   * rows at or beyond sum(group_sizes) are zero;
//   * negative group sizes count as 0 and offsets are capped at m;
//   * transpose_rhs = 1 means rhs is [G, n, k] (the pages' layout), 0 means
//     rhs is [G, k, n];
//   * tgmm(lhs, dout)[g, k, n] = sum over the rows r of group g of
//     lhs[r, k] * dout[r, n]; an empty group gives a zero block (the
//     visit_empty_groups note in make_group_metadata).
//
// Every result is exact-product, fp64-sum.  Alongside the value `ref` the
// oracle returns `mag`, the same sum taken over absolute values, which the
// tolerance |gpu - ref| <= 1e-3 * mag + 2^-8 * |ref| is stated in.
//
// Pins: tests/test_oracle_pins.py checks this file against hand-worked values,
// brute-force dense per-group products, the format definitions of e4m3fn,
// e5m2, int8, int4, uint4 and e2m1 (and PyTorch's own conversions where it
// has them), and
// the invariants of the method (zero tail rows, empty groups, NT == NN on the
// transposed weight, tgmm == per-group lhs_g^T dout_g, group_offset slicing).

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// Stored formats.  The 4-bit ones hold two values per byte, the even-indexed
// value in the low nibble; element i of such an array is nibble i % 2 of byte
// i / 2.
enum { DT_BF16 = 0, DT_F32 = 1, DT_E4M3 = 2, DT_E5M2 = 3, DT_INT8 = 4, DT_INT4 = 5, DT_UINT4 = 6, DT_E2M1 = 7,
       DT_E8M0 = 8 /* scales only */ };

// bfloat16: the top 16 bits of an IEEE binary32.
double decode_bf16(uint16_t bits) {
  uint32_t u = uint32_t(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return double(f);
}

double decode_f32(uint32_t bits) {
  float f;
  std::memcpy(&f, &bits, sizeof f);
  return double(f);
}

// float8_e4m3fn (the dtype named in common.py's supported list): 1 sign bit,
// 4 exponent bits with bias 7, 3 mantissa bits, no infinities; exponent 15
// with mantissa 7 is NaN.  Exponent 0 encodes subnormals m/8 * 2^-6.
double decode_e4m3fn(uint8_t code) {
  const int s = code >> 7;
  const int e = (code >> 3) & 0xF;
  const int m = code & 0x7;
  if (e == 15 && m == 7) return std::nan("");
  const double mag = (e == 0) ? std::ldexp(m / 8.0, -6) : std::ldexp(1.0 + m / 8.0, e - 7);
  return s ? -mag : mag;
}

// float8_e5m2 (in common.py's list): 1 sign bit, 5 exponent bits with bias 15,
// 2 mantissa bits, IEEE-style: exponent 31 is infinity (mantissa 0) or NaN;
// exponent 0 encodes subnormals m/4 * 2^-14.
double decode_e5m2(uint8_t code) {
  const int s = code >> 7;
  const int e = (code >> 2) & 0x1F;
  const int m = code & 0x3;
  double mag;
  if (e == 31)
    mag = m == 0 ? HUGE_VAL : std::nan("");
  else
    mag = (e == 0) ? std::ldexp(m / 4.0, -14) : std::ldexp(1.0 + m / 4.0, e - 15);
  return s ? -mag : mag;
}

// float4_e2m1fn (in common.py's list): 1 sign bit, 2 exponent bits with bias 1,
// 1 mantissa bit, no infinities or NaN; exponent 0 encodes the subnormal m/2.
double decode_e2m1(uint8_t nibble) {
  const int s = (nibble >> 3) & 1;
  const int e = (nibble >> 1) & 0x3;
  const int m = nibble & 1;
  const double mag = (e == 0) ? m / 2.0 : std::ldexp(1.0 + m / 2.0, e - 1);
  return s ? -mag : mag;
}

// int4: two's complement in 4 bits (-8 .. 7); uint4: 0 .. 15.
double decode_int4(uint8_t nibble) { return nibble >= 8 ? double(int(nibble) - 16) : double(nibble); }

uint8_t nibble_at(const void* base, int64_t idx) {
  const uint8_t byte = static_cast<const uint8_t*>(base)[idx / 2];
  return (idx % 2 == 0) ? (byte & 0xF) : (byte >> 4);
}

double load(const void* base, int dtype, int64_t idx) {
  switch (dtype) {
    case DT_BF16: return decode_bf16(static_cast<const uint16_t*>(base)[idx]);
    case DT_F32: return decode_f32(static_cast<const uint32_t*>(base)[idx]);
    case DT_E4M3: return decode_e4m3fn(static_cast<const uint8_t*>(base)[idx]);
    case DT_E5M2: return decode_e5m2(static_cast<const uint8_t*>(base)[idx]);
    case DT_INT8: return double(static_cast<const int8_t*>(base)[idx]);
    case DT_INT4: return decode_int4(nibble_at(base, idx));
    case DT_UINT4: return double(nibble_at(base, idx));
    case DT_E2M1: return decode_e2m1(nibble_at(base, idx));
  }
  return std::nan("");
}

bool valid_dtype(int d) { return d >= DT_BF16 && d <= DT_E2M1; }

// E8M0 block scale (page "gemm_quant.rs", widen_block_scale_f32): byte e is
// 2^(e - 127), except that 255 is 0.
double decode_e8m0(uint8_t e) { return e == 255 ? 0.0 : std::ldexp(1.0, int(e) - 127); }

// A scale value stored as f32, E8M0 or e4m3fn.
double load_scale(const void* base, int dtype, int64_t idx) {
  if (dtype == DT_E8M0) return decode_e8m0(static_cast<const uint8_t*>(base)[idx]);
  if (dtype == DT_E4M3) return decode_e4m3fn(static_cast<const uint8_t*>(base)[idx]);
  return double(static_cast<const float*>(base)[idx]);
}

// Nearest e4m3fn value to y with ties to the even code, saturating at +-448
// (|y| above 448 gives 448); NaN gives the NaN code.  Found by comparing y with
// every finite magnitude of the format (format definition above).
uint8_t encode_e4m3_rne_sat(double y) {
  if (std::isnan(y)) return 0x7F;
  const uint8_t sign = std::signbit(y) ? 0x80 : 0x00;
  const double a = std::fabs(y);
  uint8_t best = 0;
  double best_d = HUGE_VAL;
  for (int code = 0; code <= 0x7E; ++code) {
    const double v = decode_e4m3fn(uint8_t(code));
    const double d = std::fabs(a - v);
    if (d < best_d || (d == best_d && (code & 1) == 0)) {
      best = uint8_t(code);
      best_d = d;
    }
  }
  return sign | best;
}

int resolve_threads(int threads) {
  if (threads > 0) return threads;
  unsigned hc = std::thread::hardware_concurrency();
  return hc ? int(hc) : 1;
}

// Runs body(i) for i in [0, count) on `threads` workers (dynamic hand-out).
template <class F>
void parallel_for(int64_t count, int threads, F body) {
  threads = std::max(1, std::min<int>(threads, int(std::min<int64_t>(count, 1 << 20))));
  if (threads <= 1) {
    for (int64_t i = 0; i < count; ++i) body(i);
    return;
  }
  std::atomic<int64_t> next{0};
  std::vector<std::thread> pool;
  for (int t = 0; t < threads; ++t)
    pool.emplace_back([&] {
      for (int64_t i = next++; i < count; i = next++) body(i);
    });
  for (auto& th : pool) th.join();
}

// offs[0] = 0, offs[g+1] = offs[g] + max(group_sizes[g], 0), capped at m.
void group_offsets(const int32_t* sizes, int32_t groups, int64_t m, std::vector<int64_t>& offs) {
  offs.assign(size_t(groups) + 1, 0);
  for (int32_t g = 0; g < groups; ++g) {
    int64_t s = sizes[g] > 0 ? sizes[g] : 0;
    offs[g + 1] = std::min<int64_t>(offs[g] + s, m);
  }
}

// The group that owns row r, or -1 when r lies at or past the last offset.
int32_t owning_group(const std::vector<int64_t>& offs, int64_t r) {
  const int32_t groups = int32_t(offs.size()) - 1;
  for (int32_t g = 0; g < groups; ++g)
    if (offs[g] <= r && r < offs[g + 1]) return g;
  return -1;
}

}  // namespace

extern "C" {

int oracle_default_threads(void) { return resolve_threads(0); }

void oracle_group_offsets(const int32_t* group_sizes, int32_t num_groups, int64_t m, int64_t* offs_out) {
  std::vector<int64_t> offs;
  group_offsets(group_sizes, num_groups, m, offs);
  std::copy(offs.begin(), offs.end(), offs_out);
}

// Forward grouped matmul.
//   lhs        [m, k]                          (lhs_dtype)
//   rhs        [L, n, k] if transpose_rhs else [L, k, n]   (rhs_dtype), L = num_local_groups
//   group_sizes[num_total_groups] int32; local groups are
//              [group_offset, group_offset + L) and use rhs[g - group_offset]
//   rhs_scale  NULL or [L, num_blocks, 1, n] f32; block b covers
//              k in [b*k/num_blocks, (b+1)*k/num_blocks)
//   rhs_bias   NULL or [L, 1, n] (bias_dtype)
//   rows       NULL: compute every row 0..m-1; else the listed row indices
//   ref, mag   [num_rows, n] fp64 outputs (num_rows = m when rows is NULL)
// Returns 0, or -1 on an argument it cannot interpret.
// The same with activation scales and a choice of weight-scale storage (page
// "gemm_quant.rs": the W8A8 GEMM multiplies each 128-wide K-group's products by
// a_scale[m, g], and block scales may be stored as E8M0):
//   lhs_scale        NULL or f32 [m, num_lhs_blocks]; lhs block j covers
//                    k in [j*k/num_lhs_blocks, (j+1)*k/num_lhs_blocks), and
//                    lhs[r, kk] counts as lhs_scale[r, j] * lhs[r, kk]
//   rhs_scale_dtype  DT_F32 or DT_E8M0 for rhs_scale
// and with per-element block scales of the weights, the microscaling layout
// (MXFP8: e4m3 weights with an E8M0 scale per 32 consecutive k of a weight
// row; NVFP4: e2m1 weights with an e4m3 scale per 16):
//   rhs_block_scale  NULL or [L, n, k / block_size] of rhs_block_scale_dtype
//                    (DT_E8M0, DT_E4M3 or DT_F32), transpose_rhs only; the
//                    weight W(g, c, kk) counts as
//                    rhs_block_scale[g, c, kk / block_size] * W(g, c, kk)
int oracle_gmm_ex2(const void* lhs, int lhs_dtype, int64_t m, int64_t k, const void* rhs, int rhs_dtype,
                   int32_t num_local_groups, int64_t n, int transpose_rhs, const int32_t* group_sizes,
                   int32_t num_total_groups, int32_t group_offset, const void* rhs_scale, int rhs_scale_dtype,
                   int32_t num_blocks, const float* lhs_scale, int32_t num_lhs_blocks, const void* rhs_block_scale,
                   int rhs_block_scale_dtype, int32_t block_size, const void* rhs_bias, int bias_dtype,
                   const int64_t* rows, int64_t num_rows, double* ref, double* mag, int threads) {
  if (!valid_dtype(lhs_dtype) || !valid_dtype(rhs_dtype)) return -1;
  if (rhs_bias && !valid_dtype(bias_dtype)) return -1;
  if (rhs_scale && rhs_scale_dtype != DT_F32 && rhs_scale_dtype != DT_E8M0) return -1;
  if (rhs_block_scale) {
    if (rhs_block_scale_dtype != DT_F32 && rhs_block_scale_dtype != DT_E8M0 && rhs_block_scale_dtype != DT_E4M3)
      return -1;
    if (!transpose_rhs || block_size <= 0 || k % block_size != 0) return -1;
  }
  const int64_t bpr = rhs_block_scale ? k / block_size : 0;  // block scales per weight row
  if (m < 0 || k < 0 || n < 0 || num_local_groups < 0 || num_total_groups < 0) return -1;
  if (group_offset < 0 || group_offset + num_local_groups > num_total_groups) return -1;
  const int32_t nb = rhs_scale ? num_blocks : 1;
  if (nb <= 0 || (k % nb) != 0) return -1;
  const int64_t block = nb ? k / nb : k;
  const int32_t nlb = lhs_scale ? num_lhs_blocks : 1;
  if (nlb <= 0 || (k % nlb) != 0) return -1;
  const int64_t lblock = k / nlb;

  std::vector<int64_t> offs;
  group_offsets(group_sizes, num_total_groups, m, offs);
  const int64_t count = rows ? num_rows : m;

  parallel_for(count, resolve_threads(threads), [&](int64_t i) {
    const int64_t r = rows ? rows[i] : i;
    double* ref_row = ref + i * n;
    double* mag_row = mag + i * n;
    const int32_t g = (r >= 0 && r < m) ? owning_group(offs, r) : -1;
    if (g < group_offset || g >= group_offset + num_local_groups) {
      for (int64_t c = 0; c < n; ++c) ref_row[c] = mag_row[c] = 0.0;
      return;
    }
    const int64_t gl = g - group_offset;  // index into the local rhs slice
    std::vector<double> a(static_cast<size_t>(k));
    for (int64_t kk = 0; kk < k; ++kk) {
      a[kk] = load(lhs, lhs_dtype, r * k + kk);
      if (lhs_scale) a[kk] *= double(lhs_scale[r * nlb + kk / lblock]);
    }
    for (int64_t c = 0; c < n; ++c) {
      double acc = 0.0, acc_abs = 0.0;
      for (int32_t b = 0; b < nb; ++b) {
        double part = 0.0, part_abs = 0.0;
        for (int64_t kk = b * block; kk < (b + 1) * block; ++kk) {
          const int64_t widx = transpose_rhs ? (gl * n + c) * k + kk : (gl * k + kk) * n + c;
          double w = load(rhs, rhs_dtype, widx);
          if (rhs_block_scale)
            w *= load_scale(rhs_block_scale, rhs_block_scale_dtype, (gl * n + c) * bpr + kk / block_size);
          part += a[kk] * w;
          part_abs += std::fabs(a[kk] * w);
        }
        const double s = rhs_scale ? load_scale(rhs_scale, rhs_scale_dtype, (gl * nb + b) * n + c) : 1.0;
        acc += s * part;
        acc_abs += std::fabs(s) * part_abs;
      }
      if (rhs_bias) {
        const double bias = load(rhs_bias, bias_dtype, gl * n + c);
        acc += bias;
        acc_abs += std::fabs(bias);
      }
      ref_row[c] = acc;
      mag_row[c] = acc_abs;
    }
  });
  return 0;
}

int oracle_gmm_ex(const void* lhs, int lhs_dtype, int64_t m, int64_t k, const void* rhs, int rhs_dtype,
                  int32_t num_local_groups, int64_t n, int transpose_rhs, const int32_t* group_sizes,
                  int32_t num_total_groups, int32_t group_offset, const void* rhs_scale, int rhs_scale_dtype,
                  int32_t num_blocks, const float* lhs_scale, int32_t num_lhs_blocks, const void* rhs_bias,
                  int bias_dtype, const int64_t* rows, int64_t num_rows, double* ref, double* mag, int threads) {
  return oracle_gmm_ex2(lhs, lhs_dtype, m, k, rhs, rhs_dtype, num_local_groups, n, transpose_rhs, group_sizes,
                        num_total_groups, group_offset, rhs_scale, rhs_scale_dtype, num_blocks, lhs_scale,
                        num_lhs_blocks, nullptr, 0, 0, rhs_bias, bias_dtype, rows, num_rows, ref, mag, threads);
}

int oracle_gmm(const void* lhs, int lhs_dtype, int64_t m, int64_t k, const void* rhs, int rhs_dtype,
               int32_t num_local_groups, int64_t n, int transpose_rhs, const int32_t* group_sizes,
               int32_t num_total_groups, int32_t group_offset, const float* rhs_scale, int32_t num_blocks,
               const void* rhs_bias, int bias_dtype, const int64_t* rows, int64_t num_rows, double* ref,
               double* mag, int threads) {
  return oracle_gmm_ex(lhs, lhs_dtype, m, k, rhs, rhs_dtype, num_local_groups, n, transpose_rhs, group_sizes,
                       num_total_groups, group_offset, rhs_scale, DT_F32, num_blocks, nullptr, 0, rhs_bias,
                       bias_dtype, rows, num_rows, ref, mag, threads);
}

// Per-token-group activation quantisation (page "gemm_quant.rs",
// per_token_group_quant_fp8: A_fp8 [M, K] e4m3 and a_scale [M, K/128] f32 from
// bf16 activations).  The page prints no formula; the reading taken here: for
// each row r and each group j of `group` consecutive k,
//   amax = max |x|  (NaN if any x is NaN),
//   scale[r, j] = amax / 448 in fp32 (448 is e4m3fn's largest value), or 1 when
//                 amax is 0,
//   q[r, kk] = e4m3fn nearest to x / scale[r, j] (the quotient formed in fp32),
//              ties to even, saturating at +-448.
// The fp32 steps are IEEE single-precision operations, as the kernel's are: the
// codes are fixed by those fp32 values.
int oracle_quantize_e4m3(const uint16_t* x, int64_t m, int64_t k, int64_t group, uint8_t* q, float* scale) {
  if (m < 0 || k < 0 || group <= 0 || (k % group) != 0) return -1;
  const int64_t ng = k / group;
  for (int64_t r = 0; r < m; ++r) {
    for (int64_t j = 0; j < ng; ++j) {
      float amax = 0.f;
      bool nan = false;
      for (int64_t kk = j * group; kk < (j + 1) * group; ++kk) {
        const float v = float(decode_bf16(x[r * k + kk]));
        if (std::isnan(v)) nan = true;
        amax = std::max(amax, std::fabs(v));
      }
      if (nan) amax = std::nanf("");
      const float s = amax == 0.f ? 1.f : amax / 448.f;
      scale[r * ng + j] = s;
      for (int64_t kk = j * group; kk < (j + 1) * group; ++kk) {
        const float y = float(decode_bf16(x[r * k + kk])) / s;
        q[r * k + kk] = encode_e4m3_rne_sat(double(y));
      }
    }
  }
  return 0;
}

// Backward weight gradient: out[g, kk, c] = sum_{r in group g} lhs[r, kk] * dout[r, c].
//   lhs  [m, k], dout [m, n]; out blocks [num_groups, k, n] (every group,
//   empty ones all-zero).
//   k_rows NULL: every kk in 0..k-1; else the listed kk (the same list for
//   every group); ref, mag are [num_groups, num_k_rows, n].
int oracle_tgmm(const void* lhs, int lhs_dtype, int64_t m, int64_t k, const void* dout, int dout_dtype,
                int64_t n, const int32_t* group_sizes, int32_t num_groups, const int64_t* k_rows,
                int64_t num_k_rows, double* ref, double* mag, int threads) {
  if (!valid_dtype(lhs_dtype) || !valid_dtype(dout_dtype)) return -1;
  if (m < 0 || k < 0 || n < 0 || num_groups < 0) return -1;
  std::vector<int64_t> offs;
  group_offsets(group_sizes, num_groups, m, offs);
  const int64_t kc = k_rows ? num_k_rows : k;

  parallel_for(int64_t(num_groups) * kc, resolve_threads(threads), [&](int64_t job) {
    const int64_t g = job / kc;
    const int64_t j = job % kc;
    const int64_t kk = k_rows ? k_rows[j] : j;
    double* ref_row = ref + (g * kc + j) * n;
    double* mag_row = mag + (g * kc + j) * n;
    for (int64_t c = 0; c < n; ++c) ref_row[c] = mag_row[c] = 0.0;
    for (int64_t r = offs[g]; r < offs[g + 1]; ++r) {
      const double a = load(lhs, lhs_dtype, r * k + kk);
      for (int64_t c = 0; c < n; ++c) {
        const double p = a * load(dout, dout_dtype, r * n + c);
        ref_row[c] += p;
        mag_row[c] += std::fabs(p);
      }
    }
  });
  return 0;
}

// Decodes `count` stored values of `dtype` into fp64 (used by the format pins).
int oracle_decode(const void* src, int dtype, int64_t count, double* dst) {
  if (dtype == DT_E8M0) {
    for (int64_t i = 0; i < count; ++i) dst[i] = decode_e8m0(static_cast<const uint8_t*>(src)[i]);
    return 0;
  }
  if (!valid_dtype(dtype)) return -1;
  for (int64_t i = 0; i < count; ++i) dst[i] = load(src, dtype, i);
  return 0;
}

}  // extern "C"
