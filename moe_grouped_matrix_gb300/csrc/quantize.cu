// Per-token-group e4m3 quantisation of bf16 activations (page "gemm_quant.rs",
// per_token_group_quant_fp8: A_fp8 [M, K] e4m3 and a_scale [M, K/128] f32, the
// activation side of the W8A8 grouped matmul).  For each row and each group of
// `group` consecutive k:
//   amax  = max |x| (NaN if any x is NaN),
//   scale = amax / 448 (fp32, IEEE division), 1 when amax is 0,
//   q     = e4m3 nearest to x / scale (fp32, IEEE division), ties to even,
//           saturating at +-448.
// One warp per (row, group); each lane holds group / 32 consecutive values
// (group 64, 128 or 256).
// HBM-bound: 2 bytes read and 1 byte written per value.
#include <cuda_bf16.h>

#include <climits>

#include "internal.h"

namespace gmmk {
namespace {

template <int V>  // values per lane: group / 32 (even)
__global__ void __launch_bounds__(256) quantize_e4m3_kernel(const uint16_t* __restrict__ x, int64_t m, int64_t k,
                                                           uint8_t* __restrict__ q, float* __restrict__ scale) {
  constexpr int kGroup = 32 * V;
  const int lane = threadIdx.x & 31;
  const int64_t ngroups = k / kGroup;
  const int64_t w = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;  // (row, group) index
  if (w >= m * ngroups) return;
  const int64_t row = w / ngroups, grp = w - row * ngroups;
  const int64_t base = row * k + grp * kGroup + int64_t(lane) * V;
  uint16_t xs[V];
  if constexpr (V == 4) {
    const uint2 v = *reinterpret_cast<const uint2*>(x + base);
    xs[0] = uint16_t(v.x), xs[1] = uint16_t(v.x >> 16), xs[2] = uint16_t(v.y), xs[3] = uint16_t(v.y >> 16);
  } else {
#pragma unroll
    for (int i = 0; i < V; ++i) xs[i] = x[base + i];
  }
  // |x| as ordered bits: every NaN compares above infinity, so a NaN wins.
  uint32_t amax_bits = 0;
#pragma unroll
  for (int i = 0; i < V; ++i) amax_bits = max(amax_bits, (uint32_t(xs[i]) << 16) & 0x7FFFFFFFu);
  amax_bits = __reduce_max_sync(0xffffffffu, amax_bits);
  const float amax = __uint_as_float(amax_bits);
  const float s = amax_bits == 0 ? 1.f : __fdiv_rn(amax, 448.f);
  uint8_t out[V];
#pragma unroll
  for (int i = 0; i < V; i += 2) {
    const float y0 = __fdiv_rn(__uint_as_float(uint32_t(xs[i]) << 16), s);
    const float y1 = __fdiv_rn(__uint_as_float(uint32_t(xs[i + 1]) << 16), s);
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(y1), "f"(y0));
    out[i] = uint8_t(r), out[i + 1] = uint8_t(r >> 8);
  }
  if constexpr (V == 4) {
    *reinterpret_cast<uint32_t*>(q + base) =
        uint32_t(out[0]) | (uint32_t(out[1]) << 8) | (uint32_t(out[2]) << 16) | (uint32_t(out[3]) << 24);
  } else {
#pragma unroll
    for (int i = 0; i < V; ++i) q[base + i] = out[i];
  }
  if (lane == 0) scale[row * ngroups + grp] = s;
}

}  // namespace

cudaError_t launch_quantize_e4m3(const void* x, int64_t m, int64_t k, int64_t group, void* q, float* scale,
                                 cudaStream_t stream) {
  const int64_t warps = m * (k / group);
  if (warps == 0) return cudaSuccess;
  const int64_t blocks = (warps * 32 + 255) / 256;
  if (blocks > INT32_MAX) return cudaErrorInvalidValue;
  const auto* xs = static_cast<const uint16_t*>(x);
  auto* qs = static_cast<uint8_t*>(q);
  switch (group) {
    case 64: quantize_e4m3_kernel<2><<<unsigned(blocks), 256, 0, stream>>>(xs, m, k, qs, scale); break;
    case 128: quantize_e4m3_kernel<4><<<unsigned(blocks), 256, 0, stream>>>(xs, m, k, qs, scale); break;
    case 256: quantize_e4m3_kernel<8><<<unsigned(blocks), 256, 0, stream>>>(xs, m, k, qs, scale); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace gmmk
