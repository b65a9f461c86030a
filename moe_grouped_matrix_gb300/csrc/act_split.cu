// The exact two-term e4m3 split of bf16 activation rows, made once per row
// for the fp8 kernel's split-activation mode (gemm_fp8.cuh, kPS), which would
// otherwise make it once per row and 128-wide weight tile.  For each row r and
// each k step s of the kernel (256 wide, the last one 128 wide when k % 256 ==
// 128; 128 wide for int8 weights), with M the largest |x| of the step and e
// its biased exponent clamped to [8, 254]:
//   y = x * 2^(134 - e),  h = rne_e4m3(y),  l = rne_e4m3(16 (y - h)),
//   planes[0][r, kk] = h,  planes[1][r, kk] = l,
//   scale[r, s] = 2^(e - 134)   (NaN when M is an infinity or a NaN),
// so that x = scale * (h + l / 16) (see the exactness argument in
// gemm_fp8.cuh).  The arithmetic is the kernel's own split_e4m3 and exponent
// rule, so both modes give the same codes.
// One warp per (row, step), 8 (256-wide steps) or 4 values per lane.
// HBM-bound: 2 bytes read and 2 written per value.  The fp8 kernel that
// follows is launched as its programmatic dependent (gemm_fp8.cuh).
#include <cuda_bf16.h>

#include <climits>

#include "gemm_fp8.cuh"

namespace gmmk {
namespace {

template <int V>  // values per lane: step / 32
__global__ void __launch_bounds__(256) act_split_kernel(const uint16_t* __restrict__ x, int64_t m, int64_t k,
                                                       int32_t ksteps, uint8_t* __restrict__ planes,
                                                       float* __restrict__ scale) {
  constexpr int W = V / 2;  // 32-bit words of bf16 pairs per lane
  const int lane = threadIdx.x & 31;
  const int64_t w = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;  // (row, step)
  if (w >= m * ksteps) return;
  const int64_t row = w / ksteps;
  const int32_t s = int32_t(w - row * ksteps);
  const int64_t kk = int64_t(s) * (32 * V) + lane * V;
  const bool mine = kk < k;  // k % 128 == 0: a 128-wide last step of 256 fills lanes 0-15
  uint32_t xw[W];
#pragma unroll
  for (int i = 0; i < W; ++i) xw[i] = 0u;
  if (mine) {
    if constexpr (V == 8) {
      const uint4 v = *reinterpret_cast<const uint4*>(x + row * k + kk);
      xw[0] = v.x, xw[1] = v.y, xw[2] = v.z, xw[3] = v.w;
    } else {
      const uint2 v = *reinterpret_cast<const uint2*>(x + row * k + kk);
      xw[0] = v.x, xw[1] = v.y;
    }
  }
  uint32_t amax = 0;
#pragma unroll
  for (int i = 0; i < W; ++i) amax = max(amax, max((xw[i] << 16) & 0x7FFFFFFFu, xw[i] & 0x7FFF0000u));
  amax = __reduce_max_sync(0xffffffffu, amax);
  const uint32_t e = min(max(amax >> 23, 8u), 254u);
  const float inv_s = __uint_as_float((261u - e) << 23);
  float y[V];
#pragma unroll
  for (int i = 0; i < W; ++i) {
    y[2 * i] = __uint_as_float(xw[i] << 16) * inv_s;
    y[2 * i + 1] = __uint_as_float(xw[i] & 0xFFFF0000u) * inv_s;
  }
  uint32_t hw[V / 4], lw[V / 4];
  fp8::split_e4m3<V>(y, hw, lw);
  if (mine) {
    if constexpr (V == 8) {
      *reinterpret_cast<uint2*>(planes + row * k + kk) = make_uint2(hw[0], hw[1]);
      *reinterpret_cast<uint2*>(planes + (m + row) * k + kk) = make_uint2(lw[0], lw[1]);
    } else {
      *reinterpret_cast<uint32_t*>(planes + row * k + kk) = hw[0];
      *reinterpret_cast<uint32_t*>(planes + (m + row) * k + kk) = lw[0];
    }
  }
  if (lane == 0)
    scale[row * ksteps + s] = amax < 0x7F800000u ? __uint_as_float((e - 7u) << 23) : __uint_as_float(0x7FC00000u);
  // The matmul that reads these rows may start now (it waits for this grid's
  // completion before its first read of them).  Signalled after the work, so
  // that its CTAs never hold SMs this grid still needs.
  griddep_launch_dependents();
}

}  // namespace

cudaError_t launch_act_split(const void* x, int64_t m, int64_t k, int32_t step, void* planes, float* scale,
                             cudaStream_t stream) {
  if (step != 256 && step != 128) return cudaErrorInvalidValue;
  const int64_t ksteps = (k + step - 1) / step;
  const int64_t warps = m * ksteps;
  if (warps == 0) return cudaSuccess;
  const int64_t blocks = (warps * 32 + 255) / 256;
  if (blocks > INT32_MAX) return cudaErrorInvalidValue;
  const auto* xs = static_cast<const uint16_t*>(x);
  auto* ps = static_cast<uint8_t*>(planes);
  if (step == 256)
    act_split_kernel<8><<<unsigned(blocks), 256, 0, stream>>>(xs, m, k, int32_t(ksteps), ps, scale);
  else
    act_split_kernel<4><<<unsigned(blocks), 256, 0, stream>>>(xs, m, k, int32_t(ksteps), ps, scale);
  return cudaGetLastError();
}

}  // namespace gmmk
