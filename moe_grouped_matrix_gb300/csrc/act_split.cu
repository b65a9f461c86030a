// The two-level e4m3 split of bf16 activation rows (split_step in gemm_fp8.cuh),
// made once per row for the fp8 kernel's split-activation mode (kPS), which
// would otherwise make it once per row and 128-wide weight tile.  For each row r
// and each k step s of the kernel (256 wide, the last one 128 wide when k % 256
// == 128; 128 wide for int8 weights):
//   planes[0][r, kk] = h,  planes[1][r, kk] = l,  planes[2][r, kk] = h2,
//   planes[3][r, kk] = l2,  scale[r, s] = (s1, s2),
// so that x = s1 (h + l / 16) + s2 (h2 + l2 / 16) for every value of the step
// unless s2's sign bit marks the step; a marked step also sets *pending, which
// tells the fp8 kernel to sum its row again (fix_marked_rows).  The arithmetic
// is the kernel's own split_step, so both modes give the same codes.
// One warp per (row, step), 8 (256-wide steps) or 4 values per lane.
// HBM-bound: 2 bytes read and 4 written per value.  The fp8 kernel that follows
// is launched as its programmatic dependent (gemm_fp8.cuh).
#include <cuda_bf16.h>

#include <climits>

#include "gemm_fp8.cuh"

namespace gmmk {
namespace {

template <int V>  // values per lane: step / 32
__global__ void __launch_bounds__(256) act_split_kernel(const uint16_t* __restrict__ x, int64_t m, int64_t k,
                                                       int32_t ksteps, uint8_t* __restrict__ planes,
                                                       float2* __restrict__ scale, uint32_t* pending) {
  constexpr int W = V / 2;  // 32-bit words of bf16 pairs per lane
  const int lane = threadIdx.x & 31;
  const int64_t w = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;  // (row, step)
  if (w >= m * ksteps) return;  // whole warps: blockDim is a multiple of 32
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
  uint32_t hw[V / 4], lw[V / 4], hw2[V / 4], lw2[V / 4];
  float s1, s2;
  fp8::split_step<V, 32>(xw, hw, lw, hw2, lw2, s1, s2);
  if (mine) {
    const int64_t plane = m * k;
    uint8_t* p = planes + row * k + kk;
    if constexpr (V == 8) {
      *reinterpret_cast<uint2*>(p) = make_uint2(hw[0], hw[1]);
      *reinterpret_cast<uint2*>(p + plane) = make_uint2(lw[0], lw[1]);
      *reinterpret_cast<uint2*>(p + 2 * plane) = make_uint2(hw2[0], hw2[1]);
      *reinterpret_cast<uint2*>(p + 3 * plane) = make_uint2(lw2[0], lw2[1]);
    } else {
      *reinterpret_cast<uint32_t*>(p) = hw[0];
      *reinterpret_cast<uint32_t*>(p + plane) = lw[0];
      *reinterpret_cast<uint32_t*>(p + 2 * plane) = hw2[0];
      *reinterpret_cast<uint32_t*>(p + 3 * plane) = lw2[0];
    }
  }
  if (lane == 0) {
    scale[row * ksteps + s] = make_float2(s1, s2);
    if (__float_as_uint(s2) >> 31) atomicOr(pending, 1u);
  }
  // The matmul that reads these rows may start now (it waits for this grid's
  // completion before its first read of them).  Signalled after the work, so
  // that its CTAs never hold SMs this grid still needs.
  griddep_launch_dependents();
}

}  // namespace

cudaError_t launch_act_split(const void* x, int64_t m, int64_t k, int32_t step, void* planes, float* scale,
                             uint32_t* pending, cudaStream_t stream) {
  if (step != 256 && step != 128) return cudaErrorInvalidValue;
  const int64_t ksteps = (k + step - 1) / step;
  const int64_t warps = m * ksteps;
  if (warps == 0) return cudaSuccess;
  const int64_t blocks = (warps * 32 + 255) / 256;
  if (blocks > INT32_MAX) return cudaErrorInvalidValue;
  const auto* xs = static_cast<const uint16_t*>(x);
  auto* ps = static_cast<uint8_t*>(planes);
  auto* sc = reinterpret_cast<float2*>(scale);
  if (step == 256)
    act_split_kernel<8><<<unsigned(blocks), 256, 0, stream>>>(xs, m, k, int32_t(ksteps), ps, sc, pending);
  else
    act_split_kernel<4><<<unsigned(blocks), 256, 0, stream>>>(xs, m, k, int32_t(ksteps), ps, sc, pending);
  return cudaGetLastError();
}

}  // namespace gmmk
