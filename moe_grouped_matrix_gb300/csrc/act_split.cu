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
#include <cuda_fp16.h>

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

// The fp16 split of bf16 activation rows, for the weight formats that run on
// the fp16 tensor cores (gemm_f16w.cu): per row r and 128-wide step s, with E the
// exponent field of the step's largest |x| (at least 15, so that the scale is
// an fp32 normal),
//   sc = 2^(E - 141),  plane[r, kk] = rne_f16(x / sc),
// exact for every x within 2^28 of the largest (fp16 normals) and for smaller
// ones down to fp16's subnormal grid, 2^-24 sc.  A step with an x that this does
// not hold, or with an infinity or a NaN, is marked: scale[r, s] = (sc, -0),
// else (sc, +0), and *pending is set (the matmul then sums the row again).
// With `perm` (4-bit weights) each 8 k are stored in the order
// 0, 4, 1, 5, 2, 6, 3, 7, the order in which the weight rewrite produces them.
// One warp per (row, step), 4 values per lane.
__global__ void __launch_bounds__(256) act_split_f16_kernel(const uint16_t* __restrict__ x, int64_t m, int64_t k,
                                                           int32_t ksteps, uint16_t* __restrict__ plane,
                                                           float2* __restrict__ scale, uint32_t* pending, int perm) {
  const int lane = threadIdx.x & 31;
  const int64_t w = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;  // (row, step)
  if (w >= m * ksteps) return;  // whole warps: blockDim is a multiple of 32
  const int64_t row = w / ksteps;
  const int32_t s = int32_t(w - row * ksteps);
  const int64_t kk = int64_t(s) * 128 + lane * 4;  // k % 128 == 0: every lane is in range
  const uint2 v = *reinterpret_cast<const uint2*>(x + row * k + kk);
  const uint32_t b[4] = {v.x << 16, v.x & 0xFFFF0000u, v.y << 16, v.y & 0xFFFF0000u};  // fp32 bits
  uint32_t amax = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) amax = max(amax, b[i] & 0x7FFFFFFFu);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const uint32_t e = max(amax >> 23, 15u);
  const bool finite = amax < 0x7F800000u;
  const float sc = __uint_as_float((e - 14u) << 23);       // 2^(e - 141), e <= 254
  const float inv = __uint_as_float((268u - e) << 23);     // 2^(141 - e)
  uint16_t h[4];
  bool inexact = false;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float xf = __uint_as_float(b[i]);
    const __half q = __float2half_rn(xf * inv);
    h[i] = __half_as_ushort(q);
    inexact |= __half2float(q) * sc != xf;
  }
  const bool marked = __any_sync(0xffffffffu, inexact) || !finite;
  uint32_t lo = uint32_t(h[0]) | (uint32_t(h[1]) << 16), hi = uint32_t(h[2]) | (uint32_t(h[3]) << 16);
  if (perm) {
    // lanes 2g and 2g + 1 hold k 8g + 0..3 and 8g + 4..7: the even lane keeps
    // (0, 4, 1, 5), the odd one (2, 6, 3, 7)
    const bool odd = lane & 1;
    const uint32_t other = __shfl_xor_sync(0xffffffffu, odd ? lo : hi, 1);
    const uint32_t mine = odd ? hi : lo;  // even: (x0, x1); odd: (x6, x7)
    if (!odd) {
      lo = (mine & 0xFFFFu) | (other << 16);                 // x0, x4
      hi = (mine >> 16) | (other & 0xFFFF0000u);             // x1, x5
    } else {
      lo = (other & 0xFFFFu) | (mine << 16);                 // x2, x6
      hi = (other >> 16) | (mine & 0xFFFF0000u);             // x3, x7
    }
  }
  *reinterpret_cast<uint2*>(plane + row * k + kk) = make_uint2(lo, hi);
  if (lane == 0) {
    scale[row * ksteps + s] = make_float2(sc, marked ? -0.f : 0.f);
    if (marked) atomicOr(pending, 1u);
  }
  griddep_launch_dependents();
}

}  // namespace

cudaError_t launch_act_split_f16(const void* x, int64_t m, int64_t k, void* plane, float* scale, uint32_t* pending,
                                 bool perm, cudaStream_t stream) {
  if (k % 128 != 0) return cudaErrorInvalidValue;
  const int64_t ksteps = k / 128;
  const int64_t warps = m * ksteps;
  if (warps == 0) return cudaSuccess;
  const int64_t blocks = (warps * 32 + 255) / 256;
  if (blocks > INT32_MAX) return cudaErrorInvalidValue;
  act_split_f16_kernel<<<unsigned(blocks), 256, 0, stream>>>(static_cast<const uint16_t*>(x), m, k, int32_t(ksteps),
                                                            static_cast<uint16_t*>(plane),
                                                            reinterpret_cast<float2*>(scale), pending, perm ? 1 : 0);
  return cudaGetLastError();
}

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
