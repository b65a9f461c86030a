// e4m3, e5m2 and e2m1 weights: the fp8 tensor-core kernel reads the TMA tiles
// as its A operand directly.  Dispatch for every weight format of that kernel.
#include "gemm_fp8.cuh"

namespace gmmk {

cudaError_t launch_fp8(const ScaledLaunch& p, int weight_format, bool out_f32, int grid, cudaStream_t stream) {
  if (p.lhs_split) return launch_fp8_ps(p, weight_format, out_f32, grid, stream);
  if (p.lhs_e4m3) return launch_fp8_a8(p, weight_format, out_f32, grid, stream);
  switch (weight_format) {
    case kWeightE4M3: return fp8::launch_format<fp8::WFmt::kE4M3, false>(p, out_f32, grid, stream);
    case kWeightE5M2: return fp8::launch_format<fp8::WFmt::kE5M2, false>(p, out_f32, grid, stream);
    case kWeightE2M1: return fp8::launch_format<fp8::WFmt::kE2M1, false>(p, out_f32, grid, stream);
    default: return launch_fp8_converted(p, weight_format, out_f32, grid, stream);
  }
}

}  // namespace gmmk
