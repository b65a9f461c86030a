// e4m3 activations with int4 and uint4 weights, rewritten as e4m3 tiles by the
// weight-rewrite warps.
#include "gemm_fp8.cuh"

namespace gmmk {

cudaError_t launch_fp8_a8_packed(const ScaledLaunch& p, int weight_format, bool out_f32, int grid,
                                 cudaStream_t stream) {
  switch (weight_format) {
    case kWeightInt4: return fp8::launch_format<fp8::WFmt::kInt4, true>(p, out_f32, grid, stream);
    case kWeightUint4: return fp8::launch_format<fp8::WFmt::kUint4, true>(p, out_f32, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace gmmk
