// int8, int4 and uint4 weights: the fp8 tensor-core kernel with the
// weight-rewrite warps (each tile rewritten exactly as e4m3 A tiles).
#include "gemm_fp8.cuh"

namespace gmmk {

cudaError_t launch_fp8_converted(const ScaledLaunch& p, int weight_format, bool out_f32, int grid,
                                 cudaStream_t stream) {
  switch (weight_format) {
    case kWeightInt8: return fp8::launch_format<fp8::WFmt::kInt8, false>(p, out_f32, grid, stream);
    case kWeightInt4: return fp8::launch_format<fp8::WFmt::kInt4, false>(p, out_f32, grid, stream);
    case kWeightUint4: return fp8::launch_format<fp8::WFmt::kUint4, false>(p, out_f32, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace gmmk
