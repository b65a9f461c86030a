// Split bf16 activations (act_split.cu) with int8, int4 and uint4 weights: the
// e4m3-activation shape of the fp8 kernel, whose single token warp leaves room
// for 8 weight-rewrite warps.
#include "gemm_fp8.cuh"

namespace gmmk {

cudaError_t launch_fp8_ps_converted(const ScaledLaunch& p, int weight_format, bool out_f32, int grid,
                                   cudaStream_t stream) {
  switch (weight_format) {
    case kWeightInt8: return fp8::launch_format<fp8::WFmt::kInt8, true, true>(p, out_f32, grid, stream);
    case kWeightInt4: return fp8::launch_format<fp8::WFmt::kInt4, true, true>(p, out_f32, grid, stream);
    case kWeightUint4: return fp8::launch_format<fp8::WFmt::kUint4, true, true>(p, out_f32, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gmmk
