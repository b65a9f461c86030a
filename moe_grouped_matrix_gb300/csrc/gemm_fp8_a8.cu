// e4m3 activations (W8A8 and the other weight formats): the fp8 tensor-core
// kernel takes the token rows by TMA as its B operand, scaled per sub-tile.
// e4m3, e5m2, e2m1 and int8 weights here; int4 and uint4 in gemm_fp8_a8_int.cu.
#include "gemm_fp8.cuh"

namespace gmmk {

cudaError_t launch_fp8_a8(const ScaledLaunch& p, int weight_format, bool out_f32, int grid, cudaStream_t stream) {
  switch (weight_format) {
    case kWeightE4M3: return fp8::launch_format<fp8::WFmt::kE4M3, true>(p, out_f32, grid, stream);
    case kWeightE5M2: return fp8::launch_format<fp8::WFmt::kE5M2, true>(p, out_f32, grid, stream);
    case kWeightE2M1: return fp8::launch_format<fp8::WFmt::kE2M1, true>(p, out_f32, grid, stream);
    case kWeightInt8: return fp8::launch_format<fp8::WFmt::kInt8, true>(p, out_f32, grid, stream);
    default: return launch_fp8_a8_packed(p, weight_format, out_f32, grid, stream);
  }
}

}  // namespace gmmk
