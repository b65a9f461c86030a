// Split bf16 activations (act_split.cu): the fp8 tensor-core kernel takes the
// h and l rows by TMA, as it takes e4m3 activations.  e4m3, e5m2 and e2m1
// weights here; int8, int4 and uint4 in gemm_fp8_ps_int.cu.
#include "gemm_fp8.cuh"

namespace gmmk {

cudaError_t launch_fp8_ps(const ScaledLaunch& p, int weight_format, bool out_f32, int grid, cudaStream_t stream) {
  switch (weight_format) {
    case kWeightE4M3: return fp8::launch_format<fp8::WFmt::kE4M3, true, true>(p, out_f32, grid, stream);
    case kWeightE5M2: return fp8::launch_format<fp8::WFmt::kE5M2, true, true>(p, out_f32, grid, stream);
    case kWeightE2M1: return fp8::launch_format<fp8::WFmt::kE2M1, true, true>(p, out_f32, grid, stream);
    default: return launch_fp8_ps_converted(p, weight_format, out_f32, grid, stream);
  }
}

}  // namespace gmmk
