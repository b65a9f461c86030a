// gmm_noalloc: the forward grouped matmul for callers that cannot allocate
// device memory.
//
// gmm() needs a small caller-owned device workspace (the kernel's error-flag
// word).  Some callers cannot provide one: code whose device memory is owned
// entirely by another component's allocator and that has no way to request a
// buffer from it, or code on a path where calling cudaMalloc is not allowed
// (cudaMalloc may synchronise the device and its latency is unbounded).  This
// entry point serves them by using a scratch array compiled into the library
// instead: a file-scope __device__ array that every GPU which loads the
// library holds until the process exits.  It calls no cudaMalloc, cudaFree or
// allocating library routine.
//
// The kernels need one 32-bit word of device-side error flags, so any problem
// size the ABI accepts fits the fixed array below.  The optional scratch of a
// gmm_workspace_bytes() workspace (split bf16 activations for the fp8
// kernels) is not provided here: those kernels then split inside.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/libgmm.h"

namespace {

// The scratch: error flags in word 0, the rest reserved.  Shared by every call
// on a device.
static __device__ __align__(256) uint8_t g_noalloc_scratch[GMM_NOALLOC_SCRATCH_BYTES];

// The host-side name g_noalloc_scratch is only a stand-in for the symbol, not a
// device address.  The device address of the current device's copy is looked up
// on every call (a host-side lookup, no allocation), so it stays right after the
// device's context is destroyed and created again (cudaDeviceReset), which moves
// the array.
int scratch_for_current_device(void** ptr) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return GMM_ERR_CUDA;
  *ptr = p;
  return GMM_OK;
}

}  // namespace

extern "C" int gmm_noalloc(const void* lhs, int lhs_dtype, int64_t m, int64_t k, const void* rhs, int rhs_dtype,
                           int32_t num_local_groups, int64_t n, int transpose_rhs, const int32_t* group_sizes,
                           int32_t num_total_groups, int32_t group_offset, const float* rhs_scale,
                           int32_t num_quant_blocks, const void* rhs_bias, int bias_dtype, void* out,
                           int out_dtype, void* stream) {
  static_assert(GMM_NOALLOC_SCRATCH_BYTES >= GMM_WORKSPACE_MIN_BYTES, "scratch below the workspace minimum");
  void* scratch = nullptr;
  if (int st = scratch_for_current_device(&scratch)) return st;
  // The flags must start at zero for this call; the array keeps whatever the
  // previous call on this device left in it.
  if (cudaMemsetAsync(scratch, 0, sizeof(uint32_t), static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return GMM_ERR_CUDA;
  return gmm(lhs, lhs_dtype, m, k, rhs, rhs_dtype, num_local_groups, n, transpose_rhs, group_sizes,
             num_total_groups, group_offset, rhs_scale, num_quant_blocks, rhs_bias, bias_dtype, out, out_dtype,
             scratch, sizeof(g_noalloc_scratch), stream);
}
