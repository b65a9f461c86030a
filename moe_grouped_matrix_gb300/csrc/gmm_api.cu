// C ABI of libgmm: host-side validation, TMA tensor-map encoding and kernel
// launch.  Argument rules follow the page "tpu-inference 0.12.0.dev20251213 ->
// 0.13.2.dev20251230", gmm.py (_validate_args: lhs 2-D, rhs 3-D with matching
// k, int32 group_sizes, rhs_scale [G, nb, 1, n], rhs_bias [G, 1, n]; gmm:
// k // num_quant_blocks block width) plus the alignment rules of TMA.
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/libgmm.h"
#include "internal.h"

namespace {

// Workspace: [0, 256) word 0 the sticky error flags, word 1 the split marks
// pending and word 2 the count of finished CTAs of the fp8 kernels (their last
// CTA sums marked rows again); then, used only when the
// caller's workspace holds all of it, scratch for the split bf16 activations
// of the fp8 kernels (h / l / h2 / l2 planes [4, m, k] and the (s1, s2) step
// scales [m, k steps, 2]).
constexpr size_t kWorkspaceMinBytes = 256;
constexpr size_t kActOffset = 256;
constexpr size_t kActScratchBytes = size_t(16) << 20;
constexpr size_t kWorkspaceBytes = kActOffset + kActScratchBytes;
thread_local int t_last_cuda_error = 0;

int cuda_fail(int code) {
  t_last_cuda_error = code;
  return GMM_ERR_CUDA;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

struct DeviceInfo {
  int sms = 0, major = 0, minor = 0;
  cudaError_t status = cudaSuccess;
};
constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];
std::once_flag g_device_once[kMaxDevices];

// Current device's SM count; GMM_ERR_ARCH unless it is compute capability 10.3.
int current_device(DeviceInfo* info) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return GMM_ERR_ARCH;
  std::call_once(g_device_once[dev], [dev] {
    DeviceInfo d;
    d.status = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (d.status == cudaSuccess) d.status = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev);
    if (d.status == cudaSuccess) d.status = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev);
    g_devices[dev] = d;
  });
  *info = g_devices[dev];
  if (info->status != cudaSuccess) return cuda_fail(info->status);
  if (info->major != 10 || info->minor != 3) return GMM_ERR_ARCH;
  return GMM_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Tiled tensor map over a row-major array; dims are innermost first.
int make_map(CUtensorMap* map, CUtensorMapDataType dt, int elem_bytes, int rank, const void* base,
             const uint64_t* dims, const uint32_t* box, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return cuda_fail(cudaErrorNotSupported);
  cuuint64_t gdim[5], gstride[4];
  cuuint32_t bdim[5], estride[5];
  uint64_t pitch = uint64_t(elem_bytes);
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estride[i] = 1;
    if (i > 0) gstride[i - 1] = pitch;
    pitch *= dims[i];
  }
  CUresult r = fn(map, dt, cuuint32_t(rank), const_cast<void*>(base), gdim, gstride, bdim, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(int(r));
  return GMM_OK;
}

// A map with explicit byte strides (strides[i] between consecutive indices of
// dimension i + 1); dimension 0 is contiguous.
int make_map_strided(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base, const uint64_t* dims,
                     const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return cuda_fail(cudaErrorNotSupported);
  cuuint64_t gdim[5], gstride[4];
  cuuint32_t bdim[5], estride[5];
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estride[i] = 1;
    if (i > 0) gstride[i - 1] = strides[i - 1];
  }
  CUresult r = fn(map, dt, cuuint32_t(rank), const_cast<void*>(base), gdim, gstride, bdim, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(int(r));
  return GMM_OK;
}

// e2m1 weights [L, n, k], two codes per byte (even k in the low nibble), in
// {128 k, 128 rows} boxes that land in shared memory as 128-byte rows, each 8
// bytes of codes followed by an 8-byte gap (the 4-bit operand layout of
// tcgen05.mma.kind::f8f6f4).  Needs k % 128 == 0 and a 32-byte-aligned base.
int make_map_e2m1(CUtensorMap* map, const void* base, int64_t k, int64_t n, int64_t L) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return cuda_fail(cudaErrorNotSupported);
  cuuint64_t gdim[3] = {cuuint64_t(k), cuuint64_t(n), cuuint64_t(L)};
  cuuint64_t gstride[2] = {cuuint64_t(k / 2), cuuint64_t(n) * cuuint64_t(k / 2)};
  cuuint32_t bdim[3] = {128, 128, 1}, estride[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<void*>(base), gdim, gstride, bdim, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(int(r));
  return GMM_OK;
}

bool fits_i32(int64_t v) { return v >= 0 && v <= INT32_MAX; }

// The bf16 forward kernels:
//   kPair     256 x 256 tiles of rows x n on SM pairs: the fastest per MMA, but
//             a group's last 256-row tile may be mostly padding;
//   kSwapPair SM pairs with 256 weight rows on the MMA's M side and up to 256
//             of a group's rows on its N side (rounded to 32): little padding,
//             pair-level traffic per SM;
//   kSwap     one SM, 128 weight rows x up to 256 rows (rounded to 16);
//   kSingle   one SM, 128 x 256 tiles of rows x n.
// Groups averaging 1024 rows or more go to kPair, 16 or more to kSwapPair,
// fewer to kSwap, unless the tiling table has an entry for the problem's class
// (tuning.cu).  A per-call gmm_options.bf16_kernel overrides both (for tuning
// and tests).
enum class BF16Kernel { kSingle, kPair, kSwap, kSwapPair, kInvalid };

BF16Kernel kernel_of_id(int id) {
  switch (id) {
    case GMM_KERNEL_PAIR: return BF16Kernel::kPair;
    case GMM_KERNEL_SWAP_PAIR: return BF16Kernel::kSwapPair;
    case GMM_KERNEL_SWAP: return BF16Kernel::kSwap;
    case GMM_KERNEL_SINGLE: return BF16Kernel::kSingle;
  }
  return BF16Kernel::kInvalid;
}

// The kernel and raster (0: default) for a problem; `forced` (a GMM_KERNEL_* id,
// from gmm_tune or the caller's options) wins over everything.
BF16Kernel choose_bf16_kernel(int64_t m, int64_t k, int64_t n, int32_t num_total_groups, int transpose_rhs,
                              int out_dtype, int forced, int32_t* raster) {
  *raster = 0;
  if (forced != GMM_KERNEL_AUTO) return kernel_of_id(forced);
  int32_t id = GMM_KERNEL_AUTO;
  if (gmmk::tuning_lookup(gmmk::tuning_rows_log2(m, num_total_groups), k, n, num_total_groups, transpose_rhs != 0,
                          out_dtype, &id, raster))
    return kernel_of_id(id);
  if (m >= int64_t(1024) * num_total_groups) return BF16Kernel::kPair;
  if (m >= int64_t(16) * num_total_groups) return BF16Kernel::kSwapPair;
  return BF16Kernel::kSwap;
}

// Every field of the caller's options in range (GMM_ERR_SHAPE otherwise).
bool options_valid(const gmm_options& o) {
  return o.bf16_kernel >= GMM_KERNEL_AUTO && o.bf16_kernel <= GMM_KERNEL_SINGLE && o.e4m3_kernel >= GMM_E4M3_AUTO &&
         o.e4m3_kernel <= GMM_E4M3_DECODE && o.act_split >= GMM_SPLIT_AUTO && o.act_split <= GMM_SPLIT_KERNEL &&
         o.tgmm_kernel >= GMM_TGMM_AUTO && o.tgmm_kernel <= GMM_TGMM_PAIR && o.wait_limit_cycles >= 0 &&
         o.test_drop_stage >= 0 && o.reserved == 0;
}

// GMM_LOG: one line per call on stderr when the variable is set and not "0".
bool log_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("GMM_LOG");
    return v != nullptr && v[0] != '\0' && std::strcmp(v, "0") != 0;
  }();
  return on;
}

const char* dtype_name(int d) {
  static const char* names[] = {"bf16", "f32", "e4m3", "e5m2", "int8", "int4", "uint4", "e2m1", "e8m0"};
  return d >= 0 && d <= GMM_DTYPE_E8M0 ? names[d] : "?";
}

}  // namespace

extern "C" {

size_t gmm_workspace_bytes(void) { return kWorkspaceBytes; }

size_t gmm_workspace_bytes_for(int64_t m, int64_t k, int64_t n, int32_t num_total_groups, int32_t num_local_groups,
                               int lhs_dtype, int rhs_dtype) {
  (void)n, (void)num_total_groups, (void)num_local_groups;
  if (m < 0 || k < 0) return 0;
  const bool split = lhs_dtype == GMM_DTYPE_BF16 && rhs_dtype >= GMM_DTYPE_E4M3 && rhs_dtype <= GMM_DTYPE_E2M1;
  if (!split) return kWorkspaceMinBytes;
  // int8 and int4: the fp16 split, 2 m k bytes, then (scale, mark) per 128-wide step
  const bool intw = rhs_dtype == GMM_DTYPE_INT8 || rhs_dtype == GMM_DTYPE_INT4;
  const int64_t step = intw ? 128 : 256;
  const size_t scales_at = (kActOffset + size_t((intw ? 2 : 4) * m * k) + 255) & ~size_t(255);
  return scales_at + size_t(m * ((k + step - 1) / step)) * 2 * sizeof(float);
}

const char* gmm_status_string(int status) {
  switch (status) {
    case GMM_OK: return "ok";
    case GMM_ERR_NULL: return "a required pointer is NULL";
    case GMM_ERR_DTYPE: return "unsupported dtype combination";
    case GMM_ERR_SHAPE: return "inconsistent or unsupported sizes";
    case GMM_ERR_ALIGN: return "pointer or row pitch not 16-byte aligned";
    case GMM_ERR_GROUP_OFFSET: return "group_offset out of range";
    case GMM_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case GMM_ERR_ARCH: return "current device is not compute capability 10.3";
    case GMM_ERR_CUDA: return "CUDA call failed";
    case GMM_ERR_IO: return "tiling-table file could not be read, parsed or written";
    case GMM_ERR_DEVICE_GROUP_SIZES: return "the device saw negative group sizes or sizes summing past m";
    case GMM_ERR_TIMEOUT: return "an internal pipeline wait gave up (the call's output is undefined)";
  }
  return "unknown status";
}

int gmm_last_cuda_error(void) { return t_last_cuda_error; }

int gmm_read_device_errors(void* workspace, void* stream, uint32_t* flags) {
  if (workspace == nullptr || flags == nullptr) return GMM_ERR_NULL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpy(flags, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(workspace, 0, sizeof(uint32_t));
  if (e != cudaSuccess) return cuda_fail(e);
  return GMM_OK;
}

int gmm_get_device_error(void* workspace, void* stream) {
  uint32_t flags = 0;
  if (int st = gmm_read_device_errors(workspace, stream, &flags)) return st;
  if (flags & GMM_DEVERR_TIMEOUT) return GMM_ERR_TIMEOUT;
  if (flags & (GMM_DEVERR_NEGATIVE_GROUP_SIZE | GMM_DEVERR_GROUP_SIZES_EXCEED_M)) return GMM_ERR_DEVICE_GROUP_SIZES;
  if (flags & GMM_DEVERR_GROUP_OFFSET) return GMM_ERR_GROUP_OFFSET;
  return GMM_OK;
}

}  // extern "C"

namespace {

// The arguments only gmm_ex takes: activation scales and the storage of rhs_scale.
struct ExtArgs {
  const float* lhs_scale = nullptr;
  int32_t num_lhs_blocks = 0;
  int rhs_scale_dtype = GMM_DTYPE_F32;
  const void* rhs_block_scale = nullptr;  // microscaling: [L, n, k / block_size]
  int rhs_block_scale_dtype = GMM_DTYPE_E8M0;
  int32_t block_size = 0;
};

// Shared body of gmm and gmm_into: zero_rest says whether rows of the
// groups outside the local slice are written as zero (gmm) or left as the
// caller filled them (gmm_into).
int gmm_impl(const void* lhs, int lhs_dtype, int64_t m, int64_t k, const void* rhs, int rhs_dtype,
             int32_t num_local_groups, int64_t n, int transpose_rhs, const int32_t* group_sizes,
             int32_t num_total_groups, int32_t group_offset, const void* rhs_scale, int32_t num_quant_blocks,
             const void* rhs_bias, int bias_dtype, void* out, int out_dtype, void* workspace,
             size_t workspace_bytes, void* stream, int32_t zero_rest, const int32_t* group_offset_dev,
             const gmm_options* options = nullptr, int32_t forced_raster = 0, const ExtArgs& ext = ExtArgs{},
             const char* entry = "gmm") {
  if (lhs == nullptr || rhs == nullptr || group_sizes == nullptr || out == nullptr) return GMM_ERR_NULL;
  const gmm_options opt = options != nullptr ? *options : gmm_options{};
  if (!options_valid(opt)) return GMM_ERR_SHAPE;
  const int forced_kernel = opt.bf16_kernel;
  // e4m3 activations (W8A8) run on the fp8 kernels only: 8- or 4-bit weights.
  const bool lhs8 = lhs_dtype == GMM_DTYPE_E4M3;
  if (lhs_dtype != GMM_DTYPE_BF16 && !lhs8) return GMM_ERR_DTYPE;
  if (lhs8 && rhs_dtype == GMM_DTYPE_BF16) return GMM_ERR_DTYPE;
  if (!lhs8 && ext.lhs_scale != nullptr) return GMM_ERR_DTYPE;
  const bool scale_e8m0 = ext.rhs_scale_dtype == GMM_DTYPE_E8M0;
  if (ext.rhs_scale_dtype != GMM_DTYPE_F32 && !scale_e8m0) return GMM_ERR_DTYPE;
  if (scale_e8m0 && rhs_dtype == GMM_DTYPE_BF16) return GMM_ERR_DTYPE;
  // Microscaling, on the decoding kernel with bf16 activations: MXFP8 (e4m3
  // weights, an E8M0 scale per 32 k of a weight row) or NVFP4 (e2m1 weights,
  // an e4m3 scale per 16 k).
  const bool mx = ext.rhs_block_scale != nullptr;
  const bool nvfp4 = mx && rhs_dtype == GMM_DTYPE_E2M1;
  if (mx) {
    const bool mxfp8 = rhs_dtype == GMM_DTYPE_E4M3 && ext.rhs_block_scale_dtype == GMM_DTYPE_E8M0;
    const bool fp4 = nvfp4 && ext.rhs_block_scale_dtype == GMM_DTYPE_E4M3;
    if ((!mxfp8 && !fp4) || lhs8 || !transpose_rhs || scale_e8m0) return GMM_ERR_DTYPE;
    if (ext.block_size != (fp4 ? 16 : 32)) return GMM_ERR_SHAPE;
  }
  if (rhs_dtype < GMM_DTYPE_BF16 || rhs_dtype > GMM_DTYPE_E2M1 || rhs_dtype == GMM_DTYPE_F32) return GMM_ERR_DTYPE;
  if (out_dtype != GMM_DTYPE_BF16 && out_dtype != GMM_DTYPE_F32) return GMM_ERR_DTYPE;
  if (rhs_bias != nullptr && bias_dtype != GMM_DTYPE_BF16 && bias_dtype != GMM_DTYPE_F32) return GMM_ERR_DTYPE;
  const bool quantized = rhs_dtype != GMM_DTYPE_BF16;
  const bool packed4 = rhs_dtype == GMM_DTYPE_INT4 || rhs_dtype == GMM_DTYPE_UINT4 || rhs_dtype == GMM_DTYPE_E2M1;
  if (quantized && !transpose_rhs) return GMM_ERR_DTYPE;
  if (!fits_i32(m) || !fits_i32(k) || !fits_i32(n) || k < 8 || n < 8 || k % 8 != 0 || n % 8 != 0)
    return GMM_ERR_SHAPE;
  if (num_total_groups < 1 || num_total_groups > GMM_MAX_GROUPS || num_local_groups < 1 ||
      num_local_groups > num_total_groups)
    return GMM_ERR_SHAPE;
  // A device-side offset is checked by the kernels (GMM_DEVERR_GROUP_OFFSET).
  if (group_offset_dev == nullptr && (group_offset < 0 || group_offset > num_total_groups - num_local_groups))
    return GMM_ERR_GROUP_OFFSET;
  if (group_offset_dev != nullptr && reinterpret_cast<uintptr_t>(group_offset_dev) % 4 != 0) return GMM_ERR_ALIGN;
  const bool scaled_path = quantized || rhs_scale != nullptr;
  if (rhs_scale != nullptr) {
    if (num_quant_blocks < 1 || k % num_quant_blocks != 0) return GMM_ERR_SHAPE;
  }
  if (ext.lhs_scale != nullptr) {
    if (ext.num_lhs_blocks < 1 || k % ext.num_lhs_blocks != 0 || (k / ext.num_lhs_blocks) % 128 != 0)
      return GMM_ERR_SHAPE;
    if (reinterpret_cast<uintptr_t>(ext.lhs_scale) % 4 != 0) return GMM_ERR_ALIGN;
  }
  // Block-scaled / e4m3 path: NT layout, k and the quant-block width multiples of 128.
  const int32_t nb = rhs_scale != nullptr ? num_quant_blocks : 1;
  if (scaled_path) {
    if (!transpose_rhs) return GMM_ERR_DTYPE;
    if (k % 128 != 0 || (k / nb) % 128 != 0) return GMM_ERR_SHAPE;
  }
  if (!aligned16(lhs) || !aligned16(rhs) || !aligned16(out) || (rhs_bias && !aligned16(rhs_bias)) ||
      (rhs_scale && !aligned16(rhs_scale)))
    return GMM_ERR_ALIGN;
  if (rhs_dtype == GMM_DTYPE_E2M1 && (reinterpret_cast<uintptr_t>(rhs) & 31u) != 0) return GMM_ERR_ALIGN;
  // the e4m3 decoding kernel takes bf16 activations and f32 scales
  if (rhs_dtype == GMM_DTYPE_E4M3 && opt.e4m3_kernel == GMM_E4M3_DECODE && (lhs8 || scale_e8m0)) return GMM_ERR_DTYPE;
  if (workspace == nullptr || workspace_bytes < kWorkspaceMinBytes || !aligned16(workspace)) return GMM_ERR_WORKSPACE;
  DeviceInfo dev;
  if (int st = current_device(&dev)) return st;
  if (m == 0) return GMM_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* err = static_cast<uint32_t*>(workspace);

  if (scaled_path) {
    const int64_t items = ((m + 15) / 16 + num_local_groups) * ((n + 127) / 128);
    if (items > INT32_MAX) return GMM_ERR_SHAPE;
    gmmk::ScaledLaunch S{};
    {
      // bf16 rows in {64 k, 16 rows} boxes, e4m3 rows in {128 k, 16 rows} boxes (128 bytes wide either way)
      const uint64_t dims[2] = {uint64_t(k), uint64_t(m)};
      const uint32_t box[2] = {lhs8 ? 128u : 64u, 16};
      if (int st = make_map(&S.tm_lhs, lhs8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                            lhs8 ? 1 : 2, 2, lhs, dims, box, CU_TENSOR_MAP_SWIZZLE_128B))
        return st;
    }
    if (nvfp4) {
      // packed e2m1 bytes for the decoders: {64 bytes (128 k), 128 rows} boxes, unswizzled
      const uint64_t dims[3] = {uint64_t(k / 2), uint64_t(n), uint64_t(num_local_groups)};
      const uint32_t box[3] = {64u, 128u, 1u};
      if (int st = make_map(&S.tm_rhs, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 3, rhs, dims, box,
                            CU_TENSOR_MAP_SWIZZLE_NONE))
        return st;
    } else if (rhs_dtype == GMM_DTYPE_E2M1) {
      if (int st = make_map_e2m1(&S.tm_rhs, rhs, k, n, num_local_groups)) return st;
    } else {
      // Weight rows as bytes: k of an 8-bit format, k / 2 of a 4-bit one; bf16 as elements.
      const uint64_t row = packed4 ? uint64_t(k / 2) : uint64_t(k);
      const uint64_t dims[3] = {row, uint64_t(n), uint64_t(num_local_groups)};
      const uint32_t box[3] = {quantized ? 128u : 64u, 128u, 1u};
      if (int st = make_map(&S.tm_rhs, quantized ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                            quantized ? 1 : 2, 3, rhs, dims, box, CU_TENSOR_MAP_SWIZZLE_128B))
        return st;
    }
    S.group_sizes = group_sizes;
    S.num_total_groups = num_total_groups;
    S.group_offset = group_offset;
    S.num_local_groups = num_local_groups;
    S.m = int32_t(m);
    S.n = int32_t(n);
    S.k = int32_t(k);
    S.scale = rhs_scale;
    S.num_blocks = nb;
    S.bias = rhs_bias;
    S.bias_f32 = bias_dtype == GMM_DTYPE_F32 ? 1 : 0;
    S.out = out;
    S.err = err;
    S.zero_rest = zero_rest;
    S.group_offset_dev = group_offset_dev;
    S.scale_e8m0 = scale_e8m0 ? 1 : 0;
    S.lhs_e4m3 = lhs8 ? 1 : 0;
    S.lhs_scale = ext.lhs_scale;
    S.num_lhs_blocks = ext.lhs_scale != nullptr ? ext.num_lhs_blocks : 1;
    S.mx_scale = static_cast<const uint8_t*>(ext.rhs_block_scale);
    S.lhs_raw = lhs;
    S.rhs_raw = rhs;
    const bool f32 = out_dtype == GMM_DTYPE_F32;
    // 1: split pass when the workspace holds it, 2: the pass or GMM_ERR_WORKSPACE, 0: in the kernel
    const int act_split = opt.act_split == GMM_SPLIT_KERNEL ? 0 : (opt.act_split == GMM_SPLIT_PASS ? 2 : 1);
    // The fp8 kernels; bf16 activations are split once per row into the
    // workspace when it has room (act_split.cu), in the kernel's k steps.
    // The fp16 split (2 m k bytes of fp16 values, then (scale, mark) per
    // 128-wide step) and the fp16-MMA kernel (gemm_f16w.cu) on launch `L`; -1
    // when the workspace cannot hold the split.
    auto run_f16w = [&](gmmk::ScaledLaunch& L, int fmt) -> int {
      {
        const int64_t ksteps = k / 128;
        const size_t scales_at = (kActOffset + size_t(2 * m * k) + 255) & ~size_t(255);
        const size_t end = scales_at + size_t(m * ksteps) * 2 * sizeof(float);
        if (end <= workspace_bytes) {
          uint8_t* plane = static_cast<uint8_t*>(workspace) + kActOffset;
          float* scales = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + scales_at);
          // the plane as [k / 64, m, 64]: a {64, 16, 2} box is a step's two
          // 128-byte swizzled atoms of 16 rows, one after the other
          const uint64_t dims[3] = {64u, uint64_t(m), uint64_t(k / 64)};
          const uint64_t strides[2] = {uint64_t(2 * k), 128u};
          const uint32_t box[3] = {64u, 16u, 2u};
          if (int st = make_map_strided(&L.tm_lhs, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, plane, dims, strides, box,
                                        CU_TENSOR_MAP_SWIZZLE_128B))
            return st;
          L.lhs_split = 1;
          L.lhs_scale = scales;
          L.num_lhs_blocks = int32_t(ksteps);
          // 4-bit codes come out of their rewrite as k (0, 4), (1, 5), ..: the split
          // stores those rows in the same order
          const bool perm = fmt == gmmk::kWeightInt4 || fmt == gmmk::kWeightUint4 || fmt == gmmk::kWeightE2M1;
          if (cudaError_t e1 = gmmk::launch_act_split_f16(lhs, m, k, plane, scales, err + 1, perm, s))
            return cuda_fail(e1);
          if (log_enabled())
            std::fprintf(stderr, "libgmm: %s m=%lld k=%lld n=%lld groups=%d local=%d offset=%s lhs=%s rhs=%s out=%s "
                                 "kernel=f16w split=f16\n",
                         entry, (long long)m, (long long)k, (long long)n, num_total_groups, num_local_groups,
                         group_offset_dev ? "device" : "host", dtype_name(lhs_dtype), dtype_name(rhs_dtype),
                         dtype_name(out_dtype));
          if (cudaError_t e2 = gmmk::launch_f16w(L, fmt, f32, dev.sms, s)) return cuda_fail(e2);
          return GMM_OK;
        }
      }
      return -1;
    };
    auto fp8_kernel = [&](int fmt) -> int {
      // int8 and int4 with bf16 activations: the fp16 split and the fp16-MMA
      // kernel, when the workspace holds the split; else the e4m3 path below.
      // uint4 stays on the e4m3 path: its code table makes the e4m3 rewrite
      // cheap, and there the e4m3 kernel measured faster (120 us against 129 us
      // on the decode workload; int4 131 against 136, int8 124 against 229).
      const bool intw = fmt == gmmk::kWeightInt8 || fmt == gmmk::kWeightInt4;
      if (!lhs8 && act_split != 0 && intw) {
        const int r = run_f16w(S, fmt);
        if (r != -1) return r;
        if (act_split == 2) return GMM_ERR_WORKSPACE;
      }
      if (!lhs8 && act_split != 0 && !intw) {
        const int32_t step = fmt == gmmk::kWeightInt8 ? 128 : 256;
        const int64_t ksteps = (k + step - 1) / step;
        const size_t scales_at = (kActOffset + size_t(4 * m * k) + 255) & ~size_t(255);
        const size_t end = scales_at + size_t(m * ksteps) * 2 * sizeof(float);
        if (end <= workspace_bytes) {
          uint8_t* planes = static_cast<uint8_t*>(workspace) + kActOffset;
          float* scales = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + scales_at);
          const uint64_t dims[3] = {uint64_t(k), uint64_t(m), 4};
          const uint32_t box[3] = {128u, 8u, 4u};
          if (int st = make_map(&S.tm_lhs, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 3, planes, dims, box,
                                CU_TENSOR_MAP_SWIZZLE_128B))
            return st;
          S.lhs_split = 1;
          S.lhs_scale = scales;
          S.num_lhs_blocks = int32_t(ksteps);
          if (cudaError_t e1 = gmmk::launch_act_split(lhs, m, k, step, planes, scales, err + 1, s))
            return cuda_fail(e1);
        } else if (act_split == 2) {
          return GMM_ERR_WORKSPACE;
        }
      }
      if (log_enabled())
        std::fprintf(stderr, "libgmm: %s m=%lld k=%lld n=%lld groups=%d local=%d offset=%s lhs=%s rhs=%s out=%s "
                             "kernel=fp8 split=%s\n",
                     entry, (long long)m, (long long)k, (long long)n, num_total_groups, num_local_groups,
                     group_offset_dev ? "device" : "host", dtype_name(lhs_dtype), dtype_name(rhs_dtype),
                     dtype_name(out_dtype), lhs8 ? "none" : (S.lhs_split ? "pass" : "kernel"));
      if (cudaError_t e2 = gmmk::launch_fp8(S, fmt, f32, dev.sms, s)) return cuda_fail(e2);
      return GMM_OK;
    };
    auto log_decoding = [&] {
      if (log_enabled())
        std::fprintf(stderr, "libgmm: %s m=%lld k=%lld n=%lld groups=%d local=%d offset=%s lhs=%s rhs=%s out=%s "
                             "kernel=decoding%s\n",
                     entry, (long long)m, (long long)k, (long long)n, num_total_groups, num_local_groups,
                     group_offset_dev ? "device" : "host", dtype_name(lhs_dtype), dtype_name(rhs_dtype),
                     dtype_name(out_dtype), mx ? " block-scales" : "");
    };
    cudaError_t e;
    if (rhs_dtype == GMM_DTYPE_BF16) {
      log_decoding();
      e = gmmk::launch_scaled(S, false, f32, dev.sms, s);
    } else if (rhs_dtype == GMM_DTYPE_E4M3) {
      const bool decode = opt.e4m3_kernel == GMM_E4M3_DECODE;
      if (!decode && !mx) return fp8_kernel(gmmk::kWeightE4M3);
      // MXFP8 with bf16 activations on the fp16-MMA kernel (e4m3 codes are fp16
      // values; each 32-k block sums into its own accumulator and is scaled by its
      // power of two after) when the scales are 4-byte aligned and the workspace
      // holds the split; else (or with GMM_E4M3_DECODE) the decoding kernel, which
      // applies the per-32 scales as it decodes.
      if (mx && !decode && act_split != 0 && reinterpret_cast<uintptr_t>(ext.rhs_block_scale) % 4 == 0) {
        const int r = run_f16w(S, gmmk::kWeightE4M3);
        if (r != -1) return r;
        if (act_split == 2) return GMM_ERR_WORKSPACE;
      }
      log_decoding();
      e = gmmk::launch_scaled(S, true, f32, dev.sms, s);
    } else if (nvfp4) {
      // NVFP4 with bf16 activations on the fp16-MMA kernel (each code times its
      // block scale is exact in fp16) when k % 256 == 0 (the block scales'
      // rows, k / 16 bytes, are then whole 16-byte units for TMA), the scales
      // are 16-byte aligned and the workspace holds the split; else the
      // decoding kernel.
      if (act_split != 0 && k % 256 == 0 && aligned16(ext.rhs_block_scale)) {
        gmmk::ScaledLaunch L2 = S;
        const uint64_t wdims[3] = {uint64_t(k / 2), uint64_t(n), uint64_t(num_local_groups)};
        const uint32_t wbox[3] = {128u, 128u, 1u};
        if (int st = make_map(&L2.tm_rhs, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 3, rhs, wdims, wbox,
                              CU_TENSOR_MAP_SWIZZLE_128B))
          return st;
        const uint64_t sdims[3] = {uint64_t(k / 16), uint64_t(n), uint64_t(num_local_groups)};
        const uint32_t sbox[3] = {16u, 128u, 1u};
        if (int st = make_map(&L2.tm_bs, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 3, ext.rhs_block_scale, sdims, sbox,
                              CU_TENSOR_MAP_SWIZZLE_NONE))
          return st;
        const int r = run_f16w(L2, gmmk::kWeightE2M1);
        if (r != -1) return r;
        if (act_split == 2) return GMM_ERR_WORKSPACE;
      }
      log_decoding();
      e = gmmk::launch_scaled_nvfp4(S, f32, dev.sms, s);
    } else {
      const int fmt = rhs_dtype == GMM_DTYPE_E5M2   ? gmmk::kWeightE5M2
                      : rhs_dtype == GMM_DTYPE_INT8  ? gmmk::kWeightInt8
                      : rhs_dtype == GMM_DTYPE_INT4  ? gmmk::kWeightInt4
                      : rhs_dtype == GMM_DTYPE_UINT4 ? gmmk::kWeightUint4
                                                     : gmmk::kWeightE2M1;
      return fp8_kernel(fmt);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    return GMM_OK;
  }

  int32_t raster = 0;
  const BF16Kernel kind =
      choose_bf16_kernel(m, k, n, num_total_groups, transpose_rhs, out_dtype, forced_kernel, &raster);
  if (kind == BF16Kernel::kInvalid) return GMM_ERR_SHAPE;
  if (forced_kernel != GMM_KERNEL_AUTO) raster = forced_raster;
  gmmk::GemmLaunch L{};
  {
    const uint64_t dims[2] = {uint64_t(k), uint64_t(m)};
    const bool swapped = kind == BF16Kernel::kSwap || kind == BF16Kernel::kSwapPair;
    const uint32_t box[2] = {64, swapped ? 64u : 128u};
    if (int st = make_map(&L.tm_lhs, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 2, lhs, dims, box,
                          CU_TENSOR_MAP_SWIZZLE_128B))
      return st;
  }
  if (transpose_rhs) {
    const uint64_t dims[3] = {uint64_t(k), uint64_t(n), uint64_t(num_local_groups)};
    const uint32_t box[3] = {64, kind == BF16Kernel::kSingle ? 256u : 128u, 1};
    if (int st = make_map(&L.tm_rhs, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 3, rhs, dims, box,
                          CU_TENSOR_MAP_SWIZZLE_128B))
      return st;
  } else {
    const uint64_t dims[3] = {uint64_t(n), uint64_t(k), uint64_t(num_local_groups)};
    const uint32_t box[3] = {64, 64, 1};
    if (int st = make_map(&L.tm_rhs, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 3, rhs, dims, box,
                          CU_TENSOR_MAP_SWIZZLE_128B))
      return st;
  }
  L.group_sizes = group_sizes;
  L.num_total_groups = num_total_groups;
  L.group_offset = group_offset;
  L.num_local_groups = num_local_groups;
  L.m = int32_t(m);
  L.n = int32_t(n);
  L.k = int32_t(k);
  L.out = out;
  L.bias = rhs_bias;
  L.bias_f32 = bias_dtype == GMM_DTYPE_F32 ? 1 : 0;
  L.err = err;
  // Default tile order: group by group, blocks of 4096 rows (16 pair tiles, 32
  // one-SM tiles) meeting the n tiles in turn, so that every weight tile and
  // every lhs row block comes from DRAM once (on the Mixtral up-projection the
  // pair kernel's DRAM reads drop from 1.74x to 1.03x the algorithmic bytes).
  L.raster = raster != 0 ? raster : (kind == BF16Kernel::kPair ? -16 : -32);
  L.zero_rest = zero_rest;
  L.group_offset_dev = group_offset_dev;
  L.wait_limit = opt.wait_limit_cycles;
  L.drop_stage = opt.test_drop_stage;
  if (log_enabled()) {
    static const char* kname[] = {"single", "pair", "swap_pair", "swap", "single"};
    const int id = kind == BF16Kernel::kPair ? 1 : kind == BF16Kernel::kSwapPair ? 2 : kind == BF16Kernel::kSwap ? 3 : 4;
    std::fprintf(stderr, "libgmm: %s m=%lld k=%lld n=%lld groups=%d local=%d offset=%s layout=%s out=%s kernel=%s "
                         "raster=%d\n",
                 entry, (long long)m, (long long)k, (long long)n, num_total_groups, num_local_groups,
                 group_offset_dev ? "device" : "host", transpose_rhs ? "nt" : "nn", dtype_name(out_dtype), kname[id],
                 L.raster);
  }
  // Work items (row tiles x n tiles, at most (m/128 + groups) x n/128) must fit in int32.
  const int64_t m_tiles_max = (m + 127) / 128 + num_local_groups;
  if (m_tiles_max * ((n + 127) / 128) > INT32_MAX) return GMM_ERR_SHAPE;
  const bool nt = transpose_rhs != 0, f32 = out_dtype == GMM_DTYPE_F32;
  cudaError_t e = kind == BF16Kernel::kPair       ? gmmk::launch_gemm_bf16_2sm(L, nt, f32, dev.sms, s)
                  : kind == BF16Kernel::kSwapPair ? gmmk::launch_gemm_bf16_2sm_swap(L, nt, f32, dev.sms, s)
                  : kind == BF16Kernel::kSwap     ? gmmk::launch_gemm_bf16_swap(L, nt, f32, dev.sms, s)
                                                  : gmmk::launch_gemm_bf16(L, nt, f32, dev.sms, s);
  if (e != cudaSuccess) return cuda_fail(e);
  return GMM_OK;
}

}  // namespace

extern "C" {

int gmm(const void* lhs, int lhs_dtype, int64_t m, int64_t k, const void* rhs, int rhs_dtype,
        int32_t num_local_groups, int64_t n, int transpose_rhs, const int32_t* group_sizes,
        int32_t num_total_groups, int32_t group_offset, const float* rhs_scale, int32_t num_quant_blocks,
        const void* rhs_bias, int bias_dtype, void* out, int out_dtype, void* workspace, size_t workspace_bytes,
        void* stream) {
  return gmm_impl(lhs, lhs_dtype, m, k, rhs, rhs_dtype, num_local_groups, n, transpose_rhs, group_sizes,
                  num_total_groups, group_offset, rhs_scale, num_quant_blocks, rhs_bias, bias_dtype, out,
                  out_dtype, workspace, workspace_bytes, stream, 1, nullptr);
}

int gmm_into(const void* lhs, int lhs_dtype, int64_t m, int64_t k, const void* rhs, int rhs_dtype,
             int32_t num_local_groups, int64_t n, int transpose_rhs, const int32_t* group_sizes,
             int32_t num_total_groups, int32_t group_offset, const float* rhs_scale, int32_t num_quant_blocks,
             const void* rhs_bias, int bias_dtype, void* out, int out_dtype, void* workspace,
             size_t workspace_bytes, void* stream) {
  return gmm_impl(lhs, lhs_dtype, m, k, rhs, rhs_dtype, num_local_groups, n, transpose_rhs, group_sizes,
                  num_total_groups, group_offset, rhs_scale, num_quant_blocks, rhs_bias, bias_dtype, out,
                  out_dtype, workspace, workspace_bytes, stream, 0, nullptr, nullptr, 0, ExtArgs{}, "gmm_into");
}

int gmm_device_offset(const void* lhs, int lhs_dtype, int64_t m, int64_t k, const void* rhs, int rhs_dtype,
                      int32_t num_local_groups, int64_t n, int transpose_rhs, const int32_t* group_sizes,
                      int32_t num_total_groups, const int32_t* group_offset, const float* rhs_scale,
                      int32_t num_quant_blocks, const void* rhs_bias, int bias_dtype, void* out, int out_dtype,
                      int keep_other_rows, void* workspace, size_t workspace_bytes, void* stream) {
  if (group_offset == nullptr) return GMM_ERR_NULL;
  return gmm_impl(lhs, lhs_dtype, m, k, rhs, rhs_dtype, num_local_groups, n, transpose_rhs, group_sizes,
                  num_total_groups, 0, rhs_scale, num_quant_blocks, rhs_bias, bias_dtype, out, out_dtype, workspace,
                  workspace_bytes, stream, keep_other_rows ? 0 : 1, group_offset, nullptr, 0, ExtArgs{},
                  "gmm_device_offset");
}

int gmm_ex(const void* lhs, int lhs_dtype, const float* lhs_scale, int32_t num_lhs_blocks, int64_t m, int64_t k,
           const void* rhs, int rhs_dtype, int32_t num_local_groups, int64_t n, int transpose_rhs,
           const int32_t* group_sizes, int32_t num_total_groups, int32_t group_offset,
           const int32_t* group_offset_dev, const void* rhs_scale, int rhs_scale_dtype, int32_t num_quant_blocks,
           const void* rhs_block_scale, int rhs_block_scale_dtype, int32_t block_size, const void* rhs_bias,
           int bias_dtype, void* out, int out_dtype, int keep_other_rows, const gmm_options* options, void* workspace,
           size_t workspace_bytes, void* stream) {
  ExtArgs ext;
  ext.lhs_scale = lhs_scale;
  ext.num_lhs_blocks = num_lhs_blocks;
  ext.rhs_scale_dtype = rhs_scale_dtype;
  ext.rhs_block_scale = rhs_block_scale;
  ext.rhs_block_scale_dtype = rhs_block_scale_dtype;
  ext.block_size = block_size;
  return gmm_impl(lhs, lhs_dtype, m, k, rhs, rhs_dtype, num_local_groups, n, transpose_rhs, group_sizes,
                  num_total_groups, group_offset, rhs_scale, num_quant_blocks, rhs_bias, bias_dtype, out, out_dtype,
                  workspace, workspace_bytes, stream, keep_other_rows ? 0 : 1, group_offset_dev, options, 0, ext,
                  "gmm_ex");
}

int gmm_quantize_e4m3(const void* x, int x_dtype, int64_t m, int64_t k, int64_t group, void* q, float* scale,
                      void* stream) {
  if (x == nullptr || q == nullptr || scale == nullptr) return GMM_ERR_NULL;
  if (x_dtype != GMM_DTYPE_BF16) return GMM_ERR_DTYPE;
  if (m < 0 || k < 0 || (group != 64 && group != 128 && group != 256) || k % group != 0) return GMM_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(q) || reinterpret_cast<uintptr_t>(scale) % 4 != 0) return GMM_ERR_ALIGN;
  DeviceInfo dev;
  if (int st = current_device(&dev)) return st;
  cudaError_t e = gmmk::launch_quantize_e4m3(x, m, k, group, q, scale, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return GMM_OK;
}

int gmm_tune(const void* lhs, int lhs_dtype, int64_t m, int64_t k, const void* rhs, int rhs_dtype,
             int32_t num_local_groups, int64_t n, int transpose_rhs, const int32_t* group_sizes,
             int32_t num_total_groups, int32_t group_offset, const void* rhs_bias, int bias_dtype, void* out,
             int out_dtype, void* workspace, size_t workspace_bytes, void* stream, int iterations, int* kernel,
             int* raster, float* ms) {
  if (kernel == nullptr || raster == nullptr || ms == nullptr) return GMM_ERR_NULL;
  if (rhs_dtype != GMM_DTYPE_BF16) return GMM_ERR_DTYPE;
  if (iterations < 1 || iterations > 1000) return GMM_ERR_SHAPE;
  struct Candidate {
    int kernel;
    int32_t raster;
  };
  static const Candidate kCandidates[] = {{GMM_KERNEL_PAIR, -16},    {GMM_KERNEL_PAIR, -4}, {GMM_KERNEL_PAIR, 8},
                                          {GMM_KERNEL_SWAP_PAIR, 0}, {GMM_KERNEL_SWAP, 0},  {GMM_KERNEL_SINGLE, -32}};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaEvent_t t0 = nullptr, t1 = nullptr;
  cudaError_t e = cudaEventCreate(&t0);
  if (e == cudaSuccess) e = cudaEventCreate(&t1);
  if (e != cudaSuccess) {
    if (t0) cudaEventDestroy(t0);
    return cuda_fail(e);
  }
  int status = GMM_OK;
  float best = -1.f;
  Candidate chosen{GMM_KERNEL_AUTO, 0};
  for (const Candidate& c : kCandidates) {
    gmm_options o{};
    o.bf16_kernel = c.kernel;
    auto run = [&]() {
      return gmm_impl(lhs, lhs_dtype, m, k, rhs, rhs_dtype, num_local_groups, n, transpose_rhs, group_sizes,
                      num_total_groups, group_offset, nullptr, 0, rhs_bias, bias_dtype, out, out_dtype, workspace,
                      workspace_bytes, stream, 1, nullptr, &o, c.raster, ExtArgs{}, "gmm_tune");
    };
    status = run();  // warm-up; also validates the arguments
    if (status != GMM_OK) break;
    if ((e = cudaEventRecord(t0, s)) != cudaSuccess) break;
    for (int i = 0; i < iterations && status == GMM_OK; ++i) status = run();
    if (status != GMM_OK) break;
    if ((e = cudaEventRecord(t1, s)) != cudaSuccess || (e = cudaEventSynchronize(t1)) != cudaSuccess) break;
    float elapsed = 0.f;
    if ((e = cudaEventElapsedTime(&elapsed, t0, t1)) != cudaSuccess) break;
    elapsed /= float(iterations);
    if (best < 0.f || elapsed < best) {
      best = elapsed;
      chosen = c;
    }
  }
  cudaEventDestroy(t0);
  cudaEventDestroy(t1);
  if (status != GMM_OK) return status;
  if (e != cudaSuccess) return cuda_fail(e);
  gmmk::tuning_store(gmmk::tuning_rows_log2(m, num_total_groups), k, n, num_total_groups, transpose_rhs != 0,
                     out_dtype, chosen.kernel, chosen.raster);
  *kernel = chosen.kernel;
  *raster = chosen.raster;
  *ms = best;
  return GMM_OK;
}

int tgmm_ex(const void* lhs, int lhs_dtype, const void* dout, int dout_dtype, int64_t m, int64_t k, int64_t n,
            const int32_t* group_sizes, int32_t num_total_groups, int32_t group_offset, int32_t num_local_groups,
            void* out, int out_dtype, const gmm_options* options, void* workspace, size_t workspace_bytes,
            void* stream) {
  const gmm_options opt = options != nullptr ? *options : gmm_options{};
  if (!options_valid(opt)) return GMM_ERR_SHAPE;
  if (lhs == nullptr || dout == nullptr || group_sizes == nullptr || out == nullptr) return GMM_ERR_NULL;
  if (lhs_dtype != GMM_DTYPE_BF16 || dout_dtype != GMM_DTYPE_BF16) return GMM_ERR_DTYPE;
  if (out_dtype != GMM_DTYPE_BF16 && out_dtype != GMM_DTYPE_F32) return GMM_ERR_DTYPE;
  if (!fits_i32(m) || !fits_i32(k) || !fits_i32(n) || k < 8 || n < 8 || k % 8 != 0 || n % 8 != 0)
    return GMM_ERR_SHAPE;
  if (num_total_groups < 1 || num_total_groups > GMM_MAX_GROUPS || num_local_groups < 1 ||
      num_local_groups > num_total_groups)
    return GMM_ERR_SHAPE;
  if (group_offset < 0 || group_offset > num_total_groups - num_local_groups) return GMM_ERR_GROUP_OFFSET;
  if (!aligned16(lhs) || !aligned16(dout) || !aligned16(out)) return GMM_ERR_ALIGN;
  if (workspace == nullptr || workspace_bytes < kWorkspaceMinBytes || !aligned16(workspace)) return GMM_ERR_WORKSPACE;
  const int64_t items = int64_t(num_local_groups) * ((k + 127) / 128) * ((n + 255) / 256);
  if (items > INT32_MAX) return GMM_ERR_SHAPE;
  DeviceInfo dev;
  if (int st = current_device(&dev)) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  gmmk::TgmmLaunch L{};
  // With m == 0 every group is empty and no copy is issued; the maps still
  // need a non-zero extent.
  const uint64_t rows = m > 0 ? uint64_t(m) : 1;
  // One SM per tile by default; options.tgmm_kernel = GMM_TGMM_PAIR selects the
  // SM-pair kernel (256 x 256 tiles; as fast on the 128-expert workload, kept for
  // comparison).
  const bool pair = opt.tgmm_kernel == GMM_TGMM_PAIR;
  // The one-SM kernel reads a chunk's 128 lhs columns and 256 dout columns as one
  // box each, over the matrices viewed as [features / 64, rows, 64] (the 64-wide
  // 128-byte swizzle atoms one after the other).  The view needs the feature
  // count to be a multiple of 64: its last atom would otherwise reach past the
  // row into the next one (and past the end of the matrix on the last row).
  auto feature_map = [&](CUtensorMap* map, const void* base, int64_t features, bool view3, uint32_t atoms) {
    if (view3) {
      const uint64_t dims[3] = {64u, rows, uint64_t(features / 64)};
      const uint64_t strides[2] = {uint64_t(2 * features), 128u};
      const uint32_t box[3] = {64u, 64u, atoms};
      return make_map_strided(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_128B);
    }
    const uint64_t dims[2] = {uint64_t(features), rows};
    const uint32_t box[2] = {64, 64};
    return make_map(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 2, base, dims, box, CU_TENSOR_MAP_SWIZZLE_128B);
  };
  L.lhs_3d = !pair && k % 64 == 0 ? 1 : 0;
  L.dout_3d = !pair && n % 64 == 0 ? 1 : 0;
  if (int st = feature_map(&L.tm_lhs, lhs, k, L.lhs_3d != 0, 2u)) return st;
  if (int st = feature_map(&L.tm_dout, dout, n, L.dout_3d != 0, 4u)) return st;
  {
    const bool f32 = out_dtype == GMM_DTYPE_F32;
    const uint64_t dims[3] = {uint64_t(n), uint64_t(k), uint64_t(num_local_groups)};
    const uint32_t box[3] = {f32 ? 32u : 64u, 32u, 1u};
    if (int st = make_map(&L.tm_out, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                          f32 ? 4 : 2, 3, out, dims, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return st;
  }
  L.group_sizes = group_sizes;
  L.num_total_groups = num_total_groups;
  L.group_offset = group_offset;
  L.num_local_groups = num_local_groups;
  L.m = int32_t(m);
  L.n = int32_t(n);
  L.k = int32_t(k);
  L.out = out;
  L.err = static_cast<uint32_t*>(workspace);
  L.wait_limit = opt.wait_limit_cycles;
  L.drop_stage = opt.test_drop_stage;
  if (log_enabled())
    std::fprintf(stderr, "libgmm: tgmm m=%lld k=%lld n=%lld groups=%d local=%d offset=%d out=%s kernel=%s\n",
                 (long long)m, (long long)k, (long long)n, num_total_groups, num_local_groups, group_offset,
                 dtype_name(out_dtype), pair ? "pair" : "single");
  cudaError_t e = pair ? gmmk::launch_tgmm_2sm(L, out_dtype == GMM_DTYPE_F32, dev.sms, s)
                       : gmmk::launch_tgmm(L, out_dtype == GMM_DTYPE_F32, dev.sms, s);
  if (e != cudaSuccess) return cuda_fail(e);
  return GMM_OK;
}

int tgmm_local(const void* lhs, int lhs_dtype, const void* dout, int dout_dtype, int64_t m, int64_t k,
               int64_t n, const int32_t* group_sizes, int32_t num_total_groups, int32_t group_offset,
               int32_t num_local_groups, void* out, int out_dtype, void* workspace, size_t workspace_bytes,
               void* stream) {
  return tgmm_ex(lhs, lhs_dtype, dout, dout_dtype, m, k, n, group_sizes, num_total_groups, group_offset,
                 num_local_groups, out, out_dtype, nullptr, workspace, workspace_bytes, stream);
}

int tgmm(const void* lhs, int lhs_dtype, const void* dout, int dout_dtype, int64_t m, int64_t k, int64_t n,
         const int32_t* group_sizes, int32_t num_groups, void* out, int out_dtype, void* workspace,
         size_t workspace_bytes, void* stream) {
  return tgmm_local(lhs, lhs_dtype, dout, dout_dtype, m, k, n, group_sizes, num_groups, 0, num_groups, out,
                    out_dtype, workspace, workspace_bytes, stream);
}

}  // extern "C"
