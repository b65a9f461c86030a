// Host-side interface between the C ABI (gmm_api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace gmmk {

// Forward grouped matmul with bf16 operands (NT or NN weight layout).
struct GemmLaunch {
  CUtensorMap tm_lhs;  // lhs [m, k], box {64, 128}, 128-byte swizzle
  CUtensorMap tm_rhs;  // NT: [L, n, k] box {64, 256, 1};  NN: [L, k, n] box {64, 64, 1}
  const int32_t* group_sizes;
  int32_t num_total_groups, group_offset, num_local_groups;
  int32_t m, n, k;
  void* out;
  const void* bias;  // NULL or [L, 1, n]
  int32_t bias_f32;  // bias dtype: 1 = f32, 0 = bf16
  uint32_t* err;
  int32_t raster;     // n-tiles per L2 super-column
  int32_t zero_rest;                // 1: zero rows outside the local groups; 0: leave them as they are
  const int32_t* group_offset_dev;  // NULL, or a device int32 that replaces group_offset
  int64_t wait_limit;               // single/pair/swap_pair: 0, or the bound of their pipeline waits (cycles)
  int32_t drop_stage;               // 0, or s > 0 (test): single: CTA 0 skips its s-th stage's copies;
                                    // pair, swap_pair: the first pair's second CTA stops before its s-th
};

cudaError_t launch_gemm_bf16(const GemmLaunch& p, bool nt, bool out_f32, int grid, cudaStream_t stream);

// Same computation on SM pairs (256 x 256 tiles, cta_group::2).  tm_rhs boxes:
// NT {64, 128, 1}; NN {64, 64, 1}.  Launches at most max_ctas CTAs.
// Same computation with the roles swapped for small groups: 128 weight rows
// on the MMA's M side, up to 256 of a group's rows on its N side.  tm_lhs box
// {64, 64}; tm_rhs boxes: NT {64, 128, 1}; NN {64, 64, 1}.
cudaError_t launch_gemm_bf16_swap(const GemmLaunch& p, bool nt, bool out_f32, int grid, cudaStream_t stream);

// Pairs with the roles swapped: 256 weight rows on the MMA's M side (128 per
// CTA), up to 256 of a group's rows on its N side.  tm_lhs box {64, 64};
// tm_rhs boxes: NT {64, 128, 1}; NN {64, 64, 1}.
cudaError_t launch_gemm_bf16_2sm_swap(const GemmLaunch& p, bool nt, bool out_f32, int max_ctas,
                                      cudaStream_t stream);

cudaError_t launch_gemm_bf16_2sm(const GemmLaunch& p, bool nt, bool out_f32, int max_ctas, cudaStream_t stream);

// tgmm: out[g] = lhs_g^T dout_g (bf16 operands, fp32 accumulate).
struct TgmmLaunch {
  CUtensorMap tm_lhs;   // lhs  [m, k], box {64, 64}; lhs_3d: [k / 64, m, 64], box {64, 64, 2}
  CUtensorMap tm_dout;  // dout [m, n], box {64, 64}; dout_3d: [n / 64, m, 64], box {64, 64, 4}
  CUtensorMap tm_out;   // out [L, k, n], box {128 bytes of n, 32, 1}
  const int32_t* group_sizes;  // [num_total_groups]
  int32_t num_total_groups, group_offset, num_local_groups;
  int32_t m, n, k;
  void* out;  // [L, k, n]: local group g is group group_offset + g
  uint32_t* err;
  int64_t wait_limit;  // pair kernel: 0, or the bound of its pipeline waits (cycles)
  int32_t drop_stage;  // pair kernel: 0, or s > 0: the first pair's second CTA stops before its s-th stage (test)
  int32_t lhs_3d, dout_3d;  // one-SM kernel: the maps are the 3D views (k % 64 == 0, n % 64 == 0)
};

cudaError_t launch_tgmm(const TgmmLaunch& p, bool out_f32, int grid, cudaStream_t stream);
// The same on SM pairs (256 x 256 output tiles, tcgen05.mma.cta_group::2).
cudaError_t launch_tgmm_2sm(const TgmmLaunch& p, bool out_f32, int max_ctas, cudaStream_t stream);

// Block-scaled grouped matmul for small groups (decode): rhs e4m3 or bf16
// [L, n, k], per-(group, k-block, n) fp32 scale, optional bias.
struct ScaledLaunch {
  CUtensorMap tm_lhs;  // lhs [m, k] bf16, box {64, 16}; e4m3 (lhs_e4m3), box {128, 16}
  CUtensorMap tm_rhs;  // rhs [L, n, k]: e4m3 box {128, 128, 1} / bf16 box {64, 128, 1}
  CUtensorMap tm_bs;   // fp16-weight kernel, NVFP4: the e4m3 block scales [L, n, k / 16], box {16, 128, 1}
  const int32_t* group_sizes;
  int32_t num_total_groups, group_offset, num_local_groups;
  int32_t m, n, k;
  const void* scale;  // NULL or [L, nb, 1, n], f32 or (scale_e8m0) E8M0 bytes
  int32_t num_blocks;
  const void* bias;
  int32_t bias_f32;
  void* out;
  uint32_t* err;
  int32_t zero_rest;                // 1: zero rows outside the local groups; 0: leave them as they are
  const int32_t* group_offset_dev;  // NULL, or a device int32 that replaces group_offset
  int32_t scale_e8m0;               // scale holds E8M0 bytes (fp8 kernels only)
  int32_t lhs_e4m3;                 // lhs holds e4m3 codes (fp8 kernels only)
  const float* lhs_scale;           // lhs_e4m3: NULL or f32 [m, num_lhs_blocks]
  int32_t num_lhs_blocks;
  const uint8_t* mx_scale;          // decoding and fp16-weight kernels: NULL, E8M0 [L, n, k / 32]
                                    // (e4m3 weights) or e4m3 [L, n, k / 16] (e2m1 weights)
  int32_t lhs_split;                // fp8 kernels: tm_lhs spans act_split's h / l / h2 / l2 planes
                                    // [4, m, k] (box {128, 8, 4}); lhs_scale its (s1, s2) step
                                    // scales [m, k steps, 2]
  const void* lhs_raw;              // fp8 kernels with bf16 lhs: the lhs itself, [m, k] bf16
  const void* rhs_raw;              // fp8 kernels: the weights as stored, [L, n, k or k / 2]
};

cudaError_t launch_scaled(const ScaledLaunch& p, bool rhs_e4m3, bool out_f32, int grid, cudaStream_t stream);
// NVFP4 on the decoding kernel: e2m1 weights (tm_rhs over the packed bytes
// [L, n, k / 2], box {64, 128, 1}, no swizzle) with e4m3 block scales per 16 k
// in mx_scale.
cudaError_t launch_scaled_nvfp4(const ScaledLaunch& p, bool out_f32, int grid, cudaStream_t stream);

// The same operation for 8- and 4-bit weights on the fp8 tensor cores (the
// bf16 activations are split exactly into two e4m3 terms; e4m3 / e5m2 weights
// are used as stored, the other formats rewritten exactly as e4m3 tiles).
// tm_rhs for the 4-bit formats spans [L, n, k / 2] bytes with box {128, 128, 1}.
enum WeightFormat : int {
  kWeightE4M3 = 0,
  kWeightE5M2 = 1,
  kWeightInt8 = 2,
  kWeightInt4 = 3,
  kWeightUint4 = 4,
  kWeightE2M1 = 5,
};
cudaError_t launch_fp8(const ScaledLaunch& p, int weight_format, bool out_f32, int grid, cudaStream_t stream);
// e4m3 activations (lhs_e4m3): the same kernel with the token rows loaded as
// e4m3 operand tiles and each 128-wide sub-tile scaled by lhs_scale.
cudaError_t launch_fp8_a8(const ScaledLaunch& p, int weight_format, bool out_f32, int grid, cudaStream_t stream);
cudaError_t launch_fp8_a8_packed(const ScaledLaunch& p, int weight_format, bool out_f32, int grid,
                                 cudaStream_t stream);
cudaError_t launch_fp8_converted(const ScaledLaunch& p, int weight_format, bool out_f32, int grid,
                                 cudaStream_t stream);
// Split activations (lhs_split), every weight format of the fp8 kernel.
cudaError_t launch_fp8_ps(const ScaledLaunch& p, int weight_format, bool out_f32, int grid, cudaStream_t stream);
cudaError_t launch_fp8_ps_converted(const ScaledLaunch& p, int weight_format, bool out_f32, int grid,
                                   cudaStream_t stream);
// The two-level e4m3 split of bf16 rows [m, k] (k % 128 == 0) into e4m3 planes
// h / l / h2 / l2 [4, m, k] and step scales (s1, s2) [m, ceil(k / step), 2], step
// 256 or 128 (the fp8 kernel's k step: 128 for int8 weights); sets *pending when a
// step is marked (act_split.cu).
cudaError_t launch_act_split(const void* x, int64_t m, int64_t k, int32_t step, void* planes, float* scale,
                             uint32_t* pending, cudaStream_t stream);
// The fp16 split of bf16 rows [m, k] (k % 128 == 0) for the fp16-MMA kernel of
// the integer formats: plane [m, k] fp16 (each 8 k in the order 0, 4, 1, 5, 2,
// 6, 3, 7 when `perm`) and (scale, mark) pairs [m, k / 128, 2]; sets *pending
// when a step is marked (act_split.cu).
cudaError_t launch_act_split_f16(const void* x, int64_t m, int64_t k, void* plane, float* scale, uint32_t* pending,
                                 bool perm, cudaStream_t stream);
// int8, int4 and uint4 weights on the fp16 tensor cores (gemm_f16w.cu): tm_lhs
// spans the fp16 split plane [m, k] (box {64, 16}, 128-byte swizzle), lhs_scale
// its (scale, mark) pairs, num_lhs_blocks = k / 128; tm_rhs the weight bytes
// (box {128, 128, 1}, 128-byte swizzle).  Launched as the programmatic
// dependent of the split pass.
cudaError_t launch_f16w(const ScaledLaunch& p, int weight_format, bool out_f32, int grid, cudaStream_t stream);

// Per-token-group e4m3 quantisation of bf16 activations (quantize.cu); group
// 64, 128 or 256, k % group == 0.
cudaError_t launch_quantize_e4m3(const void* x, int64_t m, int64_t k, int64_t group, void* q, float* scale,
                                 cudaStream_t stream);

// Per-shape kernel table (tuning.cu).  kernel: a GMM_KERNEL_* id; raster 0 =
// the default super-column width.
int32_t tuning_rows_log2(int64_t m, int32_t num_total_groups);
bool tuning_lookup(int32_t rows_log2, int64_t k, int64_t n, int32_t groups, int32_t transpose, int32_t out_dtype,
                   int32_t* kernel, int32_t* raster);
void tuning_store(int32_t rows_log2, int64_t k, int64_t n, int32_t groups, int32_t transpose, int32_t out_dtype,
                  int32_t kernel, int32_t raster);
bool tuning_valid(int32_t kernel, int32_t raster);

}  // namespace gmmk
