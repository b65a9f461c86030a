/*
 * libgmm: grouped matrix multiplication for GB300 (sm_103a).
 *
 * The rows of lhs [m, k] are split into consecutive groups by an int32
 * group_sizes vector; each group is multiplied by its own expert weight from
 * a 3-D rhs.  Definitions follow the page "tpu-inference 0.12.0.dev20251213
 * -> 0.13.2.dev20251230", file tpu_inference/kernels/megablox/gmm.py (the gmm
 * signature and docstring, _validate_args, _accum, make_group_metadata,
 * rhs_transform_indices and _zero_uninitialized_memory), and the page
 * "Megablox: transposed-RHS gmm_v2 kernel for the backward dlhs" (Context
 * section: dlhs = dout @ W^T read from the untransposed [groups, n, k]
 * weight; drhs per group).
 *
 * Conventions shared by every call:
 *  - Every tensor argument is a DEVICE pointer to a dense row-major array
 *    owned by the caller.  The library never allocates, frees or
 *    synchronises inside gmm() / tgmm(); work is enqueued on `stream` (a
 *    cudaStream_t; NULL is the legacy default stream) and runs
 *    asynchronously.
 *  - Host-checkable argument errors return a status below before anything is
 *    launched; outputs are then untouched.
 *  - Errors that only the device can see (bad group_sizes, an internal wait
 *    that timed out) set sticky flags in the workspace; the call still
 *    completes, treating negative sizes as 0 and cutting the groups at row m.
 *    Read them with gmm_read_device_errors().
 *  - The workspace is caller-owned device memory of gmm_workspace_bytes()
 *    bytes (at least GMM_WORKSPACE_MIN_BYTES), 256-byte aligned, zero-filled
 *    once before its first use.  Calls that share a workspace must be
 *    stream-ordered.
 *  - Requires the current device to be compute capability 10.3 (GB300).
 *  - The only environment variable read is GMM_LOG: when set (and not "0"),
 *    every forward and tgmm call writes one line to stderr with its sizes, dtypes
 *    and the kernel it chose.  Kernel choices are per-call arguments
 *    (gmm_options) or tiling-table entries, never environment variables.
 */
#ifndef LIBGMM_H_
#define LIBGMM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types (stored layout). */
enum {
  GMM_DTYPE_BF16 = 0, /* bfloat16 */
  GMM_DTYPE_F32 = 1,  /* IEEE binary32 */
  GMM_DTYPE_E4M3 = 2, /* float8_e4m3fn: bias 7, no infinities, 0x7F/0xFF NaN */
  GMM_DTYPE_E5M2 = 3, /* float8_e5m2: bias 15, IEEE infinities and NaN */
  GMM_DTYPE_INT8 = 4, /* two's complement int8 */
  /* 4-bit formats: two values per byte, the even-indexed value in the low nibble */
  GMM_DTYPE_INT4 = 5,  /* two's complement, -8 .. 7 */
  GMM_DTYPE_UINT4 = 6, /* 0 .. 15 */
  GMM_DTYPE_E2M1 = 7,  /* float4_e2m1fn: values 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives */
  /* block scales only (gmm_ex rhs_scale): byte e is 2^(e - 127), 0 is 2^-127, 255 is 0 */
  GMM_DTYPE_E8M0 = 8
};

/* Status codes returned by every entry point. */
enum {
  GMM_OK = 0,
  GMM_ERR_NULL = 1,         /* a required pointer is NULL */
  GMM_ERR_DTYPE = 2,        /* dtype combination not supported */
  GMM_ERR_SHAPE = 3,        /* inconsistent or unsupported sizes */
  GMM_ERR_ALIGN = 4,        /* a pointer is not 16-byte aligned or a row pitch is not a multiple of 16 bytes */
  GMM_ERR_GROUP_OFFSET = 5, /* group_offset outside [0, num_total_groups - num_local_groups] */
  GMM_ERR_WORKSPACE = 6,    /* workspace NULL, misaligned or smaller than GMM_WORKSPACE_MIN_BYTES */
  GMM_ERR_ARCH = 7,         /* current device is not compute capability 10.3 */
  GMM_ERR_CUDA = 8,         /* a CUDA runtime or driver call failed; see gmm_last_cuda_error() */
  GMM_ERR_IO = 9,           /* a tiling-table file could not be read, parsed or written */
  /* from gmm_get_device_error() only: what the device recorded */
  GMM_ERR_DEVICE_GROUP_SIZES = 10, /* some group_sizes[g] < 0, or sum(group_sizes) > m */
  GMM_ERR_TIMEOUT = 11             /* an internal pipeline wait gave up; that call's output is undefined */
};

/* Sticky device-side error flags kept in the workspace. */
#define GMM_DEVERR_NEGATIVE_GROUP_SIZE 0x1u /* some group_sizes[g] < 0 (counted as 0) */
#define GMM_DEVERR_GROUP_SIZES_EXCEED_M 0x2u /* sum(group_sizes) > m (groups cut at row m) */
#define GMM_DEVERR_TIMEOUT 0x4u              /* an internal pipeline wait gave up; output is undefined */
#define GMM_DEVERR_GROUP_OFFSET 0x8u         /* gmm_device_offset: offset out of range; nothing written */

/* Largest num_total_groups (gmm, tgmm_local) or num_groups (tgmm) accepted. */
#define GMM_MAX_GROUPS 1024

/* Smallest workspace a call accepts: the error flags alone. */
#define GMM_WORKSPACE_MIN_BYTES 256

/*
 * Size in bytes of a full workspace (a constant, 16 MiB + 256): the error
 * flags, then scratch for the 8- and 4-bit weight kernels.  With bf16
 * activations, a call of those kernels whose split activations fit the
 * caller's workspace first splits each activation row once there:
 *  - e4m3, e5m2, e2m1 and uint4 weights: 256 bytes of flags, then 4 m k bytes of e4m3
 *    terms rounded up to 256, then 8 m ceil(k / 256) bytes of step scales; the
 *    fp8 kernel reads the terms instead of splitting every row again for each
 *    128-wide weight tile, and the result is the same, bit for bit;
 *  - int8 and int4 weights, and MXFP8 and NVFP4 block-scaled weights
 *    (gmm_ex): 256 bytes of flags, then 2 m k bytes of fp16 values rounded up
 *    to 256, then 8 m k / 128 bytes of (scale, mark) pairs; the weights are
 *    then rewritten as fp16 and multiplied on the fp16 tensor cores.  Both
 *    ways give exact products and fp32 sums, but the sums may round
 *    differently from the in-kernel split's.  (The e4m3 and e2m1 sizes below
 *    cover this layout too.)
 * With a smaller workspace (at least GMM_WORKSPACE_MIN_BYTES) the fp8 kernel
 * splits inside (e4m3 terms, for every format).
 */
size_t gmm_workspace_bytes(void);

/*
 * The workspace size that lets a gmm() / gmm_ex() call of this shape run its
 * fastest way: GMM_WORKSPACE_MIN_BYTES, plus for bf16 activations (lhs_dtype
 * GMM_DTYPE_BF16) with an 8- or 4-bit rhs_dtype the split scratch described above
 * (e4m3, e5m2, e2m1, uint4: 4 m k bytes rounded up to 256, then 8 m ceil(k / 256)
 * bytes; int8, int4: 2 m k bytes rounded up to 256, then 8 m k / 128 bytes).
 * num_total_groups, num_local_groups and n do not change it today; they are taken
 * so that callers size workspaces by the problem.  0 for negative sizes.
 */
size_t gmm_workspace_bytes_for(int64_t m, int64_t k, int64_t n, int32_t num_total_groups, int32_t num_local_groups,
                               int lhs_dtype, int rhs_dtype);

/* bf16 forward kernels, as gmm_options and the tiling table name them. */
enum {
  GMM_KERNEL_AUTO = 0,      /* no choice / built-in rule */
  GMM_KERNEL_PAIR = 1,      /* SM-pair 256 x 256 row tiles */
  GMM_KERNEL_SWAP_PAIR = 2, /* SM-pair, 256 weight rows x up to 256 group rows */
  GMM_KERNEL_SWAP = 3,      /* one SM, 128 weight rows x up to 256 group rows */
  GMM_KERNEL_SINGLE = 4     /* one SM, 128 x 256 row tiles */
};

/* gmm_options.e4m3_kernel */
enum { GMM_E4M3_AUTO = 0, GMM_E4M3_TENSOR = 1, GMM_E4M3_DECODE = 2 };
/* gmm_options.act_split */
enum { GMM_SPLIT_AUTO = 0, GMM_SPLIT_PASS = 1, GMM_SPLIT_KERNEL = 2 };
/* gmm_options.tgmm_kernel */
enum { GMM_TGMM_AUTO = 0, GMM_TGMM_SINGLE = 1, GMM_TGMM_PAIR = 2 };

/*
 * Per-call choices for gmm_ex() and tgmm_ex(); NULL, or a zero-filled struct,
 * means every default.  Every field is checked: an unknown value is
 * GMM_ERR_SHAPE.  These replace no result: every choice computes the same
 * outputs within the bound (the kernels differ in speed).
 *   bf16_kernel   bf16 weights without scale: GMM_KERNEL_AUTO (the tiling table's
 *                 entry for the problem's class, else the built-in rule) or one of
 *                 the GMM_KERNEL_* kernels.
 *   e4m3_kernel   e4m3 weights with bf16 activations: GMM_E4M3_AUTO / _TENSOR (the
 *                 e4m3 tensor cores, the activations split exactly) or _DECODE (the
 *                 kernel that decodes the weights to bf16; f32 rhs_scale only).
 *   act_split     8- and 4-bit weights with bf16 activations: GMM_SPLIT_AUTO (split
 *                 each row once by a pass when the workspace holds it, else inside
 *                 the kernel), _PASS (the pass; GMM_ERR_WORKSPACE when the workspace
 *                 cannot hold it) or _KERNEL (inside the kernel).  With the pass,
 *                 int8 and int4 weights run on the fp16 tensor cores (an fp16
 *                 split); inside the kernel every format runs on the fp8 ones.
 *   tgmm_kernel   tgmm_ex(): GMM_TGMM_AUTO / _SINGLE (one SM per 128 x 256 output
 *                 tile) or _PAIR (SM pairs on 256 x 256 tiles).
 *   wait_limit_cycles  0: the default bound of every internal pipeline wait (about
 *                 4e9 clock cycles, ~2 s).  Otherwise the bound used by the bf16
 *                 gmm kernels GMM_KERNEL_SINGLE, _PAIR and _SWAP_PAIR and by the
 *                 tgmm pair kernel (GMM_TGMM_PAIR), for tests of the timeout path;
 *                 other kernels ignore it.
 *   test_drop_stage  0: none.  s > 0 (test of the timeout path): in the one-SM bf16
 *                 kernel, CTA 0 does not issue the copies of its s-th pipeline
 *                 stage; in the pair kernels above, the second CTA of the first
 *                 pair stops issuing copies before its s-th stage.  The wait for
 *                 that stage runs out: GMM_DEVERR_TIMEOUT is set, the call still
 *                 returns, every copy and MMA in flight is waited for and the
 *                 tensor memory freed; that call's output is undefined.  Other
 *                 kernels ignore it.
 */
typedef struct gmm_options {
  int32_t bf16_kernel;
  int32_t e4m3_kernel;
  int32_t act_split;
  int32_t tgmm_kernel;
  int64_t wait_limit_cycles;
  int32_t test_drop_stage;
  int32_t reserved;
} gmm_options;

/*
 * Forward grouped matmul (page "tpu-inference ...", gmm.py: gmm).
 *
 *   For every local group g in [group_offset, group_offset + num_local_groups)
 *   and every row r of that group (rows offs[g] <= r < offs[g+1], offs the
 *   exclusive prefix sum of group_sizes):
 *     out[r, c] = sum_b  s[g', b, c] * sum_{kk in block b} lhs[r, kk] * W(g', c, kk)
 *                 + bias[g', c]                                  (g' = g - group_offset)
 *   with fp32 accumulation and one rounding to out_dtype.  Every other row of
 *   out (rows of non-local groups, rows at or past sum(group_sizes)) is set to 0:
 *   out is fully overwritten.
 *
 *   lhs          [m, k], lhs_dtype must be GMM_DTYPE_BF16.
 *   rhs          transpose_rhs != 0: [num_local_groups, n, k] (the pages' layout,
 *                W(g, c, kk) = rhs[g, c, kk]); transpose_rhs == 0: [num_local_groups, k, n].
 *                rhs_dtype GMM_DTYPE_BF16, or (transpose_rhs != 0 only) one of the weight
 *                formats of common.py's supported list: E4M3, E5M2, INT8, INT4, UINT4, E2M1;
 *                a row of the 4-bit formats is k / 2 bytes.
 *   group_sizes  device int32 [num_total_groups], 1 <= num_total_groups <= GMM_MAX_GROUPS.
 *   group_offset first local group; 0 <= group_offset <= num_total_groups - num_local_groups.
 *   rhs_scale    NULL (s = 1, one block) or device f32 [num_local_groups, num_quant_blocks, 1, n];
 *                block b covers kk in [b*k/nb, (b+1)*k/nb); k % num_quant_blocks == 0.
 *                With rhs_scale given or a non-bf16 rhs, a block-scaled kernel runs: it needs
 *                transpose_rhs != 0 (else GMM_ERR_DTYPE), k % 128 == 0 and
 *                (k / num_quant_blocks) % 128 == 0 (else GMM_ERR_SHAPE).  These are built for
 *                decode-sized groups (a few rows each) and stream every weight tile once per
 *                chunk of rows of its group (16 rows; 32 for e4m3 activations in gmm_ex).
 *                8- and 4-bit weights run on the fp8 tensor cores: e4m3, e5m2 and e2m1 as
 *                stored, int8, int4 and uint4 rewritten exactly as e4m3 (int8 as 16 * high
 *                nibble + low nibble, two e4m3 terms).  Each bf16 lhs row is split per k step (256 wide;
 *                128 for int8) into e4m3 terms at two powers of two, which hold every value of
 *                the step exactly when its magnitudes fall within two ranges of 2^13 (the
 *                largest value's and the largest of what that leaves): so the products with
 *                the weights are exact and the tensor cores sum them in fp32, as the pages'
 *                dot_general does.  A row with a step that the two levels do not hold, or
 *                that holds an infinity or a NaN, is summed again by the same kernel from the
 *                stored bf16 values and weights (exact products, fp32 sums, IEEE infinities
 *                and NaNs); realistic activations almost never need it.  Infinite e5m2
 *                weights give +-inf or NaN in the columns they touch (the split's terms can
 *                be zero: inf * 0 is NaN).
 *                With a workspace that holds it the split of bf16 activations is made once
 *                per row (see gmm_workspace_bytes); gmm_ex() options choose the other ways
 *                (gmm_options: e4m3_kernel, act_split).
 *                Without scale, bf16 weights run on one of four kernels chosen from the average
 *                group size m / num_total_groups: SM-pair 256x256 row tiles (>= 1024 rows),
 *                SM-pair tiles of 256 weight rows x up to 256 group rows rounded to 32 (>= 16),
 *                or single-SM tiles of 128 weight rows x group rows rounded to 16 (fewer).
 *                A tiling-table entry for the problem's class (gmm_tune, gmm_tuning_set)
 *                replaces that rule, and gmm_ex()'s options.bf16_kernel both.  All give
 *                results within the same bound; they may differ in the last bits.
 *   rhs_bias     NULL or device [num_local_groups, 1, n] of bias_dtype (BF16 or F32).
 *   out          [m, n] of out_dtype (BF16 or F32).
 *   Sizes: m >= 0, k >= 8, n >= 8, k % 8 == 0, n % 8 == 0 (16-byte rows); lhs, rhs,
 *   out and bias 16-byte aligned (E2M1 rhs 32-byte aligned).  Row counts and offsets must fit
 *   in int32.
 *   Returns GMM_OK or an error status above.
 */
int gmm(const void* lhs, int lhs_dtype, int64_t m, int64_t k, const void* rhs, int rhs_dtype,
        int32_t num_local_groups, int64_t n, int transpose_rhs, const int32_t* group_sizes,
        int32_t num_total_groups, int32_t group_offset, const float* rhs_scale, int32_t num_quant_blocks,
        const void* rhs_bias, int bias_dtype, void* out, int out_dtype, void* workspace,
        size_t workspace_bytes, void* stream);

/*
 * gmm_into: gmm() writing into an output the caller has already filled (page
 * "tpu-inference ...", gmm.py: the existing_out argument, aliased to the
 * output, whose tiles are first seeded from existing_out; the zeroing pass
 * _zero_uninitialized_memory runs only when no existing_out is given).
 *
 *   Rows of the local groups are computed exactly as gmm() computes them (same
 *   kernels, same rounding).  Every other row of out (rows of non-local groups,
 *   rows at or past sum(group_sizes)) is neither read nor written: it keeps what
 *   the caller put there.  The pages' existing_out has the output's dtype, so
 *   here it is simply `out`, of out_dtype.
 *
 *   Arguments, layouts, alignment and errors are those of gmm().  A typical use
 *   is expert parallelism without a combine: shards whose expert slices are
 *   disjoint call gmm_into on one shared [m, n] buffer, one after another or on
 *   streams ordered so that no two run at once on overlapping rows.
 */
int gmm_into(const void* lhs, int lhs_dtype, int64_t m, int64_t k, const void* rhs, int rhs_dtype,
             int32_t num_local_groups, int64_t n, int transpose_rhs, const int32_t* group_sizes,
             int32_t num_total_groups, int32_t group_offset, const float* rhs_scale, int32_t num_quant_blocks,
             const void* rhs_bias, int bias_dtype, void* out, int out_dtype, void* workspace,
             size_t workspace_bytes, void* stream);

/*
 * gmm_device_offset: gmm() or gmm_into() with group_offset read from device
 * memory (page "tpu-inference ...", gmm.py: group_offset is a ()-shaped int32
 * jnp array, a device value, turned into the kernels' scalar prefetch).
 *
 *   group_offset      device int32 [1], 4-byte aligned; read by the kernel when it
 *                     runs, so a captured CUDA graph can be replayed with another
 *                     offset written into it, and an offset computed on the device
 *                     needs no copy to the host.
 *   keep_other_rows   0: rows outside the local groups are set to 0 (gmm);
 *                     1: they keep the caller's contents (gmm_into).
 *   Everything else as gmm().  The host cannot check the offset: a value outside
 *   [0, num_total_groups - num_local_groups] sets GMM_DEVERR_GROUP_OFFSET in the
 *   workspace and the call writes nothing.  GMM_ERR_NULL if group_offset is NULL,
 *   GMM_ERR_ALIGN if it is not 4-byte aligned.
 */
int gmm_device_offset(const void* lhs, int lhs_dtype, int64_t m, int64_t k, const void* rhs, int rhs_dtype,
                      int32_t num_local_groups, int64_t n, int transpose_rhs, const int32_t* group_sizes,
                      int32_t num_total_groups, const int32_t* group_offset, const float* rhs_scale,
                      int32_t num_quant_blocks, const void* rhs_bias, int bias_dtype, void* out, int out_dtype,
                      int keep_other_rows, void* workspace, size_t workspace_bytes, void* stream);

/*
 * gmm_ex: gmm(), gmm_into() and gmm_device_offset() in one call, plus the W8A8
 * form (page "gemm_quant.rs", fp8_gemm_t_blockscaled: C = bf16(sum over 128-wide
 * K-groups g of the e4m3 MMA over g times a_scale[row, g] times the weight's
 * block scale)) and E8M0 weight scales (page "gemm_quant.rs",
 * widen_block_scale_f32).
 *
 *   out[r, c] = sum_b s[g', b, c] * sum_{kk in block b} a(r, kk) * W(g', c, kk) + bias[g', c]
 *   with a(r, kk) = lhs[r, kk] for bf16 lhs, and lhs_scale[r, j] * lhs[r, kk] (j the lhs
 *   block holding kk; lhs_scale NULL counts as 1) for e4m3 lhs.
 *
 *   lhs_dtype        GMM_DTYPE_BF16, or GMM_DTYPE_E4M3 with rhs_dtype one of the 8- and 4-bit
 *                    weight formats (bf16 weights: GMM_ERR_DTYPE).
 *   lhs_scale        e4m3 lhs only (else GMM_ERR_DTYPE): NULL or device f32 [m, num_lhs_blocks],
 *                    4-byte aligned; lhs block j covers kk in [j*k/nlb, (j+1)*k/nlb) and
 *                    (k / num_lhs_blocks) % 128 == 0 (else GMM_ERR_SHAPE).  The pages' layout is
 *                    num_lhs_blocks = k / 128 (gmm_quantize_e4m3 with group 128).
 *   group_offset_dev NULL: group_offset is used as in gmm(); else read from device memory as in
 *                    gmm_device_offset() (group_offset ignored).
 *   rhs_scale        NULL or device [num_local_groups, num_quant_blocks, 1, n] of
 *                    rhs_scale_dtype: GMM_DTYPE_F32, or GMM_DTYPE_E8M0 (one byte each; 8- and
 *                    4-bit weights only, else GMM_ERR_DTYPE); 16-byte aligned.  A weight scale of
 *                    the pages' [n / 128, k / 128] layout for one group is s[b, 0, c] =
 *                    b_scale[c / 128, b].
 *   rhs_block_scale  NULL, or microscaling block scales of the weights, device
 *                    [num_local_groups, n, k / block_size] of rhs_block_scale_dtype: every weight
 *                    W(g, c, kk) counts as rhs_block_scale[g, c, kk / block_size] * W(g, c, kk).
 *                    Supported (else GMM_ERR_DTYPE / GMM_ERR_SHAPE), with bf16 lhs and an F32
 *                    rhs_scale (or none) on top:
 *                      MXFP8: E4M3 rhs, GMM_DTYPE_E8M0 scales, block_size 32;
 *                      NVFP4: E2M1 rhs, GMM_DTYPE_E4M3 scales, block_size 16 (the second-level
 *                      fp32 scale of NVFP4 is rhs_scale with num_quant_blocks = 1).
 *                    MXFP8 runs on the fp16-weight kernel (an fp16 split of the bf16 lhs in the
 *                    workspace, like int8) when the scales are 4-byte aligned, the workspace
 *                    holds the split and options->e4m3_kernel is not GMM_E4M3_DECODE: the e4m3
 *                    codes are exact fp16 weights, each 32-k block sums into its own fp32
 *                    accumulator, and the block's sum is multiplied by its power of two (exact
 *                    while it stays in fp32's range).  Otherwise it runs on the decoding kernel:
 *                    the decoders multiply each decoded bf16 weight by its block scale, exactly
 *                    while the product stays in bf16's normal range.  NVFP4 runs on the
 *                    fp16-weight kernel (an fp16 split of the bf16 lhs in the workspace, like
 *                    int4) when k % 256 == 0, the scales are 16-byte aligned and the workspace
 *                    holds the split: each e2m1 code times its e4m3 scale is an exact fp16
 *                    weight; otherwise on the decoding kernel (an e2m1 value times an e4m3 value
 *                    always fits bf16).  No other alignment requirement for the scales.
 *   keep_other_rows  0: rows outside the local groups are set to 0 (gmm); 1: they keep the
 *                    caller's contents (gmm_into).
 *   Everything else as gmm().  e4m3 activations are taken as they are: each 128-wide k
 *   sub-tile is one e4m3 MMA per token row (exact products, fp32 sums), folded in fp32 as
 *   acc += s[g', b, c] * lhs_scale[r, j] * D.  options->e4m3_kernel = GMM_E4M3_DECODE with
 *   e4m3 lhs or E8M0 scales: GMM_ERR_DTYPE.
 *   options          NULL (every default) or the per-call choices of gmm_options.
 */
int gmm_ex(const void* lhs, int lhs_dtype, const float* lhs_scale, int32_t num_lhs_blocks, int64_t m, int64_t k,
           const void* rhs, int rhs_dtype, int32_t num_local_groups, int64_t n, int transpose_rhs,
           const int32_t* group_sizes, int32_t num_total_groups, int32_t group_offset,
           const int32_t* group_offset_dev, const void* rhs_scale, int rhs_scale_dtype, int32_t num_quant_blocks,
           const void* rhs_block_scale, int rhs_block_scale_dtype, int32_t block_size, const void* rhs_bias,
           int bias_dtype, void* out, int out_dtype, int keep_other_rows, const gmm_options* options, void* workspace,
           size_t workspace_bytes, void* stream);

/*
 * Backward weight gradient (drhs) per group (page "Megablox: transposed-RHS
 * gmm_v2 kernel ...", Context section; gmm.py make_group_metadata docstring on
 * visiting empty groups so that their output is zeroed).
 *
 *   out[g, kk, c] = sum_{r in group g} lhs[r, kk] * dout[r, c]   for every g,
 *   fp32 accumulation, one rounding to out_dtype; empty groups give zero blocks.
 *
 *   lhs    [m, k] BF16;  dout [m, n] BF16;  out [num_groups, k, n] F32 or BF16.
 *   group_sizes device int32 [num_groups], 1 <= num_groups <= GMM_MAX_GROUPS.
 *   Sizes: m >= 0, k % 8 == 0, n % 8 == 0, k, n >= 8; pointers 16-byte aligned.
 *   Two kernels give the same results within the bound: one SM per 128 x 256
 *   output tile (default) and SM pairs on 256 x 256 tiles (tgmm_ex() with
 *   options.tgmm_kernel chooses).
 *   For an NT weight [G, n, k] the matching gradient is tgmm(dout, x): pass the
 *   forward output gradient as `lhs` and the forward input as `dout`.
 */
int tgmm(const void* lhs, int lhs_dtype, const void* dout, int dout_dtype, int64_t m, int64_t k, int64_t n,
         const int32_t* group_sizes, int32_t num_groups, void* out, int out_dtype, void* workspace,
         size_t workspace_bytes, void* stream);

/*
 * tgmm_local: tgmm() over one contiguous slice of the groups, the drhs of an
 * expert shard (page "tpu-inference ...", gmm.py make_group_metadata:
 * start_group and num_nonzero_groups select the groups a shard computes, and
 * visit_empty_groups keeps a tile for every empty group so that its output is
 * zeroed).
 *
 *   out[l, kk, c] = sum_{r in group group_offset + l} lhs[r, kk] * dout[r, c]
 *   for 0 <= l < num_local_groups; group rows come from the prefix sum of all
 *   num_total_groups sizes, so rows of the groups outside the slice are not read.
 *
 *   group_sizes  device int32 [num_total_groups], 1 <= num_total_groups <= GMM_MAX_GROUPS.
 *   group_offset first group of the slice; 1 <= num_local_groups and
 *                0 <= group_offset <= num_total_groups - num_local_groups
 *                (else GMM_ERR_SHAPE / GMM_ERR_GROUP_OFFSET).
 *   out          [num_local_groups, k, n] F32 or BF16.
 *   Everything else as tgmm(), which is tgmm_local(..., num_groups, 0, num_groups, ...).
 */
int tgmm_local(const void* lhs, int lhs_dtype, const void* dout, int dout_dtype, int64_t m, int64_t k,
               int64_t n, const int32_t* group_sizes, int32_t num_total_groups, int32_t group_offset,
               int32_t num_local_groups, void* out, int out_dtype, void* workspace, size_t workspace_bytes,
               void* stream);

/*
 * tgmm_ex: tgmm_local() with per-call options (NULL: every default); only
 * options->tgmm_kernel applies.
 */
int tgmm_ex(const void* lhs, int lhs_dtype, const void* dout, int dout_dtype, int64_t m, int64_t k, int64_t n,
            const int32_t* group_sizes, int32_t num_total_groups, int32_t group_offset, int32_t num_local_groups,
            void* out, int out_dtype, const gmm_options* options, void* workspace, size_t workspace_bytes,
            void* stream);

/* Size of the device scratch array compiled into the library for gmm_noalloc(). */
#define GMM_NOALLOC_SCRATCH_BYTES 256

/*
 * gmm_noalloc: gmm() without a caller-supplied workspace.  The pages have no
 * counterpart to this call.
 *
 * For callers that cannot allocate device memory: code whose device memory is
 * owned by another component's allocator with no way to ask it for a buffer,
 * or code on a path where cudaMalloc is not allowed (it may synchronise the
 * device and its latency is unbounded).  Instead of a workspace it uses a
 * GMM_NOALLOC_SCRATCH_BYTES-byte __device__ array compiled into the library,
 * which every GPU that loads the library holds until the process exits.  It
 * calls no cudaMalloc, cudaFree or allocating library routine.
 *
 *  - Arguments, layouts, results and host-side errors are those of gmm() (the
 *    same kernels run); GMM_ERR_WORKSPACE if the library's scratch need ever
 *    exceeded the array (it is one word of error flags, independent of the
 *    problem size, so every size gmm() accepts fits).
 *  - Every call looks up the array's device address on the current device
 *    (cudaGetSymbolAddress; after cudaDeviceReset it finds the new copy).  The
 *    first call on a device also loads the library's device code there: make
 *    it before any stream capture.
 *  - It takes every default of gmm_options: with bf16 activations and 8- or
 *    4-bit weights the kernel splits the rows itself (the array has no room
 *    for the split pass).
 *  - Every call on a device shares the array, and the array keeps the last
 *    call's contents; each call first clears the error-flag word (an
 *    asynchronous memset on `stream`).  Calls that overlap on the GPU (on
 *    different streams) race on it.  The device error flags of this variant
 *    cannot be read back; callers that need them use gmm() with a workspace.
 */
int gmm_noalloc(const void* lhs, int lhs_dtype, int64_t m, int64_t k, const void* rhs, int rhs_dtype,
                int32_t num_local_groups, int64_t n, int transpose_rhs, const int32_t* group_sizes,
                int32_t num_total_groups, int32_t group_offset, const float* rhs_scale, int32_t num_quant_blocks,
                const void* rhs_bias, int bias_dtype, void* out, int out_dtype, void* stream);

/*
 * Per-token-group e4m3 quantisation of bf16 activations, the activation side of
 * the W8A8 path (page "gemm_quant.rs", per_token_group_quant_fp8: A_fp8 [M, K]
 * e4m3 and a_scale [M, K/128] f32).  The page prints no formula; this library's
 * reading, for each row r and group j of `group` consecutive k:
 *   scale[r, j] = max |x| / 448 (fp32 IEEE division; 1 when the maximum is 0;
 *                 NaN when a value is NaN),
 *   q[r, kk]    = e4m3fn nearest to x / scale[r, j] (the quotient an fp32 IEEE
 *                 division), ties to even, saturating at +-448.
 *   x      device bf16 [m, k] (x_dtype GMM_DTYPE_BF16), 16-byte aligned
 *   q      device e4m3fn [m, k], 16-byte aligned
 *   scale  device f32 [m, k / group], 4-byte aligned
 *   group  64, 128 or 256; k % group == 0 (else GMM_ERR_SHAPE)
 * Asynchronous on `stream`.
 */
int gmm_quantize_e4m3(const void* x, int x_dtype, int64_t m, int64_t k, int64_t group, void* q, float* scale,
                      void* stream);

/* ------------------------------------------------------------------ tiling table
 * The pages let `tiling` be a callable that looks the problem dimensions up in a
 * LUT of tuned tile sizes (page "tpu-inference ...", gmm.py: gmm).  Here each
 * kernel's tiles are fixed and the per-problem choice is which bf16 kernel runs
 * (and, for the row-tile kernels, the width of the L2 raster's super-columns).
 * A process-wide table maps a problem class to that choice:
 *   rows_log2 = floor(log2(m / num_total_groups)) (average rows per group),
 *   k, n, num_total_groups, transpose_rhs (0/1), out_dtype.
 * gmm(), gmm_into() and gmm_device_offset() with bf16 weights and no scale use
 * the table's entry for their class when there is one (gmm_ex()'s options.bf16_kernel
 * still overrides it), else the built-in rule.  The table is
 * guarded by a mutex; calls on any thread see every completed update.
 */
/* (The kernel ids are the GMM_KERNEL_* values above.) */

/* Sets the entry of one problem class.  raster (used by PAIR and SINGLE; the
 * order in which their output tiles are visited): 0, the default; 1..64 n tiles
 * per super-column, m tiles of all groups outer and the super-column's n tiles
 * inner; or -64..-1: group by group, in blocks of up to -raster m tiles, each
 * block meeting the n tiles in turn with its m tiles inner.  GMM_ERR_SHAPE for
 * invalid values.  The default is -16 for PAIR and -32 for SINGLE (blocks of
 * 4096 rows). */
int gmm_tuning_set(int32_t rows_log2, int64_t k, int64_t n, int32_t num_total_groups, int transpose_rhs,
                   int out_dtype, int kernel, int raster);

/* *kernel = the entry's kernel (GMM_KERNEL_AUTO if the class has none), *raster its raster. */
int gmm_tuning_get(int32_t rows_log2, int64_t k, int64_t n, int32_t num_total_groups, int transpose_rhs,
                   int out_dtype, int* kernel, int* raster);

/* Empties the table. */
int gmm_tuning_clear(void);

/* Writes the table to `path` as text: a first line "# libgmm tiling table 1", then
 * one line per entry "rows_log2 k n num_total_groups transpose_rhs out_dtype kernel
 * raster".  gmm_tuning_load() reads such a file and adds its entries (replacing
 * entries of the same class); on any malformed line it adds nothing and returns
 * GMM_ERR_IO, as it does when the file cannot be opened. */
int gmm_tuning_save(const char* path);
int gmm_tuning_load(const char* path);

/*
 * Times every bf16 kernel choice (PAIR with rasters -16, -4 and 8, SWAP_PAIR, SWAP,
 * SINGLE with raster -32) on this problem, with the caller's buffers (`out` is
 * written), `iterations` launches each after one warm-up launch, using CUDA events
 * on `stream`, which it synchronises.  Records the fastest in the table and returns
 * it in *kernel, *raster and its mean time in *ms.  Arguments as gmm(); bf16
 * weights without scale only (else GMM_ERR_DTYPE); iterations in 1..1000.
 */
int gmm_tune(const void* lhs, int lhs_dtype, int64_t m, int64_t k, const void* rhs, int rhs_dtype,
             int32_t num_local_groups, int64_t n, int transpose_rhs, const int32_t* group_sizes,
             int32_t num_total_groups, int32_t group_offset, const void* rhs_bias, int bias_dtype, void* out,
             int out_dtype, void* workspace, size_t workspace_bytes, void* stream, int iterations, int* kernel,
             int* raster, float* ms);

/*
 * Synchronises `stream`, then reads and clears the sticky device error flags
 * (GMM_DEVERR_*) of `workspace` into *flags.  Returns GMM_OK or GMM_ERR_CUDA.
 */
int gmm_read_device_errors(void* workspace, void* stream, uint32_t* flags);

/*
 * The device's report as one status: synchronises `stream`, reads and clears the
 * sticky flags of `workspace` (as gmm_read_device_errors) and returns GMM_OK when
 * none is set, else GMM_ERR_TIMEOUT, GMM_ERR_DEVICE_GROUP_SIZES or
 * GMM_ERR_GROUP_OFFSET (in that order of precedence), or GMM_ERR_NULL /
 * GMM_ERR_CUDA when it cannot read them.
 */
int gmm_get_device_error(void* workspace, void* stream);

/* Static English text for a status code. */
const char* gmm_status_string(int status);

/* The cudaError_t behind the last GMM_ERR_CUDA returned on this thread (0 if none). */
int gmm_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* LIBGMM_H_ */
