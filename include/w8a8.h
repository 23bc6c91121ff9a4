/*
 * w8a8.h — C ABI of the GB300 (sm_103a) W8A8 group-scaled quantized linear layer.
 *
 * The operation ("Deploying Hunyuan 770B in INT8 on domestic accelerators
 * (FlagOS Hy4 preview 5)", §3.1, quantization granularity):
 *   - activations are quantized per token, dynamically, at every call:
 *       s_m = amax_k |A[m,k]| / 127,  qa[m,k] = round(A[m,k] / s_m)
 *     (round = nearest, ties to even; codes clamped to [-127, 127]);
 *   - weights are INT8 with one FP32 scale per group of 128 consecutive K
 *     elements of an output row n: sw[n, g], g = k / 128;
 *   - each group is multiplied INT8 x INT8 and accumulated exactly in integers,
 *       P[m,n,g] = sum_{k in group g} qa[m,k] * qw[n,k]
 *     and the FP32 scales are applied only at the end:
 *       Y[m,n] = sa[m] * sum_g sw[n,g] * P[m,n,g].
 * MoE expert layers (same page §1.3 and §4.4: each token goes to the experts
 * its router picked) run the same computation per expert over the rows that
 * were routed to it.
 *
 * Conventions for every call:
 *   - All data pointers are DEVICE pointers owned by the caller. The library
 *     never allocates device memory inside these calls.
 *   - Calls are asynchronous on `stream` (NULL = legacy default stream). They
 *     never synchronise the host and never read device data on the host, so
 *     they can be captured in a CUDA graph. The status returned covers only
 *     what the host can check (arguments, device capability, launch errors);
 *     a device-side fault shows up later through the CUDA runtime and a
 *     device-side wait that timed out through w8a8_device_error().
 *   - Matrices are row-major with unit stride in their last dimension.
 *     Pointers to int8/bf16/fp16 matrices read with TMA must be 16-byte
 *     aligned; float vectors 4-byte aligned.
 *   - Sizes are int64_t; the product of a matrix's dimensions must stay below
 *     2^31 elements per operand (checked).
 *   - Requires a device of compute capability 10.3 (GB300); any other device
 *     returns W8A8_ERR_UNSUPPORTED.
 */
#ifndef W8A8_H
#define W8A8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st *w8a8_stream_t;

typedef enum {
    W8A8_OK = 0,
    W8A8_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misalignment, K % 128 != 0 ... */
    W8A8_ERR_UNSUPPORTED = 2,   /* device is not compute capability 10.3 */
    W8A8_ERR_CUDA = 3,          /* a CUDA runtime call or kernel launch failed */
    W8A8_ERR_WORKSPACE = 4,     /* workspace pointer missing or smaller than required */
    W8A8_ERR_DEVICE_TIMEOUT = 5 /* reported by w8a8_device_error(): a device wait gave up */
} w8a8_status;

typedef enum { W8A8_BF16 = 0, W8A8_FP32 = 1 } w8a8_dtype;

/* How a quantization scale is chosen from the group's largest magnitude amax:
 * amax / 127 (IEEE FP32 division), or the smallest power of two >= amax / 127
 * (exponent clamped to [-127, 127]; 2^-127 for an all-zero group), i.e. a
 * scale that the 8-bit exponent-only UE8M0 format holds exactly. */
typedef enum { W8A8_SCALE_AMAX = 0, W8A8_SCALE_POW2 = 1 } w8a8_scale_mode;

#define W8A8_GROUP 128

/*
 * Per-token dynamic activation quantization (Hunyuan-770B page §3.1,
 * "activations quantized per token, dynamically"; "round(x / scale)").
 *   a_bf16 [M, lda] BF16 (only the first K columns are read);
 *   qa     [M, ldq] int8 output, qa[m,k] = clamp(rne(a[m,k] / sa[m]), -127, 127);
 *   sa     [M] float output, sa[m] = amax_k |a[m,k]| / 127 (IEEE FP32 division).
 * A row whose amax is 0 gets sa = 0 and all-zero codes. Inputs must be finite.
 * K >= 1, lda >= K, ldq >= K. M == 0 is a no-op. Results are bit-identical to
 * the FP32 definition above (no fast-math, no reciprocal multiply).
 */
w8a8_status w8a8_quant_act(const void *a_bf16, int64_t M, int64_t K, int64_t lda,
                           int8_t *qa, int64_t ldq, float *sa, w8a8_stream_t stream);

/*
 * Per-row, per-128-K-group weight quantization (Hunyuan-770B page §3.1,
 * "weights in groups of 128 elements, one scale per group"): offline input
 * preparation for the GEMMs below.
 *   w  [N, K] float; qw [N, K] int8; sw [N, K/128] float.
 *   sw[n,g] = amax over the group / 127; qw = clamp(rne(w / sw), -127, 127).
 * K must be a positive multiple of 128. N == 0 is a no-op.
 */
w8a8_status w8a8_quant_weight(const float *w, int64_t N, int64_t K, int8_t *qw, float *sw,
                              w8a8_stream_t stream);

/*
 * Bytes of device workspace w8a8_gemm asks for: an fp16 copy of the M x K
 * int8 activation codes (the tensor-core operand), rounded up to 256 bytes,
 * then, when 5 <= M <= 64, a split area of 1280 + 160 * 2 * M * 128 * 4
 * bytes (rounded up to 256) in which up to 160 CTAs exchange FP32 partial
 * sums of weight tiles whose K range they share. 0 when M == 0.
 * The split area is optional: a workspace that holds only the staging copy
 * (M * K * 2 bytes rounded up to 256) is accepted, and the GEMM then never
 * splits a tile's K range across CTAs (slower when the weight tiles do not
 * divide evenly among the SMs; results agree within the stated bound).
 * Calls with M <= 4 run on the CUDA cores and do not use the staging copy.
 */
size_t w8a8_gemm_workspace_size(int64_t M, int64_t N, int64_t K);

/*
 * Dense W8A8 GEMM with per-group weight scales (Hunyuan-770B page §3.1:
 * INT8 multiply-accumulate into INT32 per group, FP32 scales "multiplied back
 * only at the end").
 *   qa [M, K] int8, sa [M] float   (from w8a8_quant_act, ldq == K)
 *   qw [N, K] int8, sw [N, K/128] float
 *   y  [M, N] BF16 (round to nearest even) or FP32, per y_dtype.
 *   debug_partials: NULL, or int32 [M, N, K/128] receiving every exact group
 *                   partial P[m,n,g] (debug/parity use; slow).
 *   workspace: device buffer, 256-byte aligned, of w8a8_gemm_workspace_size(M, N, K)
 *              bytes (at least the staging part, see above); its contents
 *              are scratch.
 * K must be a positive multiple of 128; N >= 1. M == 0 is a no-op.
 * The group sums are exact integers; Y is accumulated in FP32 over the
 * groups in K order, acc = fma(P_g, sw[n,g], acc), and Y = sa[m] * acc. When
 * a tile's K range is split into n pieces (only for 5 <= M <= 64 with the
 * split area; n <= ceil(G/2), otherwise n = 1), each piece accumulates its
 * groups from zero and the pieces are added in K order, so
 *   |Y - Y*| <= (G + n + 1) * 2^-24 * sum_g |sa*sw*P_g|  for the exact Y*,
 * and the result does not depend on the order in which CTAs finish.
 */
w8a8_status w8a8_gemm(const int8_t *qa, const float *sa, const int8_t *qw, const float *sw,
                      void *y, w8a8_dtype y_dtype, int64_t M, int64_t N, int64_t K,
                      int32_t *debug_partials, void *workspace, size_t workspace_bytes,
                      w8a8_stream_t stream);

/*
 * Bytes of device workspace w8a8_grouped_gemm needs for R routed rows: an
 * fp16 copy of the R x K activation codes, rounded up to 256 bytes.
 */
size_t w8a8_grouped_gemm_workspace_size(int64_t R, int64_t E, int64_t N, int64_t K);

/*
 * MoE expert-grouped W8A8 GEMM (Hunyuan-770B page §1.3/§4.4: tokens are
 * processed by the experts the router chose; one routed row per
 * (token, expert) pair, rows sorted by expert).
 *   qa      [R, K] int8, sa [R] float: routed rows, sorted by expert
 *   offsets [E+1] int32 DEVICE array: rows of expert e are [offsets[e], offsets[e+1]).
 *           Precondition: 0 = offsets[0] <= ... <= offsets[E] <= R. Not read on the
 *           host; the kernel clamps every offset into [0, R] so a violation cannot
 *           make it access memory out of bounds. Empty segments produce no work.
 *   qw      [E, N, K] int8, sw [E, N, K/128] float: per-expert weights and scales
 *   y       [R, N] BF16 or FP32. Only rows covered by a segment are written.
 *   debug_partials: NULL or int32 [R, N, K/128].
 *   workspace: >= w8a8_grouped_gemm_workspace_size(R, E, N, K) bytes, 256-aligned.
 * Y is accumulated as in w8a8_gemm (no K split): the error bound there with n = 1.
 * E >= 1, N >= 1, K a positive multiple of 128. R == 0 is a no-op.
 */
w8a8_status w8a8_grouped_gemm(const int8_t *qa, const float *sa, const int32_t *offsets,
                              const int8_t *qw, const float *sw, void *y, w8a8_dtype y_dtype,
                              int64_t R, int64_t E, int64_t N, int64_t K,
                              int32_t *debug_partials, void *workspace, size_t workspace_bytes,
                              w8a8_stream_t stream);

/*
 * Bytes of device workspace w8a8_linear asks for: the M x K activation codes
 * (M * K * 2 bytes, rounded up to 256), the M token scales (M * 4 bytes,
 * rounded up to 256), then for 5 <= M <= 64 the optional split area of
 * w8a8_gemm_workspace_size. 0 when M == 0. A workspace without the split
 * area is accepted (tiles then are never split across CTAs).
 */
size_t w8a8_linear_workspace_size(int64_t M, int64_t N, int64_t K);

/*
 * The quantized linear layer in one call: per-token activation quantization
 * (w8a8_quant_act, Hunyuan-770B page §3.1: dynamic per-token INT8) followed by
 * the group-scaled GEMM (w8a8_gemm). For M > 4 the quantizer writes the codes
 * (fp16, the tensor-core operand) and token scales into the workspace, so no
 * staging copy is made in between; for M <= 4 the CUDA-core GEMM quantizes
 * its token rows itself when lda is a multiple of 8 and a_bf16 is 16-byte
 * aligned (one kernel), else the quantizer writes int8 codes first.
 *   a_bf16 [M, K] BF16, row stride lda >= K elements (2-byte aligned)
 *   qw [N, K] int8, sw [N, K/128] float   (from w8a8_quant_weight)
 *   y  [M, N] BF16 (round to nearest even) or FP32, per y_dtype.
 *   workspace: device buffer, 256-byte aligned, of w8a8_linear_workspace_size(M,
 *              N, K) bytes (at least the codes and scales, see above); scratch.
 * The result is identical to w8a8_quant_act followed by w8a8_gemm with the
 * same workspace split behaviour (same codes, scales and kernels), with the
 * error bound stated there. K a positive multiple of 128; N >= 1; M == 0 is
 * a no-op. Returns W8A8_ERR_WORKSPACE when the workspace is missing, not
 * 256-byte aligned or smaller than the codes and scales.
 */
w8a8_status w8a8_linear(const void *a_bf16, int64_t lda, const int8_t *qw, const float *sw,
                        void *y, w8a8_dtype y_dtype, int64_t M, int64_t N, int64_t K,
                        void *workspace, size_t workspace_bytes, w8a8_stream_t stream);

/*
 * Bytes of device workspace w8a8_grouped_linear needs for R routed rows: the
 * R x K codes (R * K * 2 bytes) and R token scales, each rounded up to 256.
 */
size_t w8a8_grouped_linear_workspace_size(int64_t R, int64_t E, int64_t N, int64_t K);

/*
 * w8a8_grouped_gemm with the per-token quantization of its routed rows in the
 * same call (as w8a8_linear): a_bf16 [R, K] BF16 rows sorted by expert (row
 * stride lda), offsets [E+1] int32 on the device, qw [E, N, K], sw [E, N, K/128],
 * y [R, N]. Identical result to w8a8_quant_act + w8a8_grouped_gemm.
 */
w8a8_status w8a8_grouped_linear(const void *a_bf16, int64_t lda, const int32_t *offsets,
                                const int8_t *qw, const float *sw, void *y, w8a8_dtype y_dtype,
                                int64_t R, int64_t E, int64_t N, int64_t K, void *workspace,
                                size_t workspace_bytes, w8a8_stream_t stream);

/* ------------------------------------------------------------------------
 * Scale formats of the DeepSeek-V4 checkpoints ("Running DeepSeek-V4-Flash-
 * Vision on 4xA800", §一: weights in [128, 128] blocks, power-of-two UE8M0
 * scales), applied to the INT8 codes of this library.
 * ------------------------------------------------------------------------ */

/*
 * w8a8_quant_act with a choice of scale: mode W8A8_SCALE_AMAX is
 * w8a8_quant_act; W8A8_SCALE_POW2 sets sa[m] to the power of two above
 * (see w8a8_scale_mode), and the codes are then round-half-even(a / sa[m])
 * with an exact division (|code| <= 127, the largest |code| of a non-zero
 * row at least 64).
 */
w8a8_status w8a8_quant_act_ex(const void *a_bf16, int64_t M, int64_t K, int64_t lda,
                              int8_t *qa, int64_t ldq, float *sa, w8a8_scale_mode mode,
                              w8a8_stream_t stream);

/*
 * Weight quantization over blocks of block_rows rows x 128 K: block_rows 1 is
 * w8a8_quant_weight's per-row groups, 128 the [128, 128] blocks (one scale
 * per block; a ragged last block of rows has its own scale). sw has
 * ceil(N / block_rows) rows of K / 128 scales; mode as above.
 */
w8a8_status w8a8_quant_weight_ex(const float *w, int64_t N, int64_t K, int32_t block_rows,
                                 w8a8_scale_mode mode, int8_t *qw, float *sw,
                                 w8a8_stream_t stream);

/*
 * w8a8_gemm / w8a8_grouped_gemm with weight scales per [sw_block_rows x 128]
 * block: sw[n / sw_block_rows, g] scales P[m, n, g] (sw_block_rows 1 or 128;
 * sw [E * ceil(N / sw_block_rows), K / 128] for grouped calls). Everything
 * else, including the accuracy bound, as w8a8_gemm / w8a8_grouped_gemm.
 */
w8a8_status w8a8_gemm_ex(const int8_t *qa, const float *sa, const int8_t *qw, const float *sw,
                         int32_t sw_block_rows, void *y, w8a8_dtype y_dtype, int64_t M, int64_t N,
                         int64_t K, int32_t *debug_partials, void *workspace,
                         size_t workspace_bytes, w8a8_stream_t stream);
w8a8_status w8a8_grouped_gemm_ex(const int8_t *qa, const float *sa, const int32_t *offsets,
                                 const int8_t *qw, const float *sw, int32_t sw_block_rows,
                                 void *y, w8a8_dtype y_dtype, int64_t R, int64_t E, int64_t N,
                                 int64_t K, int32_t *debug_partials, void *workspace,
                                 size_t workspace_bytes, w8a8_stream_t stream);

/*
 * w8a8_linear with the activation scale mode and the weight block size as
 * above (same workspace as w8a8_linear).
 */
w8a8_status w8a8_linear_ex(const void *a_bf16, int64_t lda, w8a8_scale_mode act_mode,
                           const int8_t *qw, const float *sw, int32_t sw_block_rows, void *y,
                           w8a8_dtype y_dtype, int64_t M, int64_t N, int64_t K, void *workspace,
                           size_t workspace_bytes, w8a8_stream_t stream);

/*
 * RMSNorm in front of the per-token quantizer, in one kernel (the quantizer
 * fused into the preceding normalisation: "Deploying Hunyuan 770B in INT8 on
 * domestic accelerators", §4.1 operator table, RMSNorm kept in high precision
 * next to the INT8 GEMMs, and §3.1, dynamic per-token INT8 activations).
 * Row m of x is normalised as
 *   y[m, k] = bf16_rn((x[m, k] * inv) * gamma[k]),
 *   inv = 1 / sqrt(sum_k x[m, k]^2 / K + eps),
 * with IEEE fp32 operations (every product rounded; the sum of squares in
 * fp32 in a fixed order, so results are run-to-run identical). y is the BF16
 * activation an unfused RMSNorm would write; its codes and scale are then
 * exactly what w8a8_quant_act / w8a8_quant_act_ex give for the rows y.
 *   x_bf16 [M, K] BF16, row stride ldx (multiple of 8, >= K), 16-byte aligned
 *   gamma_bf16 [K] BF16, 16-byte aligned
 *   eps > 0 and finite; K a multiple of 8, at most 32768
 * Accuracy of y against the exact value (real arithmetic on the same inputs):
 * the fp32 value before the BF16 rounding is within 2^-19 relative of it (at
 * most 32 sequential fma terms per thread and 10 tree levels in the sum of
 * squares, then five rounded operations), so y is within half a BF16 ulp plus
 * 2^-19 relative (tested).
 * Non-finite inputs give unspecified codes and scales.
 */
/* The normalised rows themselves: y_bf16 [M, K], row stride ldy (multiple of
 * 8, >= K), 16-byte aligned. */
w8a8_status w8a8_rmsnorm(const void *x_bf16, int64_t ldx, const void *gamma_bf16, float eps,
                         int64_t M, int64_t K, void *y_bf16, int64_t ldy, w8a8_stream_t stream);
/* Normalised and quantized: qa [M, ldq] int8 (ldq multiple of 8, >= K,
 * 8-byte aligned), sa [M] float; mode as for w8a8_quant_act_ex. */
w8a8_status w8a8_rmsnorm_quant(const void *x_bf16, int64_t ldx, const void *gamma_bf16, float eps,
                               w8a8_scale_mode mode, int64_t M, int64_t K, int8_t *qa,
                               int64_t ldq, float *sa, w8a8_stream_t stream);
/*
 * RMSNorm, quantization and the group-scaled GEMM: w8a8_linear applied to the
 * normalised rows y, with the normalisation done inside the quantizer kernel
 * (the BF16 rows y never reach HBM). Workspace and all GEMM arguments as for
 * w8a8_linear (w8a8_linear_workspace_size(M, N, K) bytes); x, gamma and eps as
 * above, K a multiple of 128. The result is identical to w8a8_rmsnorm
 * followed by w8a8_linear.
 */
w8a8_status w8a8_rmsnorm_linear(const void *x_bf16, int64_t ldx, const void *gamma_bf16, float eps,
                                const int8_t *qw, const float *sw, void *y, w8a8_dtype y_dtype,
                                int64_t M, int64_t N, int64_t K, void *workspace,
                                size_t workspace_bytes, w8a8_stream_t stream);

/*
 * Weight-only INT8 GEMM with BF16 activations (the "WNA16" reading of the
 * MoE runner on "Running DeepSeek-V4-Flash-Vision on 4xA800", §二: INT8
 * weights with one scale per group of 128 K, 16-bit activations that are not
 * quantized):
 *   Y[m, n] = sum_g sw[n / sw_block_rows, g] * P16[m, n, g],
 *   P16[m, n, g] = sum_{k in g} a[m, k] * qw[n, k]
 * a_bf16 [M, lda] BF16 (lda % 8 == 0, 16-byte aligned), qw [N, K] int8,
 * sw [ceil(N / sw_block_rows), K/128], y [M, N] BF16 or FP32. Each product of
 * a BF16 value and an integer of at most 7 bits is exact in FP32; the tensor
 * cores sum each group's products in FP32 (not exactly, unlike the integer
 * partials of w8a8_gemm), then the group scales are applied in the epilogue
 * in K order as in w8a8_gemm. FP32 outputs are within 1e-5 * T of the exact
 * value, T = sum_g |sw| * sum_k |a * qw| (tested). No workspace.
 */
w8a8_status w8a8_w8a16_gemm(const void *a_bf16, int64_t lda, const int8_t *qw, const float *sw,
                            int32_t sw_block_rows, void *y, w8a8_dtype y_dtype, int64_t M,
                            int64_t N, int64_t K, w8a8_stream_t stream);

/* The grouped (MoE) form over rows sorted by expert, offsets as in
 * w8a8_grouped_gemm; qw [E, N, K], sw [E, ceil(N / sw_block_rows), K/128]. */
w8a8_status w8a8_w8a16_grouped_gemm(const void *a_bf16, int64_t lda, const int32_t *offsets,
                                    const int8_t *qw, const float *sw, int32_t sw_block_rows,
                                    void *y, w8a8_dtype y_dtype, int64_t R, int64_t E, int64_t N,
                                    int64_t K, w8a8_stream_t stream);

/* ------------------------------------------------------------------------
 * MoE expert FFN ("Deploying Hunyuan 770B in INT8 on domestic accelerators":
 * §4.4, tokens are counted per destination expert first and then
 * transferred; §4.1 operator table, SwiGLU between the INT8 expert GEMMs;
 * §3.1, every INT8 GEMM input is quantized per token, dynamically). Each
 * token t has k (expert id, gate weight) pairs from its router, topk_ids and
 * topk_w [T, k] (row-major, on the device). The FFN of an expert e is
 *   h = silu(x W_gate[e]^T) * (x W_up[e]^T),   out_e(x) = h W_down[e]^T,
 * with W_gate_up[e] = [W_gate[e]; W_up[e]] ([2I, H], gate rows first) and
 * W_down[e] [H, I], both INT8 with per-row per-128-K-group scales, and
 *   y[t] = sum_j topk_w[t, j] * out_{topk_ids[t, j]}(x[t]).
 * Entries whose id lies outside [0, E) are not routed: they contribute
 * nothing. Numerics of each step are stated at its entry point below.
 * ------------------------------------------------------------------------ */

/*
 * Routing: per-expert counts of the n = T * k entries of topk_ids, their
 * exclusive prefix sum offsets [E+1] (offsets[E] = number of routed entries
 * R), and the permutation that sorts the routed entries by expert, ties in
 * entry order i = t * k + j (so by token): row_of [n] (the row of entry i,
 * -1 if not routed), token_of_row [n] and pair_of_row [n] (entry i of each
 * row; -1 for rows >= R). One CTA; all outputs are device int32 arrays. No
 * host read of any of them (the call can be captured in a CUDA graph).
 * 1 <= E <= 1024, k >= 1. T == 0 writes offsets = 0 only.
 */
w8a8_status w8a8_moe_route(const int32_t *topk_ids, int64_t T, int64_t k, int64_t E,
                           int32_t *offsets, int32_t *row_of, int32_t *token_of_row,
                           int32_t *pair_of_row, w8a8_stream_t stream);

/*
 * The transfer step fused with the per-token quantization: output row r of
 * qa [rows, K] (row stride K) and sa [rows] holds the w8a8_quant_act codes
 * and scale of row src_rows[r] of a_bf16 (row stride lda); rows whose
 * src_rows entry is negative are left untouched. Bit-identical to
 * w8a8_quant_act on the gathered rows.
 */
w8a8_status w8a8_quant_act_rows(const void *a_bf16, int64_t lda, const int32_t *src_rows,
                                int64_t rows, int64_t K, int8_t *qa, float *sa,
                                w8a8_stream_t stream);

/*
 * SwiGLU of the gate_up output followed by per-token requantization (the
 * down GEMM's input). U [rows, 2I] FP32 (gate in columns [0, I), up in
 * [I, 2I)); per row, in binary32:
 *   h = silu(gate) * up,  silu(g) = g / (1 + e^-g),
 * where e^x is evaluated by Cody and Waite's range reduction (x clamped to
 * [-87, 88], n = round-half-even(x log2 e), r = x - n ln2 with ln2 split into
 * 0.693145751953125 + 1.42860676533018e-06) and the degree-7 Taylor series of
 * e^r by Horner's rule, then scaled by 2^n; every step is a separately
 * rounded binary32 operation, so h is a fixed function of (gate, up). Then
 * sh[r] = amax|h| / 127 and qh[r, i] = clamp(round-half-even(h / sh[r]))
 * exactly as w8a8_quant_act. offsets (nullable) [E+1]: rows >= offsets[E]
 * are skipped (not routed). I % 4 == 0, I <= 8192.
 */
w8a8_status w8a8_swiglu_quant(const float *U, int64_t rows, int64_t I, const int32_t *offsets,
                              int64_t E, int8_t *qh, float *sh, w8a8_stream_t stream);

/*
 * h = silu(gate) * up alone (the first half of w8a8_swiglu_quant, same
 * arithmetic), FP32 [rows, I]; U and h 16-byte aligned.
 */
w8a8_status w8a8_swiglu(const float *U, int64_t rows, int64_t I, float *h, w8a8_stream_t stream);

/*
 * Weighted un-permute: y[t, :] = sum_{j < k} topk_w[t, j] * D[row_of[t*k + j], :]
 * over the routed entries (row_of >= 0), accumulated in FP32 in order of j
 * (fused multiply-add), then stored as BF16 (round to nearest even) or FP32.
 * D [R, H] FP32, row_of and topk_w [T, k], y [T, H]; H % 4 == 0; D and y
 * 16-byte aligned; k <= 64.
 */
w8a8_status w8a8_moe_unpermute(const float *D, const int32_t *row_of, const float *topk_w,
                               int64_t T, int64_t k, int64_t H, void *y, w8a8_dtype y_dtype,
                               w8a8_stream_t stream);

/*
 * Bytes of workspace w8a8_moe_ffn needs (n = T * k): offsets, the routing
 * arrays, the fp16 codes and scales of both GEMM inputs, and the FP32 outputs
 * of both GEMMs ([n, 2I] and [n, H]), each rounded up to 256 bytes. 0 for
 * invalid shapes or T == 0.
 */
size_t w8a8_moe_ffn_workspace_size(int64_t T, int64_t k, int64_t H, int64_t I, int64_t E);

/*
 * The MoE expert FFN in one call, six kernels on `stream`: w8a8_moe_route;
 * the transfer of the token rows into expert order fused with their
 * per-token quantization (w8a8_quant_act_rows, fp16 codes); the gate_up
 * grouped GEMM (FP32 output, as w8a8_grouped_gemm); w8a8_swiglu_quant (fp16
 * codes); the down grouped GEMM (FP32); w8a8_moe_unpermute into y.
 *   x_bf16 [T, ldx] BF16 tokens; topk_ids, topk_w [T, k] device arrays;
 *   qw_up [E, 2I, H] int8, sw_up [E, 2I, H/128]; qw_down [E, H, I] int8,
 *   sw_down [E, H, I/128]; y [T, H] BF16 or FP32 (16-byte aligned).
 * Results are identical to those separate calls (same kernels and codes).
 * H and I positive multiples of 128, I <= 8192, 1 <= k <= 64, 1 <= E <= 1024.
 * No host read of device data: the call can be captured in a CUDA graph.
 */
w8a8_status w8a8_moe_ffn(const void *x_bf16, int64_t ldx, const int32_t *topk_ids,
                         const float *topk_w, int64_t T, int64_t k, int64_t H, int64_t I,
                         int64_t E, const int8_t *qw_up, const float *sw_up,
                         const int8_t *qw_down, const float *sw_down, void *y, w8a8_dtype y_dtype,
                         void *workspace, size_t workspace_bytes, w8a8_stream_t stream);

/* ------------------------------------------------------------------------
 * INT8 KV cache ("Deploying Hunyuan 770B in INT8 on domestic accelerators",
 * §3.4: the KV cache is quantized to INT8 with a dynamic scale per key/value
 * vector, and the attention kernel dequantizes while it reads the cache
 * instead of running a separate dequantization pass; §2.2: the cache holds
 * 2 x layers x kv_heads x head_dim x seq_len x batch elements). One layer's
 * cache here: K and V [B, Hkv, S_max, head_dim] (row-major; one row per
 * vector), and for the INT8 form the scales [B, Hkv, S_max]. head_dim = 128.
 * ------------------------------------------------------------------------ */

/*
 * Writes n K or V vectors into an INT8 cache: vector i (x_bf16 [n, head_dim]
 * BF16) gets scale amax / 127 and codes clamp(round-half-even(x / scale)),
 * exactly as w8a8_quant_act, stored in row dst_rows[i] of cache [rows,
 * head_dim] int8 and scales [rows] (dst_rows NULL: row i; a negative entry:
 * not written). The caller maps (sequence, kv head, position) to a row, e.g.
 * (b * Hkv + h) * S_max + pos.
 */
w8a8_status w8a8_kv_quant(const void *x_bf16, int64_t n, int64_t head_dim,
                          const int32_t *dst_rows, int8_t *cache, float *scales,
                          w8a8_stream_t stream);

/* Bytes of workspace the decode attention calls need: per (sequence, query
 * head, chunk of 128 positions) a partial output and two statistics (FP32). */
size_t w8a8_attention_decode_workspace_size(int64_t B, int64_t Hq, int64_t S_max,
                                            int64_t head_dim);

/*
 * Decode attention of one query token per sequence over the INT8 cache,
 * grouped-query heads (query head hq reads kv head hq / (Hq / Hkv), Hq / Hkv
 * in {1, 2, 4, 8, 16}):
 *   s_j = softmax_scale * k_scale[j] * sum_d q[d] * k_code[j, d],
 *   out[d] = sum_j softmax(s)_j * v_scale[j] * v_code[j, d],  j < lens[b].
 * q [B, Hq, head_dim] BF16; lens [B] int32 on the device (clamped to
 * [0, S_max]; 0 gives zeros); out [B, Hq, head_dim] BF16 or FP32. Every
 * product and sum is FP32; a CTA handles 128 positions and the partial
 * softmax results are merged with max/sum rescaling (exact in real
 * arithmetic). Asynchronous, no host read of device data.
 */
w8a8_status w8a8_attention_decode_int8kv(const void *q_bf16, const int8_t *k_cache,
                                         const float *k_scale, const int8_t *v_cache,
                                         const float *v_scale, const int32_t *lens, int64_t B,
                                         int64_t Hq, int64_t Hkv, int64_t S_max,
                                         int64_t head_dim, float softmax_scale, void *out,
                                         w8a8_dtype out_dtype, void *workspace,
                                         size_t workspace_bytes, w8a8_stream_t stream);

/* The same attention over a BF16 cache (the unquantized baseline the fused
 * dequantization is measured against). */
w8a8_status w8a8_attention_decode_bf16kv(const void *q_bf16, const void *k_cache,
                                         const void *v_cache, const int32_t *lens, int64_t B,
                                         int64_t Hq, int64_t Hkv, int64_t S_max,
                                         int64_t head_dim, float softmax_scale, void *out,
                                         w8a8_dtype out_dtype, void *workspace,
                                         size_t workspace_bytes, w8a8_stream_t stream);

/*
 * Size of the scratch array built into the library for w8a8_gemm_noalloc:
 * 8 MiB, enough for M * K <= 4,194,304 activation codes (e.g. M <= 512 at
 * K = 8192, M <= 256 at K = 16384).
 */
#define W8A8_NOALLOC_SCRATCH_BYTES (8u << 20)

/*
 * w8a8_gemm without a caller workspace, for callers that cannot allocate
 * device memory at the point where they run the layer: for example an
 * inference engine that hands a plug-in only a stream and buffers it planned
 * ahead of time, a runtime whose memory pool forbids allocation on its hot
 * path, or code running where a cudaMalloc would synchronise the device. It
 * runs the kernels of w8a8_gemm, but its scratch is a fixed 8 MiB array that
 * is part of the library (W8A8_NOALLOC_SCRATCH_BYTES), so it allocates
 * nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 * There is no counterpart of this call on the source pages; it is a
 * deployment convenience.
 *   Arguments: as w8a8_gemm, without debug_partials and workspace.
 *   Returns W8A8_ERR_WORKSPACE when the fp16 copy of the activation codes,
 *   M * K * 2 bytes rounded up to 256, does not fit in the built-in scratch.
 *   What it computes: for M <= 4, and for M > 64, exactly what w8a8_gemm
 *   computes (same kernels, same results). For 5 <= M <= 64, w8a8_gemm splits
 *   tile K ranges over the SMs when its workspace holds the split area; here
 *   that area (1280 + 163,840 * M bytes, rounded up to 256) must fit in the
 *   scratch after the codes. When it does (e.g. M <= 46 at K = 8192, M <= 50
 *   at K = 1024) the result is again identical to w8a8_gemm's; when it does
 *   not (e.g. M >= 47 at K = 8192) the call runs unsplit, and its FP32 result
 *   may differ from w8a8_gemm's in the last bits: both are within the bound
 *   stated for w8a8_gemm (here with n = 1).
 *   The first call on a device looks up the scratch's device address (once,
 *   with that device current; make that first call before any stream
 *   capture) and keeps it for the life of the device's primary context: do
 *   not call this function again on a device after resetting it
 *   (cudaDeviceReset) in the same process. All calls on a device share the
 *   one scratch array and it keeps the last call's contents: calls that can
 *   overlap on the GPU (different streams without ordering between them)
 *   race on it and must be ordered by the caller.
 */
w8a8_status w8a8_gemm_noalloc(const int8_t *qa, const float *sa, const int8_t *qw,
                              const float *sw, void *y, w8a8_dtype y_dtype, int64_t M, int64_t N,
                              int64_t K, w8a8_stream_t stream);

/* Human-readable name of a status code (static storage). */
const char *w8a8_status_string(w8a8_status status);

/*
 * Reads (and, if clear != 0, resets) the current device's error word, which a
 * kernel sets when one of its bounded waits gives up instead of hanging.
 * Synchronises the device. *code_out = 0 means no device-side error; any other
 * value encodes the kernel, role and wait site. Returns W8A8_ERR_DEVICE_TIMEOUT
 * when the word was non-zero, W8A8_OK otherwise.
 */
w8a8_status w8a8_device_error(uint64_t *code_out, int clear);

/*
 * Diagnostic of the device-side failure path (no counterpart on the pages):
 * launches a one-thread kernel that waits, through the same bounded wait the
 * GEMM kernels use, on a barrier armed for bytes no copy will deliver. The
 * wait gives up after limit_us microseconds (1 .. 2,000,000) and records its
 * code in the error word; w8a8_device_error() then returns
 * W8A8_ERR_DEVICE_TIMEOUT with code = kernel 2, role 5, site 1, CTA 0
 * (bits 56..63, 48..55, 32..47, 0..31). Nothing traps or hangs and the
 * context stays usable. Asynchronous on `stream`.
 */
w8a8_status w8a8_selftest_wait_timeout(uint32_t limit_us, w8a8_stream_t stream);

/*
 * Rate probes of the integer-exact arithmetic the GEMMs run (diagnostics; no
 * counterpart on the pages). Each launches one kernel, asynchronously on
 * `stream`, and stores in *macs_out the number of int8 multiply-adds it
 * performs; the caller times the launch (CUDA events) to obtain the rate.
 * The operands are zeros (the rate does not depend on the values).
 *   w8a8_probe_tc_rate: one CTA per SM issues 8 * chains * steps
 *     tcgen05.mma kind::f16 instructions of shape M = 128, N = n, K = 16
 *     (A in tensor memory, B in shared memory: the instruction of the
 *     tensor-core GEMM), `chains` independent accumulators taking turns, all
 *     on the same A and B (distinct == 0) or each on its own (distinct != 0).
 *     16 <= n <= 256, n % 16 == 0, 1 <= chains <= 4, chains * n <= 256,
 *     1 <= steps <= 2^24 (keep one launch well under a second).
 *   w8a8_probe_dp4a_rate: 4 CTAs of 512 threads per SM, each thread 16 *
 *     iters dp4a (four int8 products into an int32; the CUDA-core GEMV's
 *     arithmetic). 1 <= iters <= 2^26.
 */
w8a8_status w8a8_probe_tc_rate(int32_t n, int32_t chains, int32_t distinct, int64_t steps,
                               int64_t *macs_out, w8a8_stream_t stream);
w8a8_status w8a8_probe_dp4a_rate(int64_t iters, int64_t *macs_out, w8a8_stream_t stream);

/* Library version: major * 10000 + minor * 100 + patch. */
int w8a8_version(void);

#ifdef __cplusplus
}
#endif

#endif /* W8A8_H */
