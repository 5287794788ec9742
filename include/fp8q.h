/*
 * fp8q.h -- C ABI of libfp8q: the FP8 W8A8 linear layer on NVIDIA GB300
 * (sm_103a).
 *
 * Two steps make up the layer:
 *   1. dynamic activation quantization, bf16 -> E4M3 (torch.float8_e4m3fn),
 *      either one fp32 scale per token (row) or one per (token, 128-column
 *      group) written into a row-padded buffer with column-major scales;
 *   2. the scaled FP8 GEMM, either per-token x per-output-channel scales or
 *      1x128 (activation) x 128x128 (weight) blockwise scales, with fp32
 *      accumulation, optional bias and bf16 (or fp16) output.
 *
 * Sources, cited by page title and section:
 *   [PR34331] "Tune FP8 GEMM Triton tiles on L40S and enable by default"
 *             (sgl-project/sglang PR 34331), "Key source snippets":
 *             apply_fp8_linear's channelwise branch calling
 *             fp8_scaled_mm(qinput, weight, x_scale, weight_scale,
 *             out_dtype, bias); the weight is [K, N]; the nearest-M tile
 *             lookup get_w8a8_channelwise_fp8_config.
 *   [PR27896] "Remove per-call padding overhead of the FP8 blockwise GEMM"
 *             (sgl-project/sglang PR 27896), "Key source snippets":
 *             sglang_per_token_group_quant_fp8_row_padded(x, group_size,
 *             eps=1e-10, row_alignment=4) and
 *             cutlass_w8a8_block_fp8_linear_with_fallback, which calls
 *             fp8_blockwise_scaled_mm(q_input, weight.T, x_scale,
 *             weight_scale.T, out_dtype) and slices the output to M rows.
 *
 * Conventions for every entry point:
 *   - Pointers named x, a, b, w, bias, out, *_scale and the quantized
 *     buffers are DEVICE pointers owned by the caller.  The library never
 *     allocates, frees or synchronizes; it only enqueues kernels.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  All work is asynchronous on that stream.
 *   - "bf16" data is bfloat16, "e4m3" data is one byte per element in the
 *     float8_e4m3fn encoding, scales are IEEE fp32.
 *   - Matrices are row-major with the given leading dimension (elements).
 *   - Device pointers to matrix data must be 16-byte aligned and leading
 *     dimensions must keep every row 16-byte aligned (the kernels use
 *     16-byte vector accesses and the Tensor Memory Accelerator).
 *   - Return value: FP8Q_OK, or an error code; on an error nothing was
 *     enqueued.  FP8Q_ERR_CUDA reports a failed launch (cudaGetLastError is
 *     consumed).  A GEMM whose internal pipeline wait exceeds its time limit
 *     records FP8Q_ERR_TIMEOUT in a device status word and returns early
 *     instead of hanging; read it with fp8q_device_status().
 *   - M == 0 is valid and enqueues nothing.
 *   - No C++ exception crosses this interface.
 *   - Kernels are launched with programmatic dependent launch: a kernel
 *     may start while the previous kernel in the stream is still running.
 *     Every kernel of the library first waits for its predecessor and only
 *     then lets its own successor launch, so at most the immediate
 *     predecessor can be running when a kernel starts.  A GEMM streams its
 *     WEIGHT operand before that wait unless the library's own most recent
 *     launch on the same stream writes an overlapping byte range (then it
 *     waits first).  A foreign kernel that triggers programmatic
 *     dependents before its writes are complete must therefore not write
 *     the weights of a GEMM launched right after it; ordinary kernels and
 *     copies (no such trigger) are always safe producers.
 *   - Consecutive calls on one stream are ordered as usual; calls racing on
 *     different streams need the caller's own synchronization.
 */
#ifndef FP8Q_H_
#define FP8Q_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FP8Q_API __attribute__((visibility("default")))
#else
#define FP8Q_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP8Q_OK = 0,
    FP8Q_ERR_INVALID_ARG = 1, /* null pointer, bad size, stride or alignment */
    FP8Q_ERR_UNSUPPORTED = 2, /* a shape or option the library does not implement */
    FP8Q_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
    FP8Q_ERR_TIMEOUT = 4      /* a device-side pipeline wait ran out of time */
} fp8q_status;

typedef enum { FP8Q_OUT_BF16 = 0, FP8Q_OUT_FP16 = 1 } fp8q_out_dtype;

/* Largest finite E4M3 value: the quantizers map amax to +-448. */
#define FP8Q_E4M3_MAX 448.0f

/* ---------------------------------------------------------------------------
 * fp8q_quant_per_token -- per-token dynamic quantization.
 * Defined by the channelwise path of [PR34331] "Key source snippets"
 * (qinput with one x_scale entry per row):
 *   s[m]    = max(amax_k |x[m,k]|, eps) / 448          (fp32, IEEE division)
 *   xq[m,k] = e4m3_rne_satfinite(x[m,k] / s[m])        (fp32 quotient)
 * x       : bf16 [M, K], row stride ldx >= K (ldx % 8 == 0), 16-byte aligned.
 * xq      : e4m3 [M, K], row stride K (K % 16 == 0), 16-byte aligned.
 * x_scale : fp32 [M].
 * eps     : floor on amax (the pages use 1e-10); must be > 0 and finite.
 * Errors  : INVALID_ARG for M < 0, K <= 0, K % 16 != 0, ldx < K, ldx % 8,
 *           null or misaligned pointers, eps <= 0.
 * ------------------------------------------------------------------------- */
FP8Q_API fp8q_status fp8q_quant_per_token(const void *x, int64_t M, int64_t K, int64_t ldx,
                                 void *xq, float *x_scale, float eps, void *stream);

/* ---------------------------------------------------------------------------
 * fp8q_quant_per_token_group_row_padded -- per-token-group quantization into
 * a row-padded buffer, [PR27896] "Key source snippets"
 * (sglang_per_token_group_quant_fp8_row_padded):
 *   for each row m < M and group j < K/g:
 *     s        = max(amax over x[m, j*g : (j+1)*g], eps) / 448
 *     x_scale[j * m_pad + m] = s            (column-major (m_pad, K/g) view)
 *     xq[m, j*g + i] = e4m3_rne_satfinite(x[m, j*g + i] / s)
 *   Rows m >= M of xq and of x_scale are NEVER written (the caller's
 *   padding; the GEMM never lets them reach the first M output rows).
 * x          : bf16 [M, K], row stride ldx >= K (ldx % 8 == 0).
 * group_size : g in {16, 32, 64, 128}; K % g == 0.
 * row_alignment : the padding multiple (the pages use 4); m_pad >= M and
 *              m_pad % row_alignment == 0 (the pages allocate
 *              m_pad = ceil(M / row_alignment) * row_alignment).
 * xq         : e4m3 [m_pad, K], row stride K (K % 16 == 0).
 * x_scale    : fp32 storage of K/g columns of m_pad entries (column-major).
 * Errors     : INVALID_ARG for bad sizes, m_pad < M, m_pad % row_alignment,
 *              K % g, null or misaligned pointers; UNSUPPORTED for other g.
 * ------------------------------------------------------------------------- */
FP8Q_API fp8q_status fp8q_quant_per_token_group_row_padded(const void *x, int64_t M, int64_t K, int64_t ldx,
                                                  int32_t group_size, float eps,
                                                  int32_t row_alignment, void *xq,
                                                  float *x_scale, int64_t m_pad, void *stream);

/* ---------------------------------------------------------------------------
 * fp8q_quant_per_token_group_row_padded_ex -- the group quantizer above
 * with the two options its kernel takes in [PR27896] "Key source snippets"
 * (the scale_ue8m0 and fuse_silu_and_mul arguments, passed as False
 * there); `flags` is a bitwise OR of:
 *   FP8Q_QUANT_SCALE_UE8M0  each group scale max(amax, eps) / 448 is
 *       rounded up to a power of two before use (an exact 8-bit exponent):
 *       the smallest normal fp32 power of two >= the scale (2^-126 for
 *       smaller scales).  x / s is then exact before the E4M3 rounding.
 *   FP8Q_QUANT_SILU_AND_MUL  x is bf16 [M, 2K] (row stride ldx >= 2K): the
 *       quantized values are y[m,k] = silu(x[m,k]) * x[m,K+k], computed in
 *       fp32 with no rounding in between, silu(a) = a / (1 + exp(-a)) with
 *       IEEE fp32 add and division and exp the library's fixed fp32
 *       sequence (Cody-Waite reduction with FMAs, degree-7 Taylor series,
 *       within 2 ulp of exp; exp(t) = +inf for t > 88 and 0 for t < -32).
 *       The amax, scale and y / s (IEEE division) follow as above; xq is
 *       [m_pad, K].
 * flags == 0 is exactly fp8q_quant_per_token_group_row_padded.
 * Errors     : as above; INVALID_ARG for unknown flag bits or, with
 *              SILU_AND_MUL, ldx < 2K.
 * ------------------------------------------------------------------------- */
#define FP8Q_QUANT_SCALE_UE8M0 1
#define FP8Q_QUANT_SILU_AND_MUL 2
FP8Q_API fp8q_status fp8q_quant_per_token_group_row_padded_ex(const void *x, int64_t M, int64_t K, int64_t ldx,
                                                     int32_t group_size, float eps,
                                                     int32_t row_alignment, int32_t flags, void *xq,
                                                     float *x_scale, int64_t m_pad, void *stream);

/* ---------------------------------------------------------------------------
 * fp8q_quant_static_per_tensor -- static per-tensor quantization with one
 * precomputed scale (the _static_quant_fp8 kernel named in [PR31340]
 * "Implementation breakdown"):
 *   xq[m,k] = e4m3_rne_satfinite(x[m,k] / s)        (fp32 quotient)
 *   x_scale_rep[m] = s  for m < M, if x_scale_rep != NULL (the per-token
 *   scale vector fp8q_scaled_mm_channelwise takes).
 * x           : bf16 [M, K], row stride ldx >= K (ldx % 8 == 0), 16-byte aligned.
 * scale       : DEVICE pointer to one fp32 s, read by the kernel (so it may be
 *               produced by an earlier kernel on the stream); s must be > 0
 *               and finite -- other values give unspecified codes, no error.
 * xq          : e4m3 [M, K], row stride K (K % 16 == 0), 16-byte aligned.
 * x_scale_rep : fp32 [M] or NULL.
 * Errors      : INVALID_ARG for M < 0, K <= 0, K % 16, ldx < K, ldx % 8,
 *               null or misaligned pointers.
 * ------------------------------------------------------------------------- */
FP8Q_API fp8q_status fp8q_quant_static_per_tensor(const void *x, int64_t M, int64_t K, int64_t ldx,
                                         const float *scale, void *xq, float *x_scale_rep,
                                         void *stream);

/* ---------------------------------------------------------------------------
 * fp8q_quant_weight_block128 -- weight preparation for the blockwise GEMM
 * (one fp32 scale per 128 x 128 block, same scale and cast rule as the
 * activations).  Not on the per-call hot path: weights are quantized once.
 * w       : bf16 [N, K] row-major (ld = K), N % 128 == 0, K % 128 == 0.
 * wq      : e4m3 [N, K]; w_scale: fp32 [N/128][K/128] row-major.
 * ------------------------------------------------------------------------- */
FP8Q_API fp8q_status fp8q_quant_weight_block128(const void *w, int64_t N, int64_t K, void *wq,
                                       float *w_scale, float eps, void *stream);

/* ---------------------------------------------------------------------------
 * fp8q_scaled_mm_channelwise -- [PR34331] "Key source snippets",
 * fp8_scaled_mm(qinput, weight, x_scale, weight_scale, out_dtype, bias):
 *   out[m,n] = cvt( (sum_k a[m,k] * b[k,n]) * a_scale[m] * b_scale[n]
 *                   (+ bias[n]) )
 *   fp32 accumulation; one rounding to the output type.
 * a       : e4m3 [M, K] row-major, ld = K (K % 16 == 0).
 * b       : e4m3 weight, logically [K, N], stored K-contiguous: element
 *           (k, n) at b[n * ldb + k]  (i.e. an [N, K] row-major matrix);
 *           ldb >= K, ldb % 16 == 0.
 * a_scale : fp32 [M]; b_scale : fp32 [N]; bias : bf16 [N] or NULL.
 * out     : [M, N] row-major (ld = N) of out_dtype (N % 8 == 0).
 * workspace, workspace_bytes : optional DEVICE scratch for the split-K
 *           partial sums (see fp8q_workspace_bytes); NULL / 0, too small for
 *           the schedule, or the workspace exchange not enabled: the
 *           partials are exchanged in distributed shared memory instead.
 *           Same result either way.
 * Errors  : INVALID_ARG / UNSUPPORTED as above; INVALID_ARG for a
 *           workspace that is not 16-byte aligned.
 * ------------------------------------------------------------------------- */
FP8Q_API fp8q_status fp8q_scaled_mm_channelwise(const void *a, const void *b, int64_t ldb,
                                       const float *a_scale, const float *b_scale,
                                       const void *bias, void *out, int64_t M, int64_t N,
                                       int64_t K, fp8q_out_dtype out_dtype, void *workspace,
                                       size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * fp8q_scaled_mm_blockwise -- [PR27896] "Key source snippets",
 * fp8_blockwise_scaled_mm(q_input, weight.T, x_scale, weight_scale.T) with
 * the output sliced to the first M rows and the bias added after:
 *   out[m,n] = cvt( sum_kb P_kb(m,n) * a_scale[kb * m_pad + m]
 *                                   * w_scale[(n/128) * (K/128) + kb]
 *                   (+ bias[n]) ),
 *   P_kb(m,n) = sum over the 128 k of block kb of a[m,k] * w[n,k]
 * a       : e4m3 [m_pad, K] (the row-padded quantizer's output); rows >= M
 *           are ignored, whatever they hold.
 * w       : e4m3 [N, K] row-major; N % 128 == 0, K % 128 == 0.
 * a_scale : fp32 column-major activation scales, K/128 columns of m_pad.
 * w_scale : fp32 [N/128][K/128] row-major.
 * bias    : bf16 [N] or NULL.   out : [M, N] row-major of out_dtype.
 * m_pad   : >= M and a multiple of 4 (keeps each scale column 16-byte
 *           aligned for the Tensor Memory Accelerator).
 * workspace, workspace_bytes : as fp8q_scaled_mm_channelwise.
 * Errors  : UNSUPPORTED when N or K is not a multiple of 128 (the pages
 *           fall back to another kernel there; this library refuses).
 * ------------------------------------------------------------------------- */
FP8Q_API fp8q_status fp8q_scaled_mm_blockwise(const void *a, const void *w, const float *a_scale,
                                     const float *w_scale, const void *bias, void *out,
                                     int64_t M, int64_t m_pad, int64_t N, int64_t K,
                                     fp8q_out_dtype out_dtype, void *workspace,
                                     size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * fp8q_workspace_bytes -- the split-K workspace of the GEMM the library
 * would launch for (M, N, K, blockwise) on the CURRENT device (the
 * schedule depends on its SM count and on any plan override in force).
 * 0 when that schedule does not split K (then no workspace is used).
 * The scratch argument of the GEMM calls on the pages' interface (the
 * fp8_scaled_mm / fp8_blockwise_scaled_mm callers own all device memory).
 *
 * Stream-K schedules (fp8q_plan.stream_k; decode-size M): grid slots of
 * 128 x mma_n floats, then grid 32-bit flags (grid * (512 * mma_n + 4)
 * bytes).  Such a workspace MUST BE ZERO-FILLED before its first use
 * (cudaMemset); every completed GEMM leaves its flags at zero again, so
 * later calls (and CUDA-graph replays) need no further clearing.  After a
 * call that reported FP8Q_ERR_TIMEOUT, zero it again.  A workspace that is
 * NULL or smaller than this makes the GEMM fall back to a K-split schedule
 * (correct, slower at these sizes).
 *
 * With K split over a cluster of s CTAs, each CTA computes an fp32 partial
 * tile over its range of K blocks, and each CTA adds up its share of the
 * tile's outputs over all s partials in a fixed order.  The other CTAs'
 * partials reach it in one of two ways, with identical results:
 *   - through distributed shared memory (the default);
 *   - through this workspace (one slot of 128 x mma_n floats per CTA:
 *     tiles * s * 128 * mma_n * 4 bytes): every CTA bulk-copies the rows
 *     other CTAs own into its slot, a cluster barrier publishes them, and
 *     each CTA bulk-loads its rows from the other slots.  Used only for
 *     partial tiles of 128 x 128 floats or more, and only when the process
 *     starts with FP8Q_WORKSPACE_EXCHANGE=1: on the GB300s this library was
 *     measured on, it was slower than the distributed-shared-memory
 *     exchange at every schedule (partials just written by other SMs came
 *     back through global memory at 10-30 GB/s per SM).
 * So by default this returns 0 for K-split schedules and the GEMMs
 * ignore a workspace there.  For K-split schedules nothing in the
 * workspace has to be initialised, and its contents are undefined after
 * the call.  Calls that can run concurrently on the GPU need
 * separate workspaces; calls in order on one stream can share one.
 * Returns 0 as well for invalid sizes (M <= 0, N <= 0, K <= 0).
 * ------------------------------------------------------------------------- */
FP8Q_API size_t fp8q_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t blockwise);

/* ---------------------------------------------------------------------------
 * Linear-layer compositions (no padding copies): quantize x into the
 * caller's buffers, then run the GEMM on them -- two launches, except:
 * fp8q_linear_channelwise with ONE token, K <= 12288 and N * K <= 4096^2
 * (and no schedule override set) runs as one launch, the per-token quantization fused into a
 * matrix-vector product on the CUDA cores (every CTA quantizes the row into
 * its shared memory; CTA 0 also writes xq and xs, so they hold the same
 * codes and scales as after the two launches).  Its sums are accumulated in
 * another order than the tensor-core GEMM's, so its output is within the
 * GEMM tolerance of the two-kernel result rather than bit-identical.
 * fp8q_linear_blockwise with ONE token and K <= 12288 (no override) is one
 * launch as well: the group-128 quantization fused into the matrix-vector
 * product (each 16-value partial sum scaled by its group scale times its
 * weight block's scale), xq row 0 and xs[kb * m_pad] written by CTA 0.
 * fp8q_linear_channelwise_launches / fp8q_linear_blockwise_launches tell
 * which form a call takes.
 * fp8q_linear_channelwise : xq e4m3 [M, K], xs fp32 [M].
 * fp8q_linear_blockwise   : xq e4m3 [m_pad, K], xs fp32 [K/128][m_pad],
 *   m_pad = ceil(M/4)*4 or a larger multiple of 4 -- the row-padded
 *   pipeline of [PR27896] "Implementation breakdown" (quantizer writes the
 *   GEMM's final layout; output sliced to M rows).
 * workspace, workspace_bytes : passed to the GEMM (fp8q_workspace_bytes).
 * ------------------------------------------------------------------------- */
FP8Q_API fp8q_status fp8q_linear_channelwise(const void *x, const void *b, int64_t ldb,
                                    const float *b_scale, const void *bias, void *out,
                                    int64_t M, int64_t N, int64_t K, void *xq, float *xs,
                                    fp8q_out_dtype out_dtype, void *workspace,
                                    size_t workspace_bytes, void *stream);
FP8Q_API fp8q_status fp8q_linear_blockwise(const void *x, const void *w, const float *w_scale,
                                  const void *bias, void *out, int64_t M, int64_t N, int64_t K,
                                  void *xq, float *xs, int64_t m_pad, fp8q_out_dtype out_dtype,
                                  void *workspace, size_t workspace_bytes, void *stream);
/* Kernel launches fp8q_linear_channelwise makes for M tokens of K values
 * against N output channels: 1 (the fused one-token form), 2 (quantizer +
 * GEMM), or 0 for M, N or K <= 0.  Host only; reads the schedule override. */
FP8Q_API int32_t fp8q_linear_channelwise_launches(int64_t M, int64_t N, int64_t K);
/* The same for fp8q_linear_blockwise. */
FP8Q_API int32_t fp8q_linear_blockwise_launches(int64_t M, int64_t K);

/* ---------------------------------------------------------------------------
 * fp8q_scaled_mm_w8a16 -- weight-only FP8 linear (W8A16): bf16 activations
 * against E4M3 weights with one fp32 scale per output channel, the
 * weight-only linear of [PR31340] "Implementation breakdown" / "Key source
 * snippets" (apply_fp8_marlin_linear(input, weight, weight_scale, ...,
 * bias): no input scale):
 *   out[m,n] = round(sum_k x[m,k] * e4m3(w[n,k]) * w_scale[n] + bias[n])
 * (a per-tensor weight scale is the case of equal entries).  M <= 2: matrix-
 * vector products on the CUDA cores (weights decoded exactly to fp32 in
 * registers, fp32 FMAs), the weight stream at HBM speed.  M > 2: fp32-
 * accumulated bf16 x bf16 MMAs on the weights converted exactly to bf16 into
 * tensor memory (tcgen05.mma kind::f16, A operand in TMEM), tiles of 128
 * weight rows x 16 (M <= 16) or 32 tokens, K split across a cluster while
 * the tiles do not fill the GPU (any M works; larger M simply takes more
 * token tiles).
 * x       : bf16 [M, K], row stride ldx >= K (ldx % 8 == 0), 16-byte aligned.
 * w       : e4m3 [N, K] row-major, row stride ldw >= K (ldw % 16 == 0).
 * w_scale : fp32 [N].  bias: bf16 [N] or NULL.  out: [M, N] (row stride N).
 * Errors  : INVALID_ARG for M < 0, N, K <= 0, K % 16, N % 8, bad strides,
 *           null or misaligned pointers; UNSUPPORTED for other out_dtype.
 * ------------------------------------------------------------------------- */
FP8Q_API fp8q_status fp8q_scaled_mm_w8a16(const void *x, int64_t ldx, const void *w, int64_t ldw,
                                 const float *w_scale, const void *bias, void *out, int64_t M,
                                 int64_t N, int64_t K, fp8q_out_dtype out_dtype, void *stream);

/* ---------------------------------------------------------------------------
 * fp8q_linear_blockwise_fused -- the blockwise linear layer in ONE kernel:
 * the row-padded group-128 quantization of fp8q_linear_blockwise is done
 * inside the GEMM, on the activation tiles it consumes (the quantization
 * "optionally fused" into the GEMM; group scales are local to each 128-wide
 * K block, so every CTA quantizes exactly the blocks it multiplies).  Codes
 * and scales are those of fp8q_quant_per_token_group_row_padded (g = 128,
 * eps = 1e-10), so the output is bit-identical to fp8q_linear_blockwise on
 * the same schedule.
 * Available where the planner's schedule is the 16- or 32-token swapped
 * tile (decode sizes, M <= 32 on the compiled table's shapes); other
 * problems return FP8Q_ERR_UNSUPPORTED.  A stream-K plan runs here as the
 * same tiles split along K (no workspace is taken).  Measured on GB300 it is SLOWER than the
 * two-kernel fp8q_linear_blockwise on back-to-back layers (the activation
 * reads issued after the dependency wait queue behind the weight stream),
 * so fp8q_linear_blockwise does not use it; it is for callers that want a
 * single launch per layer with the GEMM's tensor-core sums.  (For ONE token
 * fp8q_linear_blockwise is itself a single, faster launch -- the
 * matrix-vector form above -- whose sums run in another order.)
 * x   : bf16 [M, K], row stride ldx >= K (ldx % 8 == 0), 16-byte aligned.
 * w, w_scale, bias, out, out_dtype: as fp8q_linear_blockwise.  No scratch.
 * ------------------------------------------------------------------------- */
FP8Q_API fp8q_status fp8q_linear_blockwise_fused(const void *x, int64_t ldx, const void *w, const float *w_scale,
                                        const void *bias, void *out, int64_t M, int64_t N, int64_t K,
                                        fp8q_out_dtype out_dtype, void *stream);

/* ---------------------------------------------------------------------------
 * fp8q_linear_channelwise_noalloc -- the pages have no counterpart: this is
 * an addition of this library for callers that cannot allocate.
 *
 * Same computation, arguments and errors as fp8q_linear_channelwise, minus
 * the scratch buffers xq and xs and the workspace (K splits exchange their
 * partial sums in distributed shared memory): the E4M3 codes and per-token scales live
 * in a fixed array inside the library (a file-scope __device__ array of
 * FP8Q_NOALLOC_MAX_CODES + 4 * FP8Q_NOALLOC_MAX_ROWS bytes = 16 MiB + 64 KiB,
 * held on every GPU that loads the library until the process exits).
 * Where the planned schedule is stream-K (which needs a workspace), this
 * entry runs the K-split schedule of the same tiles, as
 * fp8q_linear_channelwise does without a workspace; the output can then
 * differ in the last bits (fp32 summation order) from a call with one.
 * It is meant for callers that cannot call cudaMalloc: code whose device
 * memory is handed out entirely by a host framework's own pool (a plugin
 * given no workspace, an engine that budgets every byte up front), or a
 * latency-bound loop that cannot take the device synchronisation that
 * cudaMalloc / cudaFree imply.  The call allocates and frees nothing.
 *
 * Limits  : M <= FP8Q_NOALLOC_MAX_ROWS and M * K <= FP8Q_NOALLOC_MAX_CODES;
 *           larger problems return FP8Q_ERR_UNSUPPORTED before any CUDA
 *           call (use fp8q_linear_channelwise with your own buffers).
 * Set-up  : the first call on each device looks up the array's device
 *           address (cudaGetSymbolAddress, with that device current) and
 *           caches it; make that first call before any stream capture.
 *           A failed look-up returns FP8Q_ERR_CUDA.  The device is the
 *           CURRENT device: make the device of x, out and stream current
 *           before the call.  The cached address belongs to the device's
 *           primary context; after cudaDeviceReset on that device it is no
 *           longer valid, so do not call this entry point in a process that
 *           has reset the device after its first call.
 * Sharing : every call on a device uses the same array, which keeps the
 *           last call's contents (nothing in it needs to start at zero:
 *           the quantizer writes every code and scale the GEMM reads).
 *           Calls in order on one stream are safe; calls that can overlap
 *           on the GPU (different streams without synchronisation between
 *           them) race on the array and give wrong results.
 * ------------------------------------------------------------------------- */
#define FP8Q_NOALLOC_MAX_CODES (16LL * 1024 * 1024)
#define FP8Q_NOALLOC_MAX_ROWS 16384LL
FP8Q_API fp8q_status fp8q_linear_channelwise_noalloc(const void *x, const void *b, int64_t ldb,
                                            const float *b_scale, const void *bias, void *out,
                                            int64_t M, int64_t N, int64_t K,
                                            fp8q_out_dtype out_dtype, void *stream);

/* ---------------------------------------------------------------------------
 * Tile selection (host only, no GPU needed).  The GEMM schedule for a
 * problem: which operand sits on the MMA's 128-row side, the MMA N extent,
 * the K-split count (CTAs of one thread-block cluster that share a tile and
 * add up their partial sums through the workspace or distributed shared
 * memory), pipeline depth
 * and grid size.  The choice comes from a compiled-in table keyed by
 * (N, K, scheme) with nearest-M lookup, ties to the smaller M, as in
 * get_w8a8_channelwise_fp8_config of [PR34331] "Key source snippets";
 * shapes without an entry use a generic rule.  num_sms <= 0 means "ask the
 * current device".  Errors: INVALID_ARG for M < 0, N <= 0, K <= 0 or a null
 * plan; ERR_CUDA if the SM count cannot be read.
 * ------------------------------------------------------------------------- */
typedef struct {
    int32_t swap_ab;    /* 1: 128 weight rows x mma_n tokens per tile (decode);
                           0: 128 tokens x mma_n weight rows per tile (prefill) */
    int32_t mma_n;      /* tcgen05.mma N extent: 16, 32, 64, 128 or 256 */
    int32_t tile_m;     /* tokens per output tile */
    int32_t tile_n;     /* output columns per output tile */
    int32_t split_k;    /* CTAs per cluster sharing one tile along K (1..8) */
    int32_t stages;     /* shared-memory pipeline depth */
    int32_t grid;       /* CTAs launched */
    int32_t persistent; /* 1: CTAs loop over several tiles */
    int32_t from_table; /* 1: taken from the compiled-in table */
    int32_t pair;       /* 1: CTA pairs (2-CTA clusters) on adjacent token tiles
                           (non-swapped channelwise, split_k 1, at least two
                           token tiles) */
    int32_t two_sm;     /* 1: each CTA pair computes a 256-token x 256-column
                           tile with 2-CTA MMAs (tcgen05 cta_group::2), each
                           CTA loading only its half of the weight rows
                           (always equal to pair) */
    int32_t stream_k;   /* 1 (swapped tiles of 16 or 32 tokens; split_k 1,
                           grid <= SMs):
                           stream-K -- each CTA takes an equal share of the
                           (tile, 128-wide K block) pairs in tile-major order,
                           and a CTA whose share starts inside a tile hands
                           its fp32 partial sums to the CTA holding that
                           tile's first K block through the workspace (see
                           fp8q_workspace_bytes, which then sizes it).
                           Without that workspace, and in the fused and
                           weight-only GEMMs, the GEMM runs a K-split
                           schedule of the same tiles instead. */
    int32_t kb_per_stage; /* 128-wide K blocks per pipeline stage: 2 for the
                           channelwise non-swapped tiles of 32, 64 or 128
                           columns with split_k 1, no pair and K a multiple
                           of 128 (one 3-D TMA box per operand and stage;
                           `stages` then counts double stages), else 1 */
} fp8q_plan;

FP8Q_API fp8q_status fp8q_gemm_plan(int64_t M, int64_t N, int64_t K, int32_t blockwise, int32_t num_sms,
                           fp8q_plan *plan);

/* Force the schedule of every following GEMM in this process (for tests
 * and tuning sweeps): swap_ab in {0, 1} with an mma_n that has a kernel
 * instantiation (swapped: 16, 32, 64, 128; non-swapped: 32, 64, 128, 256) and
 * split_k >= 1 (clamped to 8 and to the number of 128-wide K blocks), or
 * split_k == 0 with swap_ab == 1 and mma_n 16 or 32 for stream-K
 * (fp8q_plan.stream_k).
 * swap_ab < 0 removes the override.  Errors: INVALID_ARG for a
 * combination without an instantiation.  Not thread-safe with concurrent
 * GEMM calls. */
FP8Q_API fp8q_status fp8q_set_plan_override(int32_t swap_ab, int32_t mma_n, int32_t split_k);

/* Device status word: returns FP8Q_OK or the first device-side error the
 * GEMM kernels recorded on the current device (FP8Q_ERR_TIMEOUT).
 * Synchronizes `stream`.  reset != 0 clears the word afterwards. */
FP8Q_API fp8q_status fp8q_device_status(void *stream, int32_t reset);

/* The same word read without clearing it: fp8q_device_status(stream, 0),
 * under the name the boundary's design used. */
FP8Q_API fp8q_status fp8q_last_device_status(void *stream);

/* Diagnostics (the pages have no counterpart): enqueue a one-warp kernel
 * whose pipeline wait can never complete.  The bounded wait the GEMM uses
 * gives up after its time limit (about 2 s), records FP8Q_ERR_TIMEOUT in
 * the device status word and the kernel returns: nothing hangs and the
 * context stays usable.  Read (and reset) the word with fp8q_device_status.
 * Returns FP8Q_OK if the kernel was enqueued, ERR_CUDA otherwise. */
FP8Q_API fp8q_status fp8q_selftest_wait_timeout(void *stream);

/* Diagnostics: out[i] = silu(a[i]) * b[i] in fp32 for i < n, computed by the
 * device function of the silu_and_mul-fused group quantizer
 * (FP8Q_QUANT_SILU_AND_MUL; the silu_and_mul input of the row-padding page,
 * key source snippets): a / (1 + exp(-a)) with the library's fixed exp
 * sequence and the correctly rounded fp32 add and quotient, then one fp32
 * multiply by b.  Lets tests compare that arithmetic with a reference bit for
 * bit rather than through 8-bit codes.
 * a, b, out: device fp32 arrays of n elements (4-byte aligned); n >= 0
 * (n = 0: nothing is enqueued).  Enqueued on `stream`, not synchronized.
 * Errors: INVALID_ARG (n < 0 or above 2^40, a null pointer with n > 0),
 * ERR_CUDA (launch failure). */
FP8Q_API fp8q_status fp8q_selftest_silu_mul(const float *a, const float *b, float *out, int64_t n, void *stream);

/* Human-readable name of a status code (static string). */
FP8Q_API const char *fp8q_status_str(fp8q_status status);

/* ABI version: (major << 16) | minor. */
FP8Q_API int32_t fp8q_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8Q_H_ */
