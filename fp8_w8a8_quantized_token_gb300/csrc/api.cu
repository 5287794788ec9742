// api.cu -- the C ABI (include/fp8q.h): argument validation, schedule
// selection and kernel launches.  No allocation, no synchronization (except
// fp8q_device_status, which exists to synchronize), no exceptions.
#include <cuda_runtime.h>
#include <math.h>
#include <stdlib.h>
#include <stdint.h>

#include "../../include/fp8q.h"
#include "internal.h"

namespace {

using namespace fp8q;

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

inline fp8q_status from_cuda(cudaError_t e) { return e == cudaSuccess ? FP8Q_OK : FP8Q_ERR_CUDA; }

inline cudaStream_t as_stream(void *s) { return static_cast<cudaStream_t>(s); }

// The kernels index with 32-bit ints in places; keep every extent in range.
constexpr int64_t kMaxDim = (int64_t{1} << 31) - 1;

fp8q_status check_quant_common(const void *x, int64_t M, int64_t K, int64_t ldx, const void *xq, const float *xs,
                               float eps)
{
    if (M < 0 || K <= 0 || M > kMaxDim || K > kMaxDim) return FP8Q_ERR_INVALID_ARG;
    if (K % 16 != 0 || ldx < K || ldx % 8 != 0) return FP8Q_ERR_INVALID_ARG;
    if (!(eps > 0.0f) || !isfinite(eps)) return FP8Q_ERR_INVALID_ARG;
    if (M == 0) return FP8Q_OK;
    if (x == nullptr || xq == nullptr || xs == nullptr) return FP8Q_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(xq) || !aligned4(xs)) return FP8Q_ERR_INVALID_ARG;
    return FP8Q_OK;
}

fp8q_status launch_planned(GemmProblem p, const fp8q_plan &pl, cudaStream_t st)
{
    // Weight bytes the kernel may read before waiting for its predecessor.
    const size_t wbytes = static_cast<size_t>(p.N - 1) * static_cast<size_t>(p.ldw) + static_cast<size_t>(p.K);
    p.preload = !last_launch_writes_overlap(st, p.w, wbytes);
    unsigned *status = device_status_ptr();
    if (status == nullptr) return FP8Q_ERR_CUDA;
    // Stream-K needs its workspace and exists only for the plain E4M3
    // kernels; otherwise the same tiles run split along K.
    fp8q_plan plan = pl;
    if (plan.stream_k && (p.fused_quant || p.w16 || p.ws == nullptr ||
                          p.ws_bytes < stream_k_workspace_bytes(plan.grid, plan.mma_n)))
        plan_without_stream_k(p.M, p.N, p.K, p.blockwise ? 1 : 0, current_device_sms(), &plan);
    GemmLaunch l;
    l.swap_ab = plan.swap_ab != 0;
    l.mma_n = plan.mma_n;
    l.split = plan.split_k;
    l.grid = plan.grid;
    l.stages = plan.stages;
    l.pair = plan.pair != 0;
    l.two_sm = plan.two_sm != 0;
    l.stream_k = plan.stream_k != 0;
    l.wide = plan.kb_per_stage == 2;
    const cudaError_t e = p.blockwise ? launch_gemm_blockwise(p, l, status, st)
                                      : launch_gemm_channelwise(p, l, status, st);
    if (e == cudaSuccess) note_launch_writes(st, p.out, static_cast<size_t>(p.M) * p.N * 2);
    return from_cuda(e);
}

fp8q_status run_gemm(const GemmProblem &p, cudaStream_t st)
{
    fp8q_plan pl;
    const fp8q_status s = fp8q_gemm_plan(p.M, p.N, p.K, p.blockwise ? 1 : 0, 0, &pl);
    if (s != FP8Q_OK) return s;
    return launch_planned(p, pl, st);
}

}  // namespace

namespace fp8q {
void plan_finish(int64_t M, int64_t N, int64_t K, int blockwise, int num_sms, fp8q_plan *pl);
}

extern "C" {

fp8q_status fp8q_quant_per_token(const void *x, int64_t M, int64_t K, int64_t ldx, void *xq, float *x_scale,
                                 float eps, void *stream)
{
    const fp8q_status s = check_quant_common(x, M, K, ldx, xq, x_scale, eps);
    if (s != FP8Q_OK || M == 0) return s;
    unsigned *status = device_status_ptr();
    if (status == nullptr) return FP8Q_ERR_CUDA;
    bool early_trigger = false;
    const cudaError_t e =
        launch_quant_per_token(x, M, K, ldx, xq, x_scale, eps, status, as_stream(stream), &early_trigger);
    if (e == cudaSuccess)
        note_launch_writes(as_stream(stream), xq, static_cast<size_t>(M) * K, x_scale, static_cast<size_t>(M) * 4,
                           nullptr, 0, early_trigger);
    return from_cuda(e);
}

fp8q_status fp8q_quant_per_token_group_row_padded(const void *x, int64_t M, int64_t K, int64_t ldx,
                                                  int32_t group_size, float eps, int32_t row_alignment, void *xq,
                                                  float *x_scale, int64_t m_pad, void *stream)
{
    if (group_size != 16 && group_size != 32 && group_size != 64 && group_size != 128) {
        if (group_size <= 0) return FP8Q_ERR_INVALID_ARG;
        return FP8Q_ERR_UNSUPPORTED;
    }
    if (row_alignment <= 0 || m_pad < M || m_pad % row_alignment != 0 || m_pad > kMaxDim)
        return FP8Q_ERR_INVALID_ARG;
    if (K > 0 && K % group_size != 0) return FP8Q_ERR_INVALID_ARG;
    const fp8q_status s = check_quant_common(x, M, K, ldx, xq, x_scale, eps);
    if (s != FP8Q_OK || M == 0) return s;
    bool early_trigger = false;
    const cudaError_t e = launch_quant_group(x, M, K, ldx, group_size, xq, x_scale, m_pad, eps, current_device_sms(),
                                             as_stream(stream), false, false, &early_trigger);
    if (e == cudaSuccess)
        note_launch_writes(as_stream(stream), xq, static_cast<size_t>(M) * K, x_scale,
                           static_cast<size_t>(K / group_size) * m_pad * 4, nullptr, 0, early_trigger);
    return from_cuda(e);
}

fp8q_status fp8q_quant_per_token_group_row_padded_ex(const void *x, int64_t M, int64_t K, int64_t ldx,
                                                     int32_t group_size, float eps, int32_t row_alignment,
                                                     int32_t flags, void *xq, float *x_scale, int64_t m_pad,
                                                     void *stream)
{
    if ((flags & ~(FP8Q_QUANT_SCALE_UE8M0 | FP8Q_QUANT_SILU_AND_MUL)) != 0) return FP8Q_ERR_INVALID_ARG;
    const bool silu = (flags & FP8Q_QUANT_SILU_AND_MUL) != 0;
    if (group_size != 16 && group_size != 32 && group_size != 64 && group_size != 128) {
        if (group_size <= 0) return FP8Q_ERR_INVALID_ARG;
        return FP8Q_ERR_UNSUPPORTED;
    }
    if (row_alignment <= 0 || m_pad < M || m_pad % row_alignment != 0 || m_pad > kMaxDim)
        return FP8Q_ERR_INVALID_ARG;
    if (K > 0 && K % group_size != 0) return FP8Q_ERR_INVALID_ARG;
    // The fused input row holds 2K values (gate, then up).
    if (silu && (K > kMaxDim / 2 || ldx < 2 * K)) return FP8Q_ERR_INVALID_ARG;
    const fp8q_status s = check_quant_common(x, M, K, ldx, xq, x_scale, eps);
    if (s != FP8Q_OK || M == 0) return s;
    bool early_trigger = false;
    const cudaError_t e = launch_quant_group(x, M, K, ldx, group_size, xq, x_scale, m_pad, eps, current_device_sms(),
                                             as_stream(stream), (flags & FP8Q_QUANT_SCALE_UE8M0) != 0, silu,
                                             &early_trigger);
    if (e == cudaSuccess)
        note_launch_writes(as_stream(stream), xq, static_cast<size_t>(M) * K, x_scale,
                           static_cast<size_t>(K / group_size) * m_pad * 4, nullptr, 0, early_trigger);
    return from_cuda(e);
}

fp8q_status fp8q_quant_static_per_tensor(const void *x, int64_t M, int64_t K, int64_t ldx, const float *scale,
                                         void *xq, float *x_scale_rep, void *stream)
{
    if (M < 0 || K <= 0 || M > kMaxDim || K > kMaxDim) return FP8Q_ERR_INVALID_ARG;
    if (K % 16 != 0 || ldx < K || ldx % 8 != 0) return FP8Q_ERR_INVALID_ARG;
    if (M == 0) return FP8Q_OK;
    if (x == nullptr || xq == nullptr || scale == nullptr) return FP8Q_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(xq) || !aligned4(scale) || !aligned4(x_scale_rep))
        return FP8Q_ERR_INVALID_ARG;
    const cudaError_t e = launch_quant_static(x, M, K, ldx, scale, xq, x_scale_rep, current_device_sms(),
                                              as_stream(stream));
    if (e == cudaSuccess)
        note_launch_writes(as_stream(stream), xq, static_cast<size_t>(M) * K, x_scale_rep,
                           static_cast<size_t>(M) * 4);
    return from_cuda(e);
}

fp8q_status fp8q_quant_weight_block128(const void *w, int64_t N, int64_t K, void *wq, float *w_scale, float eps,
                                       void *stream)
{
    if (N <= 0 || K <= 0 || N > kMaxDim || K > kMaxDim) return FP8Q_ERR_INVALID_ARG;
    if (N % 128 != 0 || K % 128 != 0) return FP8Q_ERR_UNSUPPORTED;
    if (!(eps > 0.0f) || !isfinite(eps)) return FP8Q_ERR_INVALID_ARG;
    if (w == nullptr || wq == nullptr || w_scale == nullptr) return FP8Q_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(wq) || !aligned4(w_scale)) return FP8Q_ERR_INVALID_ARG;
    const cudaError_t e = launch_quant_weight_block128(w, N, K, wq, w_scale, eps, as_stream(stream));
    if (e == cudaSuccess)
        note_launch_writes(as_stream(stream), wq, static_cast<size_t>(N) * K, w_scale,
                           static_cast<size_t>(N / 128) * (K / 128) * 4);
    return from_cuda(e);
}

fp8q_status fp8q_scaled_mm_channelwise(const void *a, const void *b, int64_t ldb, const float *a_scale,
                                       const float *b_scale, const void *bias, void *out, int64_t M, int64_t N,
                                       int64_t K, fp8q_out_dtype out_dtype, void *workspace, size_t workspace_bytes,
                                       void *stream)
{
    if (workspace != nullptr && !aligned16(workspace)) return FP8Q_ERR_INVALID_ARG;
    if (M < 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return FP8Q_ERR_INVALID_ARG;
    if (out_dtype != FP8Q_OUT_BF16 && out_dtype != FP8Q_OUT_FP16) return FP8Q_ERR_UNSUPPORTED;
    if (K % 16 != 0 || ldb < K || ldb % 16 != 0 || N % 8 != 0) return FP8Q_ERR_INVALID_ARG;
    if (M == 0) return FP8Q_OK;
    if (a == nullptr || b == nullptr || a_scale == nullptr || b_scale == nullptr || out == nullptr)
        return FP8Q_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(b) || !aligned16(out) || !aligned4(a_scale) || !aligned4(b_scale))
        return FP8Q_ERR_INVALID_ARG;
    if (bias != nullptr && (reinterpret_cast<uintptr_t>(bias) & 1u)) return FP8Q_ERR_INVALID_ARG;
    GemmProblem p;
    p.M = M; p.N = N; p.K = K; p.m_pad = M;
    p.a = a; p.lda = K; p.w = b; p.ldw = ldb;
    p.a_scale = a_scale; p.w_scale = b_scale; p.bias = bias; p.out = out;
    p.out_fp16 = out_dtype == FP8Q_OUT_FP16;
    p.blockwise = false;
    p.preload = false;
    p.fused_quant = false;
    p.w16 = false;
    p.eps = 0.0f;
    p.ws = workspace;
    p.ws_bytes = workspace_bytes;
    return run_gemm(p, as_stream(stream));
}

fp8q_status fp8q_scaled_mm_blockwise(const void *a, const void *w, const float *a_scale, const float *w_scale,
                                     const void *bias, void *out, int64_t M, int64_t m_pad, int64_t N, int64_t K,
                                     fp8q_out_dtype out_dtype, void *workspace, size_t workspace_bytes,
                                     void *stream)
{
    if (workspace != nullptr && !aligned16(workspace)) return FP8Q_ERR_INVALID_ARG;
    if (M < 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return FP8Q_ERR_INVALID_ARG;
    if (out_dtype != FP8Q_OUT_BF16 && out_dtype != FP8Q_OUT_FP16) return FP8Q_ERR_UNSUPPORTED;
    if (N % 128 != 0 || K % 128 != 0) return FP8Q_ERR_UNSUPPORTED;
    if (m_pad < M || m_pad % 4 != 0 || m_pad > kMaxDim) return FP8Q_ERR_INVALID_ARG;
    if (M == 0) return FP8Q_OK;
    if (a == nullptr || w == nullptr || a_scale == nullptr || w_scale == nullptr || out == nullptr)
        return FP8Q_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(w) || !aligned16(out) || !aligned16(a_scale) || !aligned4(w_scale))
        return FP8Q_ERR_INVALID_ARG;
    if (bias != nullptr && (reinterpret_cast<uintptr_t>(bias) & 1u)) return FP8Q_ERR_INVALID_ARG;
    GemmProblem p;
    p.M = M; p.N = N; p.K = K; p.m_pad = m_pad;
    p.a = a; p.lda = K; p.w = w; p.ldw = K;
    p.a_scale = a_scale; p.w_scale = w_scale; p.bias = bias; p.out = out;
    p.out_fp16 = out_dtype == FP8Q_OUT_FP16;
    p.blockwise = true;
    p.preload = false;
    p.fused_quant = false;
    p.w16 = false;
    p.eps = 0.0f;
    p.ws = workspace;
    p.ws_bytes = workspace_bytes;
    return run_gemm(p, as_stream(stream));
}

fp8q_status fp8q_linear_channelwise(const void *x, const void *b, int64_t ldb, const float *b_scale, const void *bias,
                                    void *out, int64_t M, int64_t N, int64_t K, void *xq, float *xs,
                                    fp8q_out_dtype out_dtype, void *workspace, size_t workspace_bytes, void *stream)
{
    if (workspace != nullptr && !aligned16(workspace)) return FP8Q_ERR_INVALID_ARG;
    // Validate the GEMM's arguments before enqueueing the quantizer so that
    // an error leaves nothing enqueued.
    if (M < 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return FP8Q_ERR_INVALID_ARG;
    if (out_dtype != FP8Q_OUT_BF16 && out_dtype != FP8Q_OUT_FP16) return FP8Q_ERR_UNSUPPORTED;
    if (ldb < K || ldb % 16 != 0 || N % 8 != 0) return FP8Q_ERR_INVALID_ARG;
    fp8q_status s = check_quant_common(x, M, K, K, xq, xs, 1e-10f);
    if (s != FP8Q_OK || M == 0) return s;
    if (b == nullptr || b_scale == nullptr || out == nullptr || !aligned16(b) || !aligned16(out) || !aligned4(b_scale))
        return FP8Q_ERR_INVALID_ARG;
    if (bias != nullptr && (reinterpret_cast<uintptr_t>(bias) & 1u)) return FP8Q_ERR_INVALID_ARG;
    // A few tokens: one launch, the quantization fused into matrix-vector
    // products (unless a schedule override asks for the GEMM).
    if (linear_gemv_fits(M, N, K) && !plan_override_active()) {
        return from_cuda(launch_linear_pt_gemv(x, b, ldb, b_scale, bias, out, xq, xs, M, N, K, 1e-10f,
                                               out_dtype == FP8Q_OUT_FP16, as_stream(stream)));
    }
    s = fp8q_quant_per_token(x, M, K, K, xq, xs, 1e-10f, stream);
    if (s != FP8Q_OK) return s;
    return fp8q_scaled_mm_channelwise(xq, b, ldb, xs, b_scale, bias, out, M, N, K, out_dtype, workspace,
                                      workspace_bytes, stream);
}

int32_t fp8q_linear_channelwise_launches(int64_t M, int64_t N, int64_t K)
{
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    return linear_gemv_fits(M, N, K) && !plan_override_active() ? 1 : 2;
}

int32_t fp8q_linear_blockwise_launches(int64_t M, int64_t K)
{
    if (M <= 0 || K <= 0) return 0;
    return linear_blk_gemv_fits(M, K) && !plan_override_active() ? 1 : 2;
}

fp8q_status fp8q_linear_blockwise(const void *x, const void *w, const float *w_scale, const void *bias, void *out,
                                  int64_t M, int64_t N, int64_t K, void *xq, float *xs, int64_t m_pad,
                                  fp8q_out_dtype out_dtype, void *workspace, size_t workspace_bytes, void *stream)
{
    if (workspace != nullptr && !aligned16(workspace)) return FP8Q_ERR_INVALID_ARG;
    if (M < 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return FP8Q_ERR_INVALID_ARG;
    if (out_dtype != FP8Q_OUT_BF16 && out_dtype != FP8Q_OUT_FP16) return FP8Q_ERR_UNSUPPORTED;
    if (N % 128 != 0 || K % 128 != 0) return FP8Q_ERR_UNSUPPORTED;
    if (m_pad < M || m_pad % 4 != 0 || m_pad > kMaxDim) return FP8Q_ERR_INVALID_ARG;
    fp8q_status s = check_quant_common(x, M, K, K, xq, xs, 1e-10f);
    if (s != FP8Q_OK || M == 0) return s;
    if (w == nullptr || w_scale == nullptr || out == nullptr || !aligned16(w) || !aligned16(out) ||
        !aligned16(xs) || !aligned4(w_scale))
        return FP8Q_ERR_INVALID_ARG;
    if (bias != nullptr && (reinterpret_cast<uintptr_t>(bias) & 1u)) return FP8Q_ERR_INVALID_ARG;
    // One token: one launch, the group quantization fused into a
    // matrix-vector product (unless a schedule override asks for the GEMM).
    if (linear_blk_gemv_fits(M, K) && !plan_override_active())
        return from_cuda(launch_linear_blk_gemv(x, w, w_scale, bias, out, xq, xs, m_pad, N, K, 1e-10f,
                                                out_dtype == FP8Q_OUT_FP16, as_stream(stream)));
    s = fp8q_quant_per_token_group_row_padded(x, M, K, K, 128, 1e-10f, 4, xq, xs, m_pad, stream);
    if (s != FP8Q_OK) return s;
    return fp8q_scaled_mm_blockwise(xq, w, xs, w_scale, bias, out, M, m_pad, N, K, out_dtype, workspace,
                                    workspace_bytes, stream);
}

fp8q_status fp8q_linear_blockwise_fused(const void *x, int64_t ldx, const void *w, const float *w_scale,
                                        const void *bias, void *out, int64_t M, int64_t N, int64_t K,
                                        fp8q_out_dtype out_dtype, void *stream)
{
    if (M < 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return FP8Q_ERR_INVALID_ARG;
    if (out_dtype != FP8Q_OUT_BF16 && out_dtype != FP8Q_OUT_FP16) return FP8Q_ERR_UNSUPPORTED;
    if (N % 128 != 0 || K % 128 != 0) return FP8Q_ERR_UNSUPPORTED;
    if (ldx < K || ldx % 8 != 0 || ldx > kMaxDim) return FP8Q_ERR_INVALID_ARG;
    if (M == 0) return FP8Q_OK;
    if (x == nullptr || w == nullptr || w_scale == nullptr || out == nullptr) return FP8Q_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(out) || !aligned4(w_scale)) return FP8Q_ERR_INVALID_ARG;
    if (bias != nullptr && (reinterpret_cast<uintptr_t>(bias) & 1u)) return FP8Q_ERR_INVALID_ARG;
    fp8q_plan pl;
    const fp8q_status s = fp8q_gemm_plan(M, N, K, 1, 0, &pl);
    if (s != FP8Q_OK) return s;
    if (!pl.swap_ab || (pl.mma_n != 16 && pl.mma_n != 32)) return FP8Q_ERR_UNSUPPORTED;
    GemmProblem p;
    p.M = M; p.N = N; p.K = K; p.m_pad = M;
    p.a = x; p.lda = ldx; p.w = w; p.ldw = K;
    p.a_scale = nullptr; p.w_scale = w_scale; p.bias = bias; p.out = out;
    p.out_fp16 = out_dtype == FP8Q_OUT_FP16;
    p.blockwise = true;
    p.preload = false;
    p.fused_quant = true;
    p.w16 = false;
    p.eps = 1e-10f;
    p.ws = nullptr;
    p.ws_bytes = 0;
    return run_gemm(p, as_stream(stream));
}

fp8q_status fp8q_scaled_mm_w8a16(const void *x, int64_t ldx, const void *w, int64_t ldw, const float *w_scale,
                                 const void *bias, void *out, int64_t M, int64_t N, int64_t K,
                                 fp8q_out_dtype out_dtype, void *stream)
{
    if (M < 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return FP8Q_ERR_INVALID_ARG;
    if (out_dtype != FP8Q_OUT_BF16 && out_dtype != FP8Q_OUT_FP16) return FP8Q_ERR_UNSUPPORTED;
    if (K % 16 != 0 || ldx < K || ldx % 8 != 0 || ldw < K || ldw % 16 != 0 || N % 8 != 0)
        return FP8Q_ERR_INVALID_ARG;
    if (M == 0) return FP8Q_OK;
    if (x == nullptr || w == nullptr || w_scale == nullptr || out == nullptr) return FP8Q_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(out) || !aligned4(w_scale)) return FP8Q_ERR_INVALID_ARG;
    if (bias != nullptr && (reinterpret_cast<uintptr_t>(bias) & 1u)) return FP8Q_ERR_INVALID_ARG;
    // A few tokens: matrix-vector products on the CUDA cores.
    if (M <= kW16GemvMaxM)
        return from_cuda(launch_w8a16_gemv(x, ldx, w, ldw, w_scale, bias, out, M, N, K,
                                           out_dtype == FP8Q_OUT_FP16, as_stream(stream)));
    const int num_sms = current_device_sms();
    if (num_sms <= 0) return FP8Q_ERR_CUDA;
    // Schedule: 128 weight rows x 16 (M <= 16) or 32 tokens per tile; K split
    // across a cluster of 2, 4 or 8 while the tiles cannot fill the GPU.
    fp8q_plan pl = {};
    pl.swap_ab = 1;
    pl.mma_n = M <= 16 ? 16 : 32;
    const int64_t tiles = ((M + pl.mma_n - 1) / pl.mma_n) * ((N + 127) / 128);
    int split = 1;
    while (split < 8 && tiles * split * 2 <= num_sms) split *= 2;
    pl.split_k = split;
    plan_finish(M, N, K, 0, num_sms, &pl);
    GemmProblem p;
    p.M = M; p.N = N; p.K = K; p.m_pad = M;
    p.a = x; p.lda = ldx; p.w = w; p.ldw = ldw;
    p.a_scale = nullptr; p.w_scale = w_scale; p.bias = bias; p.out = out;
    p.out_fp16 = out_dtype == FP8Q_OUT_FP16;
    p.blockwise = false;
    p.preload = false;
    p.fused_quant = false;
    p.w16 = true;
    p.eps = 0.0f;
    p.ws = nullptr;
    p.ws_bytes = 0;
    return launch_planned(p, pl, as_stream(stream));
}

fp8q_status fp8q_device_status(void *stream, int32_t reset)
{
    unsigned v = 0;
    if (read_status_word(&v, reset != 0, as_stream(stream)) != cudaSuccess) return FP8Q_ERR_CUDA;
    if (v & 4u) return FP8Q_ERR_TIMEOUT;
    return v == 0 ? FP8Q_OK : FP8Q_ERR_CUDA;
}

fp8q_status fp8q_last_device_status(void *stream) { return fp8q_device_status(stream, 0); }

const char *fp8q_status_str(fp8q_status status)
{
    switch (status) {
        case FP8Q_OK: return "FP8Q_OK";
        case FP8Q_ERR_INVALID_ARG: return "FP8Q_ERR_INVALID_ARG";
        case FP8Q_ERR_UNSUPPORTED: return "FP8Q_ERR_UNSUPPORTED";
        case FP8Q_ERR_CUDA: return "FP8Q_ERR_CUDA";
        case FP8Q_ERR_TIMEOUT: return "FP8Q_ERR_TIMEOUT";
        default: return "FP8Q_UNKNOWN_STATUS";
    }
}

int32_t fp8q_version(void) { return (2 << 16) | 2; }

}  // extern "C"
