// linear_gemv.cu -- the channelwise W8A8 linear layer for one token in ONE
// launch on the CUDA cores: the per-token quantization of x fused into the
// matrix-vector product with the E4M3 weights.
//   s[m]     = max(amax_k |x[m,k]|, eps) / 448
//   q[m,k]   = e4m3(x[m,k] / s[m])                       (per-token quantization)
//   out[m,n] = round(sum_k dec(q[m,k]) * dec(w[n,k]) * s[m] * w_scale[n] + bias[n])
// -- the per-token activation x per-channel weight path of the "Tune FP8
// GEMM Triton tiles on L40S and enable by default" page (key source
// snippets: apply_fp8_linear, whose channelwise branch quantizes x per token
// and calls fp8_scaled_mm), with the quantization inside the GEMM launch, as
// the "Remove per-call padding overhead of the FP8 blockwise GEMM" page
// (implementation breakdown) allows it to be fused.
//
// With one token the GEMM is a matrix-vector product, bound by the weight
// stream; a tensor-core GEMM behind a separate quantizer launch pays two
// launches' fixed costs for it.  Here a persistent grid (as many CTAs as
// fit, each owning every gridDim-th group of ROWS output channels,
// gemv_common.cuh's CTA shape) first quantizes x itself: every CTA reduces
// the amax of each token row (the rows are a few KB, read from L2),
// quantizes the row and keeps the decoded codes in shared memory as bf16
// (E4M3 values are exact in bf16).  The weights of its row groups then
// stream past these activations: decoded to fp32 in registers (exact), the
// exact products code x code accumulated with packed fp32 FMAs.  The codes
// are those of the per-token quantizer bit for bit (the same amax, scale and
// quotient arithmetic, quant_common.cuh); CTA 0 also stores them and the
// scales into the caller's xq / xs, as the two-kernel composition leaves
// them.  The sum is scaled as the GEMM's epilogue does:
// fmaf(sum * s[m], w_scale[n], bias[n]), rounded once.
//
// Unless a library kernel that may still be running writes the weights,
// each warp issues its first group's weight loads before the dependency
// wait; after each row group it issues the next group's loads before the
// cross-warp reduction.
//
// The blockwise linear for one token (linear_blk_gemv_kernel) is the same
// kernel with the blockwise scheme's arithmetic ("Remove per-call padding
// overhead of the FP8 blockwise GEMM" page, key source snippets): the row is
// quantized in groups of 128 (the 8 lanes of a group reduce its amax; the
// group quantizer's codes and scales bit for bit, CTA 0 storing them in the
// row-padded layout), and each lane's 16 exact products are summed and then
// scaled by the group scale times the weight block's scale (the CTA's 8 or
// 4 output channels lie in one 128-row block) before they are accumulated;
// out = round(sum + bias[n]).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "device_common.cuh"
#include "gemv_common.cuh"
#include "internal.h"
#include "quant_common.cuh"

namespace fp8q {
namespace {

using gemv::kChunk;
using gemv::kWarps;

// NCW: chunks per warp and group (ceil(K / 4096)); a warp requests all of
// them at once.  Registers: NCW * ROWS * 4 for the weights, so the CTAs per
// SM fall from 3 to 2 to 1 as NCW grows.
// Output channels per CTA: 8, or 4 with three chunks per warp (12 uint4
// registers per row), which keeps two CTAs per SM there.
constexpr int gemv_rows_for(int ncw) { return ncw >= 3 ? 4 : 8; }
constexpr int min_ctas(int ncw) { return ncw == 1 ? 3 : 2; }

// All NCW chunks of a group for this warp (zeros past K).
template <int NCW, int ROWS>
__device__ __forceinline__ void load_group(const uint8_t *__restrict__ w, int64_t ldw, int n0, int N, int K, int warp,
                                           int lane, uint4 (&wv)[NCW][ROWS])
{
#pragma unroll
    for (int i = 0; i < NCW; ++i) gemv::load_weights<ROWS>(w, ldw, n0, N, K, warp + i * kWarps, lane, wv[i]);
}

template <int MT, int NCW, typename OutT, int ROWS = gemv_rows_for(NCW)>
__global__ void __launch_bounds__(32 * kWarps, min_ctas(NCW)) linear_pt_gemv_kernel(
    const __nv_bfloat16 *__restrict__ x, const uint8_t *__restrict__ w, int64_t ldw,
    const float *__restrict__ w_scale, const __nv_bfloat16 *__restrict__ bias, OutT *__restrict__ out,
    uint8_t *__restrict__ xq, float *__restrict__ xs, int M, int N, int K, float eps, int preload)
{
    extern __shared__ __align__(16) uint8_t xdec_raw[];   // [MT][K] bf16: the decoded codes
    __shared__ float red[2][kWarps][ROWS][MT];
    __shared__ float amax_warp[kWarps][MT];
    __shared__ float scale_sh[MT], rcp_sh[MT];
    __nv_bfloat16 *xdec = reinterpret_cast<__nv_bfloat16 *>(xdec_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int groups = (N + ROWS - 1) / ROWS;
    constexpr int kStride = 32 * kWarps * 16;   // the CTA's 16-value pieces cover kStride of K per pass

    uint4 wv[NCW][ROWS];
    int g = blockIdx.x;
    if (preload && g < groups) load_group<NCW, ROWS>(w, ldw, g * ROWS, N, K, warp, lane, wv);
    pdl_wait();
    pdl_trigger();
    if (!preload && g < groups) load_group<NCW, ROWS>(w, ldw, g * ROWS, N, K, warp, lane, wv);

    // Per-token scales: the amax of each thread's 16-value pieces k =
    // 16 * thread + kStride * j, then over lanes, then over warps.
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        float am = 0.0f;
        if (m < M)
            for (int k = threadIdx.x * 16; k < K; k += kStride)
                am = chunk_amax(load_chunk(x + static_cast<int64_t>(m) * K + k), am);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
        if (lane == 0) amax_warp[warp][m] = am;
    }
    __syncthreads();
    if (threadIdx.x < MT) {
        const int m = threadIdx.x;
        float a = amax_warp[0][m];
#pragma unroll
        for (int q = 1; q < kWarps; ++q) a = fmaxf(a, amax_warp[q][m]);
        const float sc = scale_of(a, eps);
        scale_sh[m] = sc;
        rcp_sh[m] = scale_has_reciprocal(sc) ? 1.0f / sc : 0.0f;
        if (blockIdx.x == 0 && m < M) xs[m] = sc;
    }
    __syncthreads();
    // The codes of the same pieces, decoded into shared memory (tokens past
    // M: zeros).  A decoded E4M3 value has at most 4 significant bits, so
    // its fp32 pattern's upper half is its exact bf16.
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const float sc = scale_sh[m], rc = rcp_sh[m];
        const bool recip = scale_has_reciprocal(sc);
        for (int k = threadIdx.x * 16; k < K; k += kStride) {
            uint4 q = make_uint4(0u, 0u, 0u, 0u);
            if (m < M) {
                const Chunk16 v = load_chunk(x + static_cast<int64_t>(m) * K + k);
                const uint2 lo = quant_unit8(v.lo, sc, rc, recip);
                const uint2 hi = quant_unit8(v.hi, sc, rc, recip);
                q = make_uint4(lo.x, lo.y, hi.x, hi.y);
                if (blockIdx.x == 0) *reinterpret_cast<uint4 *>(xq + static_cast<int64_t>(m) * K + k) = q;
            }
            const uint32_t words[4] = {q.x, q.y, q.z, q.w};
            uint32_t d[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float2 f = gemv::e4m3x2_to_f32x2(words[j >> 1] >> (16 * (j & 1)));
                d[j] = __byte_perm(__float_as_uint(f.x), __float_as_uint(f.y), 0x7632);
            }
            uint4 *dst = reinterpret_cast<uint4 *>(xdec + static_cast<int64_t>(m) * K + k);
            dst[0] = make_uint4(d[0], d[1], d[2], d[3]);
            dst[1] = make_uint4(d[4], d[5], d[6], d[7]);
        }
    }
    __syncthreads();

    for (int buf = 0; g < groups; g += gridDim.x, buf ^= 1) {
        const int n0 = g * ROWS;
        float2 acc[ROWS][MT];   // even and odd k of each (row, token)
#pragma unroll
        for (int r = 0; r < ROWS; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) acc[r][m] = make_float2(0.0f, 0.0f);
        // This warp's chunks c = warp + 8 i of the group are already in wv.
#pragma unroll
        for (int i = 0; i < NCW; ++i) {
            const int k = (warp + i * kWarps) * kChunk + lane * 16;
            if (k < K) {
                float2 xa[MT][8];
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(xdec + static_cast<int64_t>(m) * K + k);
                    const uint4 lo = src[0], hi = src[1];
                    const uint32_t words[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        xa[m][j] = make_float2(__uint_as_float(words[j] << 16), __uint_as_float(words[j] & 0xFFFF0000u));
                }
                gemv::fma_piece<ROWS, MT>(wv[i], xa, acc);
            }
        }
        // The next group's chunks, in flight during the reduction.
        const int gn = g + static_cast<int>(gridDim.x);
        if (gn < groups) load_group<NCW, ROWS>(w, ldw, gn * ROWS, N, K, warp, lane, wv);
        const float sum = gemv::reduce_cta<ROWS, MT>(acc, red[buf], warp, lane);
        if (threadIdx.x < ROWS * MT) {
            const int r = threadIdx.x / MT, m = threadIdx.x % MT;
            const int n = n0 + r;
            if (n < N && m < M) {
                const float b = bias != nullptr ? __bfloat162float(bias[n]) : 0.0f;
                out[static_cast<int64_t>(m) * N + n] =
                    gemv::to_out<OutT>(fmaf(sum * scale_sh[m], __ldg(w_scale + n), b));
            }
        }
    }
}

template <int NCW, typename OutT, int ROWS = gemv_rows_for(NCW)>
__global__ void __launch_bounds__(32 * kWarps, min_ctas(NCW)) linear_blk_gemv_kernel(
    const __nv_bfloat16 *__restrict__ x, const uint8_t *__restrict__ w, const float *__restrict__ w_scale,
    const __nv_bfloat16 *__restrict__ bias, OutT *__restrict__ out, uint8_t *__restrict__ xq,
    float *__restrict__ xs, int64_t m_pad, int N, int K, float eps, int preload)
{
    extern __shared__ __align__(16) uint8_t blk_dyn[];   // bf16 [K] decoded codes, then fp32 [K/128] scales
    __shared__ float red[2][kWarps][ROWS][1];
    __nv_bfloat16 *xdec = reinterpret_cast<__nv_bfloat16 *>(blk_dyn);
    float *sgrp = reinterpret_cast<float *>(blk_dyn + static_cast<size_t>(K) * 2);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int groups = (N + ROWS - 1) / ROWS;
    const int kblocks = K >> 7;
    constexpr int kStride = 32 * kWarps * 16;

    uint4 wv[NCW][ROWS];
    int g = blockIdx.x;
    if (preload && g < groups) load_group<NCW, ROWS>(w, K, g * ROWS, N, K, warp, lane, wv);
    pdl_wait();
    pdl_trigger();
    if (!preload && g < groups) load_group<NCW, ROWS>(w, K, g * ROWS, N, K, warp, lane, wv);

    // Group scales and codes.  A warp's pieces k = k0 + 16 * lane cover 512
    // values; the loop bound is the warp's (K is a multiple of 128, so a
    // group is either wholly inside or wholly past K).
    for (int k0 = warp * kChunk; k0 < K; k0 += kStride) {
        const int k = k0 + lane * 16;
        const bool in = k < K;
        Chunk16 v;
        float am = 0.0f;
        if (in) {
            v = load_chunk(x + k);
            am = chunk_amax(v, 0.0f);
        }
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
        if (in) {
            const float sc = scale_of(am, eps);
            const uint4 q = quant_chunk(v, sc);
            if ((lane & 7) == 0) sgrp[k >> 7] = sc;
            if (xq != nullptr && blockIdx.x == 0) {
                *reinterpret_cast<uint4 *>(xq + k) = q;
                if ((lane & 7) == 0) xs[static_cast<int64_t>(k >> 7) * m_pad] = sc;
            }
            const uint32_t words[4] = {q.x, q.y, q.z, q.w};
            uint32_t d[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float2 f = gemv::e4m3x2_to_f32x2(words[j >> 1] >> (16 * (j & 1)));
                d[j] = __byte_perm(__float_as_uint(f.x), __float_as_uint(f.y), 0x7632);
            }
            uint4 *dst = reinterpret_cast<uint4 *>(xdec + k);
            dst[0] = make_uint4(d[0], d[1], d[2], d[3]);
            dst[1] = make_uint4(d[4], d[5], d[6], d[7]);
        }
    }
    __syncthreads();

    for (int buf = 0; g < groups; g += gridDim.x, buf ^= 1) {
        const int n0 = g * ROWS;
        const float *ws_row = w_scale + static_cast<int64_t>(n0 >> 7) * kblocks;
        float2 acc[ROWS][1];   // the scaled sum in .x (.y stays 0)
#pragma unroll
        for (int r = 0; r < ROWS; ++r) acc[r][0] = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int i = 0; i < NCW; ++i) {
            const int k = (warp + i * kWarps) * kChunk + lane * 16;
            if (k < K) {
                float2 xa[1][8];
                const uint4 *src = reinterpret_cast<const uint4 *>(xdec + k);
                const uint4 lo = src[0], hi = src[1];
                const uint32_t words[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    xa[0][j] = make_float2(__uint_as_float(words[j] << 16), __uint_as_float(words[j] & 0xFFFF0000u));
                float2 t[ROWS][1];
#pragma unroll
                for (int r = 0; r < ROWS; ++r) t[r][0] = make_float2(0.0f, 0.0f);
                gemv::fma_piece<ROWS, 1>(wv[i], xa, t);
                const float f = sgrp[k >> 7] * __ldg(ws_row + (k >> 7));
#pragma unroll
                for (int r = 0; r < ROWS; ++r) acc[r][0].x = fmaf(t[r][0].x + t[r][0].y, f, acc[r][0].x);
            }
        }
        const int gn = g + static_cast<int>(gridDim.x);
        if (gn < groups) load_group<NCW, ROWS>(w, K, gn * ROWS, N, K, warp, lane, wv);
        const float sum = gemv::reduce_cta<ROWS, 1>(acc, red[buf], warp, lane);
        if (threadIdx.x < ROWS) {
            const int n = n0 + threadIdx.x;
            if (n < N) {
                const float b = bias != nullptr ? __bfloat162float(bias[n]) : 0.0f;
                out[n] = gemv::to_out<OutT>(sum + b);
            }
        }
    }
}

// Every CTA that fits: per_sm (from the occupancy of `kernel` with `smem`)
// times the SMs, at most one per group.
template <typename Kernel>
cudaError_t persistent_grid(Kernel kernel, size_t smem, int groups, int *grid)
{
    int per_sm = 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 32 * kWarps, smem);
    if (e != cudaSuccess) return e;
    const int sms = current_device_sms();
    if (per_sm <= 0 || sms <= 0) return cudaErrorInvalidConfiguration;
    *grid = groups < per_sm * sms ? groups : per_sm * sms;
    return cudaSuccess;
}

template <int NCW, typename OutT>
cudaError_t launch_blk(const void *x, const void *w, const float *w_scale, const void *bias, void *out, void *xq,
                       float *xs, int64_t m_pad, int N, int K, float eps, bool preload, cudaStream_t st)
{
    auto kernel = linear_blk_gemv_kernel<NCW, OutT>;
    const size_t smem = static_cast<size_t>(K) * 2u + static_cast<size_t>(K / 128) * 4u;
    if (smem > 48u * 1024u) return cudaErrorInvalidValue;
    int grid = 0;
    constexpr int kRows = gemv_rows_for(NCW);
    cudaError_t e = persistent_grid(kernel, smem, (N + kRows - 1) / kRows, &grid);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(32 * kWarps);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<const __nv_bfloat16 *>(x), static_cast<const uint8_t *>(w),
                              w_scale, static_cast<const __nv_bfloat16 *>(bias), static_cast<OutT *>(out),
                              static_cast<uint8_t *>(xq), xs, m_pad, N, K, eps, preload ? 1 : 0);
}

template <int MT, int NCW, typename OutT>
cudaError_t launch_t(const void *x, const void *w, int64_t ldw, const float *w_scale, const void *bias, void *out,
                     void *xq, float *xs, int M, int N, int K, float eps, bool preload, cudaStream_t st)
{
    auto kernel = linear_pt_gemv_kernel<MT, NCW, OutT>;
    const size_t smem = static_cast<size_t>(MT) * static_cast<size_t>(K) * 2u;   // at most 48 KB (no opt-in)
    if (smem > 48u * 1024u) return cudaErrorInvalidValue;
    // Every CTA that fits (fewer CTAs with whole rounds of groups each
    // measured slower: the rounds are latency-bound).
    constexpr int kRows = gemv_rows_for(NCW);
    int grid = 0;
    cudaError_t e = persistent_grid(kernel, smem, (N + kRows - 1) / kRows, &grid);
    if (e != cudaSuccess) return e;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(32 * kWarps);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<const __nv_bfloat16 *>(x), static_cast<const uint8_t *>(w),
                              ldw, w_scale, static_cast<const __nv_bfloat16 *>(bias), static_cast<OutT *>(out),
                              static_cast<uint8_t *>(xq), xs, M, N, K, eps, preload ? 1 : 0);
}

}  // namespace

cudaError_t launch_linear_pt_gemv(const void *x, const void *w, int64_t ldw, const float *w_scale, const void *bias,
                                  void *out, void *xq, float *xs, int64_t M, int64_t N, int64_t K, float eps,
                                  bool out_fp16, cudaStream_t st)
{
    if (!linear_gemv_fits(M, N, K)) return cudaErrorInvalidValue;
    const size_t wbytes = static_cast<size_t>(N - 1) * static_cast<size_t>(ldw) + static_cast<size_t>(K);
    const bool preload = !last_launch_writes_overlap(st, w, wbytes);
    const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
    cudaError_t e;
    switch (gemv_chunks_per_warp(K)) {
        case 1:
            e = out_fp16 ? launch_t<1, 1, __half>(x, w, ldw, w_scale, bias, out, xq, xs, m, n, k, eps, preload, st)
                         : launch_t<1, 1, __nv_bfloat16>(x, w, ldw, w_scale, bias, out, xq, xs, m, n, k, eps,
                                                         preload, st);
            break;
        case 2:
            e = out_fp16 ? launch_t<1, 2, __half>(x, w, ldw, w_scale, bias, out, xq, xs, m, n, k, eps, preload, st)
                         : launch_t<1, 2, __nv_bfloat16>(x, w, ldw, w_scale, bias, out, xq, xs, m, n, k, eps,
                                                         preload, st);
            break;
        default:
            e = out_fp16 ? launch_t<1, 3, __half>(x, w, ldw, w_scale, bias, out, xq, xs, m, n, k, eps, preload, st)
                         : launch_t<1, 3, __nv_bfloat16>(x, w, ldw, w_scale, bias, out, xq, xs, m, n, k, eps,
                                                         preload, st);
    }
    if (e == cudaSuccess)
        note_launch_writes(st, out, static_cast<size_t>(M) * N * 2, xq, static_cast<size_t>(M) * K, xs,
                           static_cast<size_t>(M) * 4);
    return e;
}

cudaError_t launch_linear_blk_gemv(const void *x, const void *w, const float *w_scale, const void *bias, void *out,
                                   void *xq, float *xs, int64_t m_pad, int64_t N, int64_t K, float eps, bool out_fp16,
                                   cudaStream_t st)
{
    if (!linear_blk_gemv_fits(1, K) || K % 128 != 0 || N % 128 != 0) return cudaErrorInvalidValue;
    const size_t wbytes = static_cast<size_t>(N) * static_cast<size_t>(K);
    const bool preload = !last_launch_writes_overlap(st, w, wbytes);
    const int n = static_cast<int>(N), k = static_cast<int>(K);
    cudaError_t e;
    switch (gemv_chunks_per_warp(K)) {
        case 1:
            e = out_fp16 ? launch_blk<1, __half>(x, w, w_scale, bias, out, xq, xs, m_pad, n, k, eps, preload, st)
                         : launch_blk<1, __nv_bfloat16>(x, w, w_scale, bias, out, xq, xs, m_pad, n, k, eps, preload,
                                                        st);
            break;
        case 2:
            e = out_fp16 ? launch_blk<2, __half>(x, w, w_scale, bias, out, xq, xs, m_pad, n, k, eps, preload, st)
                         : launch_blk<2, __nv_bfloat16>(x, w, w_scale, bias, out, xq, xs, m_pad, n, k, eps, preload,
                                                        st);
            break;
        default:
            e = out_fp16 ? launch_blk<3, __half>(x, w, w_scale, bias, out, xq, xs, m_pad, n, k, eps, preload, st)
                         : launch_blk<3, __nv_bfloat16>(x, w, w_scale, bias, out, xq, xs, m_pad, n, k, eps, preload,
                                                        st);
    }
    if (e == cudaSuccess)
        note_launch_writes(st, out, static_cast<size_t>(N) * 2, xq, xq != nullptr ? static_cast<size_t>(K) : 0, xs,
                           xs != nullptr ? static_cast<size_t>(K / 128) * static_cast<size_t>(m_pad) * 4 : 0);
    return e;
}

}  // namespace fp8q
