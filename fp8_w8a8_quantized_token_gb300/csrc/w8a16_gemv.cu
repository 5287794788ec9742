// w8a16_gemv.cu -- the weight-only FP8 linear (W8A16) for up to four tokens
// on the CUDA cores:
//   out[m,n] = round(sum_k x[m,k] * e4m3(w[n,k]) * w_scale[n] + bias[n])
// (the Marlin weight-only linear of the "Fix FP8 Triton dtype selection on
// A100" page, implementation breakdown and key source snippets: bf16
// activations, E4M3 weights, one fp32 scale per output channel).  With one
// to four tokens the layer is a few matrix-vector products: two to eight
// flops per weight byte, far below
// what the E4M3 weights cost to stream from HBM, so the weights stay on the
// CUDA cores' side -- decoded to fp32 in registers (exact) and multiplied
// with fp32 FMAs on pairs (each lane a correctly rounded fmaf) -- rather
// than being converted into tensor-core operands.
//
// A CTA owns ROWS consecutive output channels (8, or 4 for four tokens, to
// keep two CTAs per SM); its eight warps split K in 512-byte chunks (chunk c
// to warp c % 8), each lane one 16-byte piece of a chunk for all ROWS rows,
// so one activation load serves ROWS weight pieces.  Sums are reduced across
// lanes with shuffles and across warps in shared memory, then scaled, biased
// and rounded once.  Unless the previous
// launch of the library wrote the weights, each warp issues its first
// chunk's weight loads before the dependency wait, so the weight stream
// overlaps the previous kernel's tail.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "device_common.cuh"
#include "internal.h"

namespace fp8q {
namespace {

constexpr int kGemvWarps = 8;
constexpr int kChunk = 512;           // bytes of K per warp step (16 per lane)
template <int MT>
constexpr int gemv_rows() { return MT >= 4 ? 4 : 8; }   // output channels per CTA

template <typename T>
__device__ __forceinline__ T gemv_out(float v);
template <>
__device__ __forceinline__ __nv_bfloat16 gemv_out<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }
template <>
__device__ __forceinline__ __half gemv_out<__half>(float v) { return __float2half_rn(v); }

// Weights are read once: no L1 allocation.
__device__ __forceinline__ uint4 ld_stream_u4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Two E4M3 bytes -> two fp32 (exact: E4M3 -> f16 by the conversion
// instruction, f16 -> fp32 exactly).
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t pair)
{
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(static_cast<uint16_t>(pair)));
    return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}

template <int MT, typename OutT, int ROWS = gemv_rows<MT>()>
__global__ void __launch_bounds__(32 * kGemvWarps) w8a16_gemv_kernel(
    const __nv_bfloat16 *__restrict__ x, int64_t ldx, const uint8_t *__restrict__ w, int64_t ldw,
    const float *__restrict__ w_scale, const __nv_bfloat16 *__restrict__ bias, OutT *__restrict__ out, int M,
    int N, int K, int preload)
{
    __shared__ float red[kGemvWarps][ROWS][MT];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * ROWS;
    const int nchunks = (K + kChunk - 1) / kChunk;
    float2 acc[ROWS][MT];   // even and odd k of each (row, token)
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[r][m] = make_float2(0.0f, 0.0f);

    // Weight pieces of chunk c for this lane (zero where past N or K).
    auto load_w = [&](int c, uint4 (&wv)[ROWS]) {
        const int k = c * kChunk + lane * 16;
#pragma unroll
        for (int r = 0; r < ROWS; ++r)
            wv[r] = (k < K && n0 + r < N) ? ld_stream_u4(w + static_cast<int64_t>(n0 + r) * ldw + k)
                                          : make_uint4(0u, 0u, 0u, 0u);
    };
    uint4 wv[ROWS];
    int c = warp;
    if (preload && c < nchunks) load_w(c, wv);
    pdl_wait();
    pdl_trigger();
    if (!preload && c < nchunks) load_w(c, wv);
    for (; c < nchunks; c += kGemvWarps) {
        if (c != warp) load_w(c, wv);
        const int k = c * kChunk + lane * 16;
        if (k < K) {
            // This lane's 16 activations of every token, as fp32 pairs.
            float2 xa[MT][8];
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
                if (m < M) {
                    const uint4 *px = reinterpret_cast<const uint4 *>(x + static_cast<int64_t>(m) * ldx + k);
                    lo = __ldg(px);
                    hi = __ldg(px + 1);
                }
                const uint32_t words[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    xa[m][j] = make_float2(__uint_as_float(words[j] << 16), __uint_as_float(words[j] & 0xFFFF0000u));
            }
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                const uint32_t bw[4] = {wv[r].x, wv[r].y, wv[r].z, wv[r].w};
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float2 wf = e4m3x2_to_f32x2(bw[j >> 1] >> (16 * (j & 1)));
#pragma unroll
                    for (int m = 0; m < MT; ++m) acc[r][m] = __ffma2_rn(wf, xa[m][j], acc[r][m]);
                }
            }
        }
    }
    // Lanes, then warps.
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            float v = acc[r][m].x + acc[r][m].y;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) red[warp][r][m] = v;
        }
    __syncthreads();
    if (threadIdx.x < ROWS * MT) {
        const int r = threadIdx.x / MT, m = threadIdx.x % MT;
        const int n = n0 + r;
        if (n < N && m < M) {
            float s = 0.0f;
#pragma unroll
            for (int q = 0; q < kGemvWarps; ++q) s += red[q][r][m];
            const float b = bias != nullptr ? __bfloat162float(bias[n]) : 0.0f;
            out[static_cast<int64_t>(m) * N + n] = gemv_out<OutT>(fmaf(s, __ldg(w_scale + n), b));
        }
    }
}

template <int MT, typename OutT>
cudaError_t launch_gemv_t(const void *x, int64_t ldx, const void *w, int64_t ldw, const float *w_scale,
                          const void *bias, void *out, int M, int N, int K, bool preload, cudaStream_t st)
{
    cudaLaunchConfig_t cfg = {};
    constexpr int kRows = gemv_rows<MT>();
    cfg.gridDim = dim3(static_cast<unsigned>((N + kRows - 1) / kRows));
    cfg.blockDim = dim3(32 * kGemvWarps);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, w8a16_gemv_kernel<MT, OutT>, static_cast<const __nv_bfloat16 *>(x), ldx,
                              static_cast<const uint8_t *>(w), ldw, w_scale,
                              static_cast<const __nv_bfloat16 *>(bias), static_cast<OutT *>(out), M, N, K,
                              preload ? 1 : 0);
}

template <typename OutT>
cudaError_t launch_gemv_out(const void *x, int64_t ldx, const void *w, int64_t ldw, const float *w_scale,
                            const void *bias, void *out, int M, int N, int K, bool preload, cudaStream_t st)
{
    if (M == 1) return launch_gemv_t<1, OutT>(x, ldx, w, ldw, w_scale, bias, out, M, N, K, preload, st);
    if (M == 2) return launch_gemv_t<2, OutT>(x, ldx, w, ldw, w_scale, bias, out, M, N, K, preload, st);
    return launch_gemv_t<4, OutT>(x, ldx, w, ldw, w_scale, bias, out, M, N, K, preload, st);
}

}  // namespace

cudaError_t launch_w8a16_gemv(const void *x, int64_t ldx, const void *w, int64_t ldw, const float *w_scale,
                              const void *bias, void *out, int64_t M, int64_t N, int64_t K, bool out_fp16,
                              cudaStream_t st)
{
    if (M < 1 || M > kW16GemvMaxM) return cudaErrorInvalidValue;
    const size_t wbytes = static_cast<size_t>(N - 1) * static_cast<size_t>(ldw) + static_cast<size_t>(K);
    const bool preload = !last_launch_writes_overlap(st, w, wbytes);
    const cudaError_t e =
        out_fp16 ? launch_gemv_out<__half>(x, ldx, w, ldw, w_scale, bias, out, static_cast<int>(M),
                                           static_cast<int>(N), static_cast<int>(K), preload, st)
                 : launch_gemv_out<__nv_bfloat16>(x, ldx, w, ldw, w_scale, bias, out, static_cast<int>(M),
                                                  static_cast<int>(N), static_cast<int>(K), preload, st);
    if (e == cudaSuccess) note_launch_writes(st, out, static_cast<size_t>(M) * N * 2);
    return e;
}

}  // namespace fp8q
