// w8a16_gemv.cu -- the weight-only FP8 linear (W8A16) for one or two tokens
// on the CUDA cores:
//   out[m,n] = round(sum_k x[m,k] * e4m3(w[n,k]) * w_scale[n] + bias[n])
// (the Marlin weight-only linear of the "Fix FP8 Triton dtype selection on
// A100" page, implementation breakdown and key source snippets: bf16
// activations, E4M3 weights, one fp32 scale per output channel).  With one
// or two tokens the layer is one or two matrix-vector products: two or four
// flops per weight byte, far below
// what the E4M3 weights cost to stream from HBM, so the weights stay on the
// CUDA cores' side -- decoded to fp32 in registers (exact) and multiplied
// with fp32 FMAs on pairs (each lane a correctly rounded fmaf) -- rather
// than being converted into tensor-core operands.
//
// The CTA shape is that of gemv_common.cuh.  Sums are reduced across lanes
// with shuffles and across warps in shared memory, then scaled, biased and
// rounded once.  Unless a library kernel that may still be running writes
// the weights, each warp issues its first chunk's weight loads before the
// dependency wait, so the weight stream overlaps the previous kernel's tail.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "device_common.cuh"
#include "gemv_common.cuh"
#include "internal.h"

namespace fp8q {
namespace {

using gemv::kChunk;
using gemv::kWarps;

template <int MT, typename OutT, int ROWS = gemv::rows<MT>()>
__global__ void __launch_bounds__(32 * kWarps) w8a16_gemv_kernel(
    const __nv_bfloat16 *__restrict__ x, int64_t ldx, const uint8_t *__restrict__ w, int64_t ldw,
    const float *__restrict__ w_scale, const __nv_bfloat16 *__restrict__ bias, OutT *__restrict__ out, int M,
    int N, int K, int preload)
{
    __shared__ float red[kWarps][ROWS][MT];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * ROWS;
    const int nchunks = (K + kChunk - 1) / kChunk;
    float2 acc[ROWS][MT];   // even and odd k of each (row, token)
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[r][m] = make_float2(0.0f, 0.0f);

    uint4 wv[ROWS];
    int c = warp;
    if (preload && c < nchunks) gemv::load_weights<ROWS>(w, ldw, n0, N, K, c, lane, wv);
    pdl_wait();
    pdl_trigger();
    if (!preload && c < nchunks) gemv::load_weights<ROWS>(w, ldw, n0, N, K, c, lane, wv);
    for (; c < nchunks; c += kWarps) {
        if (c != warp) gemv::load_weights<ROWS>(w, ldw, n0, N, K, c, lane, wv);
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
            gemv::fma_piece<ROWS, MT>(wv, xa, acc);
        }
    }
    const float s = gemv::reduce_cta<ROWS, MT>(acc, red, warp, lane);
    if (threadIdx.x < ROWS * MT) {
        const int r = threadIdx.x / MT, m = threadIdx.x % MT;
        const int n = n0 + r;
        if (n < N && m < M) {
            const float b = bias != nullptr ? __bfloat162float(bias[n]) : 0.0f;
            out[static_cast<int64_t>(m) * N + n] = gemv::to_out<OutT>(fmaf(s, __ldg(w_scale + n), b));
        }
    }
}

template <int MT, typename OutT>
cudaError_t launch_gemv_t(const void *x, int64_t ldx, const void *w, int64_t ldw, const float *w_scale,
                          const void *bias, void *out, int M, int N, int K, bool preload, cudaStream_t st)
{
    cudaLaunchConfig_t cfg = {};
    constexpr int kRows = gemv::rows<MT>();
    cfg.gridDim = dim3(static_cast<unsigned>((N + kRows - 1) / kRows));
    cfg.blockDim = dim3(32 * kWarps);
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
    return launch_gemv_t<2, OutT>(x, ldx, w, ldw, w_scale, bias, out, M, N, K, preload, st);
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
