// gemv_common.cuh -- the pieces shared by the two matrix-vector kernels for
// one or two tokens on the CUDA cores (w8a16_gemv.cu: bf16 activations;
// linear_gemv.cu: the per-token W8A8 linear with its quantization fused):
// the CTA shape, the weight stream, the exact E4M3 -> fp32 decode and the
// final reduction.
//
// A CTA owns ROWS consecutive output channels (8, or 4 for four tokens, to
// keep two CTAs per SM); its eight warps split K in 512-byte chunks (chunk c
// to warp c % 8), each lane one 16-byte piece of a chunk for all ROWS rows,
// so one activation load serves ROWS weight pieces.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace fp8q {
namespace gemv {

constexpr int kWarps = 8;
constexpr int kChunk = 512;           // bytes of K per warp step (16 per lane)
template <int MT>
constexpr int rows() { return MT >= 4 ? 4 : 8; }   // output channels per CTA

template <typename T>
__device__ __forceinline__ T to_out(float v);
template <>
__device__ __forceinline__ __nv_bfloat16 to_out<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }
template <>
__device__ __forceinline__ __half to_out<__half>(float v) { return __float2half_rn(v); }

// Weights are read once: no L1 allocation.
__device__ __forceinline__ uint4 ld_stream_u4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Two E4M3 bytes (the lower-addressed one in the low half) -> two fp32
// (exact: E4M3 -> f16 by the conversion instruction, f16 -> fp32 exactly).
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t pair)
{
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(static_cast<uint16_t>(pair)));
    return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}

// This lane's weight pieces of chunk c for the CTA's ROWS rows from n0
// (zero where past N or K).
template <int ROWS>
__device__ __forceinline__ void load_weights(const uint8_t *__restrict__ w, int64_t ldw, int n0, int N, int K, int c,
                                             int lane, uint4 (&wv)[ROWS])
{
    const int k = c * kChunk + lane * 16;
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
        wv[r] = (k < K && n0 + r < N) ? ld_stream_u4(w + static_cast<int64_t>(n0 + r) * ldw + k)
                                      : make_uint4(0u, 0u, 0u, 0u);
}

// acc[r][m] += w[r, 16 values] * a[m, 16 values], the weights decoded in
// pairs; xa holds the 16 activations of each token as fp32 pairs.
template <int ROWS, int MT>
__device__ __forceinline__ void fma_piece(const uint4 (&wv)[ROWS], const float2 (&xa)[MT][8],
                                          float2 (&acc)[ROWS][MT])
{
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

// Sum of each (row, token) over the lanes (shuffles) and then the warps
// (shared memory, red[warp][row][token]).  Returns, to thread
// r * MT + m for r < ROWS, m < MT, the full sum of (row r, token m); other
// threads get 0.
template <int ROWS, int MT>
__device__ __forceinline__ float reduce_cta(const float2 (&acc)[ROWS][MT], float (&red)[kWarps][ROWS][MT],
                                            int warp, int lane)
{
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
    float s = 0.0f;
    if (threadIdx.x < ROWS * MT) {
        const int r = threadIdx.x / MT, m = threadIdx.x % MT;
#pragma unroll
        for (int q = 0; q < kWarps; ++q) s += red[q][r][m];
    }
    return s;
}

}  // namespace gemv
}  // namespace fp8q
