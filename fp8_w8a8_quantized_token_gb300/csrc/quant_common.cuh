// quant_common.cuh -- the quantization arithmetic shared by the standalone
// quantizers (quant.cu) and the GEMM's fused-quantization prologue
// (gemm_kernel.cuh), so both produce the same codes and scales bit for bit:
//   s = max(amax(|x| over the group), eps) / 448
//   q = cvt.rn.satfinite.e4m3(x / s)   (the correctly rounded fp32 quotient)
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "device_common.cuh"

namespace fp8q {

// 16 consecutive bf16 values held as 8 packed registers.
struct Chunk16 {
    uint4 lo, hi;
};

__device__ __forceinline__ Chunk16 load_chunk(const __nv_bfloat16 *p)
{
    Chunk16 c;
    c.lo = __ldg(reinterpret_cast<const uint4 *>(p));
    c.hi = __ldg(reinterpret_cast<const uint4 *>(p) + 1);
    return c;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float amax_word(uint32_t w, float m)
{
    return fmaxf(m, fmaxf(fabsf(bf_lo(w)), fabsf(bf_hi(w))));
}

__device__ __forceinline__ float chunk_amax(const Chunk16 &c, float m)
{
    m = amax_word(c.lo.x, m); m = amax_word(c.lo.y, m); m = amax_word(c.lo.z, m); m = amax_word(c.lo.w, m);
    m = amax_word(c.hi.x, m); m = amax_word(c.hi.y, m); m = amax_word(c.hi.z, m); m = amax_word(c.hi.w, m);
    return m;
}

// The IEEE quotient RN(x / s), given r = RN(1 / s), by Markstein's
// correction (P. Markstein, "Computation of elementary functions on the IBM
// RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990): with
// q0 = RN(x * r), the remainder x - q0 * s is exact in one FMA, and
// RN(q0 + remainder * r) is the correctly rounded quotient.  Checked
// exhaustively against the division on this GPU for every bf16 significand
// of x and every fp32 significand of s (2^30 pairs, at several exponent
// offsets): no difference.  The result carries the sign of x, as x / s
// does for s > 0 (this keeps -0 for x = -0).  The kernels use it only for
// normal finite s (the reciprocal is then a normal number); where the
// quotient would be subnormal in fp32, x / s is below 2^-11 and both round
// to a signed zero in E4M3.
__device__ __forceinline__ float quotient(float x, float s, float r)
{
    const float q0 = x * r;
    const float rem = fmaf(-q0, s, x);
    return copysignf(fmaf(rem, r, q0), x);
}

// Four bf16 (two words) / s -> four E4M3 bytes packed little-endian.
__device__ __forceinline__ uint32_t quant4(uint32_t w0, uint32_t w1, float s, float r)
{
    const uint32_t a = cvt_e4m3x2(quotient(bf_lo(w0), s, r), quotient(bf_hi(w0), s, r));
    const uint32_t b = cvt_e4m3x2(quotient(bf_lo(w1), s, r), quotient(bf_hi(w1), s, r));
    return a | (b << 16);
}

__device__ __forceinline__ uint32_t quant4_div(uint32_t w0, uint32_t w1, float s)
{
    const uint32_t a = cvt_e4m3x2(bf_lo(w0) / s, bf_hi(w0) / s);
    const uint32_t b = cvt_e4m3x2(bf_lo(w1) / s, bf_hi(w1) / s);
    return a | (b << 16);
}

__device__ __forceinline__ uint4 quant_chunk(const Chunk16 &c, float s)
{
    uint4 q;
    if (s >= 0x1p-126f && s <= 3.0e38f) {
        const float r = 1.0f / s;
        q.x = quant4(c.lo.x, c.lo.y, s, r);
        q.y = quant4(c.lo.z, c.lo.w, s, r);
        q.z = quant4(c.hi.x, c.hi.y, s, r);
        q.w = quant4(c.hi.z, c.hi.w, s, r);
    } else {
        // Infinite scale (an infinite input): x / inf = +-0, inf / inf = NaN;
        // a zero or subnormal scale (an eps below 448 * 2^-126): the IEEE
        // division as well (its reciprocal would overflow).
        q.x = quant4_div(c.lo.x, c.lo.y, s);
        q.y = quant4_div(c.lo.z, c.lo.w, s);
        q.z = quant4_div(c.hi.x, c.hi.y, s);
        q.w = quant4_div(c.hi.z, c.hi.w, s);
    }
    return q;
}

__device__ __forceinline__ float scale_of(float amax, float eps) { return fmaxf(amax, eps) / 448.0f; }

// 16 consecutive bf16 values from shared memory (16-byte aligned).
__device__ __forceinline__ Chunk16 load_chunk_smem(const void *p)
{
    Chunk16 c;
    c.lo = reinterpret_cast<const uint4 *>(p)[0];
    c.hi = reinterpret_cast<const uint4 *>(p)[1];
    return c;
}

}  // namespace fp8q
