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

__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t w) { return *reinterpret_cast<const __nv_bfloat162 *>(&w); }

// max(m, |x|) over the 16 values, on packed bf16 pairs: |x| and the max of
// bf16 values are exact in bf16 (the result is one of the inputs), and the
// packed max, like fmaxf, returns the other operand when one is NaN.
__device__ __forceinline__ float chunk_amax(const Chunk16 &c, float m)
{
    __nv_bfloat162 a = __hmax2(__habs2(as_bf2(c.lo.x)), __habs2(as_bf2(c.lo.y)));
    a = __hmax2(a, __hmax2(__habs2(as_bf2(c.lo.z)), __habs2(as_bf2(c.lo.w))));
    __nv_bfloat162 b = __hmax2(__habs2(as_bf2(c.hi.x)), __habs2(as_bf2(c.hi.y)));
    b = __hmax2(b, __hmax2(__habs2(as_bf2(c.hi.z)), __habs2(as_bf2(c.hi.w))));
    a = __hmax2(a, b);
    return fmaxf(m, fmaxf(__low2float(a), __high2float(a)));
}

// The IEEE quotients RN(x / s) of a pair, given r = RN(1 / s), by
// Markstein's correction (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1),
// 1990): with q0 = RN(x * r), the remainder x - q0 * s is exact in one FMA,
// and RN(q0 + remainder * r) is the correctly rounded quotient.  Checked
// exhaustively against the division on this GPU for every bf16 significand
// of x and every fp32 significand of s (2^30 pairs, at several exponent
// offsets): no difference.  The result carries the sign of x, as x / s
// does for s > 0 (this keeps -0 for x = -0).  The kernels use it only for
// normal finite s (the reciprocal is then a normal number); where the
// quotient would be subnormal in fp32, x / s is below 2^-11 and both round
// to a signed zero in E4M3.  Packed fp32x2 operations: each lane is the
// correctly rounded scalar operation (fma(q0, -s, x) is fma(-q0, s, x)
// exactly), two quotients per instruction.
__device__ __forceinline__ float2 quotient2(float2 x, float s, float r)
{
    const float2 r2 = make_float2(r, r);
    const float2 q0 = __fmul2_rn(x, r2);
    const float2 rem = __ffma2_rn(q0, make_float2(-s, -s), x);
    const float2 q = __ffma2_rn(rem, r2, q0);
    return make_float2(copysignf(q.x, x.x), copysignf(q.y, x.y));
}

// Four bf16 (two words) / s -> four E4M3 bytes packed little-endian.
__device__ __forceinline__ uint32_t quant4(uint32_t w0, uint32_t w1, float s, float r)
{
    const float2 q0 = quotient2(make_float2(bf_lo(w0), bf_hi(w0)), s, r);
    const float2 q1 = quotient2(make_float2(bf_lo(w1), bf_hi(w1)), s, r);
    return cvt_e4m3x2(q0.x, q0.y) | (cvt_e4m3x2(q1.x, q1.y) << 16);
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

// The same operations on 8-value units (one 16-byte word of bf16): the
// running max of |x| kept as a bf16 pair (exact, NaN-ignoring as above), and
// the codes of 8 values for a scale s with r = RN(1 / s), or, where s is not
// a normal finite number, by the IEEE division (as quant_chunk does).
__device__ __forceinline__ __nv_bfloat162 unit_amax2(const uint4 &v, __nv_bfloat162 acc)
{
    const __nv_bfloat162 a = __hmax2(__habs2(as_bf2(v.x)), __habs2(as_bf2(v.y)));
    const __nv_bfloat162 b = __hmax2(__habs2(as_bf2(v.z)), __habs2(as_bf2(v.w)));
    return __hmax2(acc, __hmax2(a, b));
}

__device__ __forceinline__ bool scale_has_reciprocal(float s) { return s >= 0x1p-126f && s <= 3.0e38f; }

__device__ __forceinline__ uint2 quant_unit8(const uint4 &v, float s, float r, bool recip)
{
    if (recip) return make_uint2(quant4(v.x, v.y, s, r), quant4(v.z, v.w, s, r));
    return make_uint2(quant4_div(v.x, v.y, s), quant4_div(v.z, v.w, s));
}

// 16 consecutive bf16 values from shared memory (16-byte aligned).
__device__ __forceinline__ Chunk16 load_chunk_smem(const void *p)
{
    Chunk16 c;
    c.lo = reinterpret_cast<const uint4 *>(p)[0];
    c.hi = reinterpret_cast<const uint4 *>(p)[1];
    return c;
}

}  // namespace fp8q
