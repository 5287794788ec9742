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

// exp(t) in fp32 as a fixed sequence of IEEE fp32 operations (no library
// exp): Cody and Waite's range reduction (W. J. Cody, W. Waite, "Software
// Manual for the Elementary Functions", 1980) with fused multiply-adds --
// n = rint(t * log2 e), r = t - n*ln2_hi - n*ln2_lo, ln2_hi = ln 2 rounded
// to fp32 and ln2_lo the fp32 rounding of the rest -- then the Taylor
// series of exp(r) to degree 7 (coefficients 1/k! rounded to fp32, Horner's
// rule with FMAs) and the exact scaling by 2^n.  t > 88: +inf; t < -32: 0
// (exp(t) < 2^-46 cannot change 1 + exp(t), its only use).
// Two values at a time: the packed fp32x2 operations (__ffma2_rn,
// __fmul2_rn, __fadd2_rn) round each lane exactly as the scalar operation
// does.  n = rint(u) for u = t * log2 e is formed as (u + 1.5 * 2^23) -
// 1.5 * 2^23, which rounds u to the nearest integer (ties to even) for
// |u| < 2^22 -- all of [-32, 88] -- and leaves n + 127 in the low bits of
// u + 1.5 * 2^23 for the exponent of 2^n.  fma(-n, c, x) is written
// fma(n, -c, x) (the same exact product).  Lanes outside [-32, 88] are
// computed and then replaced.
__device__ __forceinline__ float2 exp_fixed2(float2 t)
{
    constexpr float kShift = 0x1.8p23f;
    const float2 u = __fmul2_rn(t, make_float2(0x1.715476p+0f, 0x1.715476p+0f));
    const float2 big = __fadd2_rn(u, make_float2(kShift, kShift));
    const float2 n = __fadd2_rn(big, make_float2(-kShift, -kShift));
    float2 r = __ffma2_rn(n, make_float2(-0x1.62e430p-1f, -0x1.62e430p-1f), t);
    r = __ffma2_rn(n, make_float2(0x1.05c610p-29f, 0x1.05c610p-29f), r);
    float2 p = make_float2(0x1.a01a02p-13f, 0x1.a01a02p-13f);
    p = __ffma2_rn(p, r, make_float2(0x1.6c16c2p-10f, 0x1.6c16c2p-10f));
    p = __ffma2_rn(p, r, make_float2(0x1.111112p-7f, 0x1.111112p-7f));
    p = __ffma2_rn(p, r, make_float2(0x1.555556p-5f, 0x1.555556p-5f));
    p = __ffma2_rn(p, r, make_float2(0x1.555556p-3f, 0x1.555556p-3f));
    p = __ffma2_rn(p, r, make_float2(0.5f, 0.5f));
    p = __ffma2_rn(p, r, make_float2(1.0f, 1.0f));
    p = __ffma2_rn(p, r, make_float2(1.0f, 1.0f));
    constexpr uint32_t kBias = 127u - 0x4B400000u;   // bits of 1.5 * 2^23 + n  ->  n + 127
    const float2 scale = make_float2(__uint_as_float((__float_as_uint(big.x) + kBias) << 23),
                                     __uint_as_float((__float_as_uint(big.y) + kBias) << 23));
    float2 e = __fmul2_rn(p, scale);
    if (t.x > 88.0f) e.x = __uint_as_float(0x7F800000u);
    if (t.x < -32.0f) e.x = 0.0f;
    if (t.y > 88.0f) e.y = __uint_as_float(0x7F800000u);
    if (t.y < -32.0f) e.y = 0.0f;
    return e;
}

// silu(a) * b in fp32 for two lanes: a / (1 + exp(-a)) (IEEE add and
// division), times b -- the fuse_silu_and_mul input of the group quantizer
// (row-padding page, key source snippets): gate a from the first half of
// the row, up b from the second, no rounding to bf16 in between.  (A
// division by the approximate reciprocal, one Newton step and Markstein's
// correction matched the IEEE quotient on every finite bf16 gate but did
// not make the kernel faster, so the IEEE division stays.)
__device__ __forceinline__ float2 silu_mul2(float2 a, float2 b)
{
    const float2 den = __fadd2_rn(make_float2(1.0f, 1.0f), exp_fixed2(make_float2(-a.x, -a.y)));
    return __fmul2_rn(make_float2(__fdiv_rn(a.x, den.x), __fdiv_rn(a.y, den.y)), b);
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
