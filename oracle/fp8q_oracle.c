/*
 * fp8q_oracle.c -- plain, slow, single-threaded CPU oracle for the FP8 W8A8
 * linear layer.  TEST INFRASTRUCTURE ONLY: the product path never links,
 * loads or calls this file; only tests/, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code with the CUDA library.
 *
 * Sources (cited by page title and section):
 *   [PR27896] "Remove per-call padding overhead of the FP8 blockwise GEMM"
 *             (sgl-project/sglang PR 27896): sections "Implementation
 *             breakdown", "Key source snippets"
 *             (sglang_per_token_group_quant_fp8_row_padded,
 *             cutlass_w8a8_block_fp8_linear_with_fallback), "Risks and impact".
 *   [PR34331] "Tune FP8 GEMM Triton tiles on L40S and enable by default"
 *             (PR 34331): "Motivation" and "Key source snippets"
 *             (apply_fp8_linear channelwise branch, fp8_scaled_mm).
 *   [PR31340] "Fix FP8 Triton dtype selection on A100" (PR 31340): "Key
 *             source snippets" (fp8_dtype_to_triton: the format is
 *             torch.float8_e4m3fn).
 *   The E4M3 format itself is the OCP 8-bit floating point "E4M3" encoding
 *   (torch.float8_e4m3fn): 1 sign bit, 4 exponent bits with bias 7,
 *   3 mantissa bits, no infinities, S.1111.111 is NaN, largest finite 448.
 *
 * Precision: the quantization decisions are made in fp32, the precision the
 * pages fix for the scales (x_s is float32 in [PR27896] "Key source
 * snippets") and the fp8_min/fp8_max clamp; the GEMM is evaluated exactly in
 * double: every E4M3 value is an integer multiple of 2^-9 of magnitude below
 * 2^9, so each product is an integer multiple of 2^-18 below 2^36 such units,
 * and a sum of up to 2^14 products stays below 2^50 units -- exact in a
 * 53-bit mantissa for every K <= 16384.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared (no fast-math: the
 * fp32 division below must be the IEEE-754 correctly rounded one, and no
 * multiply-add may be contracted).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define E4M3_MAX 448.0

/* ------------------------------------------------------------------------ */
/* E4M3 (float8_e4m3fn) codec, from the format definition.                   */
/* ------------------------------------------------------------------------ */

/* Value of an E4M3 code: subnormal (e=0) m*2^-9; normal (1+m/8)*2^(e-7);
 * S.1111.111 is NaN. */
double fp8q_oracle_e4m3_decode(uint8_t code)
{
    int s = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* Round q >= 0 to the nearest integer, ties to the even integer. */
static double round_half_even(double q)
{
    double fl = floor(q);
    double d = q - fl;
    if (d > 0.5) return fl + 1.0;
    if (d < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* fp32 -> E4M3, round to nearest even, saturating to +-448 ("satfinite"):
 * the pages clamp to [fp8_min, fp8_max] before the cast.  The sign of zero
 * is kept (a negative value that rounds to zero gives 0x80).  NaN -> 0x7F. */
uint8_t fp8q_oracle_e4m3_encode(float v)
{
    if (isnan(v)) return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= E4M3_MAX) return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: grid step 2^-9; r == 8 lands on the smallest
         * normal 2^-6 whose code is also 8. */
        double r = round_half_even(a * 512.0);
        return sign | (uint8_t)r;
    }
    int ex;
    frexp(a, &ex);            /* a = f * 2^ex, f in [0.5, 1) */
    int e = ex - 1;           /* a in [2^e, 2^(e+1)) */
    double r = round_half_even((ldexp(a, -e) - 1.0) * 8.0);
    if (r == 8.0) { r = 0.0; e += 1; }
    int biased = e + 7;
    if (biased > 15 || (biased == 15 && r == 7.0)) return sign | 0x7E; /* not reached after the clamp */
    return sign | (uint8_t)((biased << 3) | (int)r);
}

void fp8q_oracle_e4m3_encode_array(const float *v, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = fp8q_oracle_e4m3_encode(v[i]);
}

void fp8q_oracle_e4m3_decode_array(const uint8_t *c, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = fp8q_oracle_e4m3_decode(c[i]);
}

/* ------------------------------------------------------------------------ */
/* 16-bit float helpers                                                      */
/* ------------------------------------------------------------------------ */

float fp8q_oracle_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* One round-to-nearest-even rounding of a double to a binary float with
 * `mbits` explicit mantissa bits, minimum normal exponent `emin` and maximum
 * finite exponent `emax`; returns sign, biased exponent and mantissa packed
 * as (sign << (ebits+mbits)) | (E << mbits) | m.  Overflow gives infinity. */
static uint32_t round_to_binary(double y, int mbits, int ebits, int emin, int emax)
{
    int bias = (1 << (ebits - 1)) - 1;
    uint32_t sign = signbit(y) ? 1u : 0u;
    uint32_t sbit = sign << (ebits + mbits);
    uint32_t inf = sbit | (((1u << ebits) - 1u) << mbits);
    if (isnan(y)) return inf | (1u << (mbits - 1));
    double a = fabs(y);
    if (isinf(a)) return inf;
    if (a == 0.0) return sbit;
    int ex;
    frexp(a, &ex);
    int e = ex - 1;
    if (e < emin) {
        /* subnormal: step 2^(emin - mbits) */
        double r = round_half_even(ldexp(a, mbits - emin));
        if (r == ldexp(1.0, mbits)) return sbit | (1u << mbits); /* rounds up to min normal */
        return sbit | (uint32_t)r;
    }
    double r = round_half_even((ldexp(a, -e) - 1.0) * ldexp(1.0, mbits));
    if (r == ldexp(1.0, mbits)) { r = 0.0; e += 1; }
    if (e > emax) return inf;
    return sbit | ((uint32_t)(e + bias) << mbits) | (uint32_t)r;
}

uint16_t fp8q_oracle_f64_to_bf16(double y) { return (uint16_t)round_to_binary(y, 7, 8, -126, 127); }
uint16_t fp8q_oracle_f64_to_f16(double y) { return (uint16_t)round_to_binary(y, 10, 5, -14, 15); }

/* ------------------------------------------------------------------------ */
/* Dynamic activation quantization                                           */
/* ------------------------------------------------------------------------ */

/* Scale of one group: s = max(amax, eps) / 448 in fp32 (IEEE division).
 * The eps floor sits on amax: eps is handed to the device kernel beside
 * fp8_min and fp8_max ([PR27896] "Key source snippets"). */
static float group_scale(const uint16_t *x, int64_t n, float eps)
{
    float amax = 0.0f;
    for (int64_t k = 0; k < n; ++k) {
        float a = fabsf(fp8q_oracle_bf16_to_f32(x[k]));
        if (a > amax) amax = a;
    }
    float floored = amax > eps ? amax : eps;
    return floored / 448.0f;
}

/* q = cast_e4m3(clamp(x / s, fp8_min, fp8_max)), x / s an fp32 division. */
static void quant_run(const uint16_t *x, int64_t n, float s, uint8_t *q)
{
    for (int64_t k = 0; k < n; ++k) {
        float v = fp8q_oracle_bf16_to_f32(x[k]) / s;
        if (v > 448.0f) v = 448.0f;
        if (v < -448.0f) v = -448.0f;
        q[k] = fp8q_oracle_e4m3_encode(v);
    }
}

/* Per-token quantization of rows [r0, r1) of x[M, K] (row stride ldx, bf16
 * bits): one fp32 scale per row; xq is [M, K] row-major, xs is [M].
 * The channelwise path's qinput / x_scale ([PR34331] "Key source snippets",
 * apply_fp8_linear: x_scale has one entry per row of qinput). */
void fp8q_oracle_quant_per_token(const uint16_t *x, int64_t K, int64_t ldx, float eps,
                                 uint8_t *xq, float *xs, int64_t r0, int64_t r1)
{
    for (int64_t r = r0; r < r1; ++r) {
        float s = group_scale(x + r * ldx, K, eps);
        xs[r] = s;
        quant_run(x + r * ldx, K, s, xq + r * K);
    }
}

/* Per-token-group quantization into a row-padded buffer, rows [r0, r1) of
 * the first M rows ([PR27896] "Key source snippets",
 * sglang_per_token_group_quant_fp8_row_padded): x_q is (m_pad, K) row-major,
 * x_s is allocated (K/g, m_pad) and viewed transposed, so the scale of row r,
 * group j lives at xs[j * m_pad + r].  Rows >= M are never written. */
void fp8q_oracle_quant_group_row_padded(const uint16_t *x, int64_t K, int64_t ldx, int64_t g,
                                        float eps, int64_t m_pad, uint8_t *xq, float *xs,
                                        int64_t r0, int64_t r1)
{
    int64_t groups = K / g;
    for (int64_t r = r0; r < r1; ++r) {
        for (int64_t j = 0; j < groups; ++j) {
            const uint16_t *xg = x + r * ldx + j * g;
            float s = group_scale(xg, g, eps);
            xs[j * m_pad + r] = s;
            quant_run(xg, g, s, xq + r * K + j * g);
        }
    }
}

/* Weight quantization with one fp32 scale per (bn x bk) block of w[N, K]
 * (K contiguous, stride ldw); ws is [ceil(N/bn)][ceil(K/bk)] row-major.
 * Same scale and cast rule as the activations.  bn = 1, bk = K gives the
 * per-output-channel weights of the channelwise path. */
void fp8q_oracle_quant_weight_blocks(const uint16_t *w, int64_t N, int64_t K, int64_t ldw,
                                     int64_t bn, int64_t bk, float eps, uint8_t *wq, float *ws)
{
    int64_t nb = (N + bn - 1) / bn, kb = (K + bk - 1) / bk;
    for (int64_t ib = 0; ib < nb; ++ib) {
        for (int64_t jb = 0; jb < kb; ++jb) {
            int64_t n0 = ib * bn, n1 = n0 + bn < N ? n0 + bn : N;
            int64_t k0 = jb * bk, k1 = k0 + bk < K ? k0 + bk : K;
            float amax = 0.0f;
            for (int64_t n = n0; n < n1; ++n)
                for (int64_t k = k0; k < k1; ++k) {
                    float a = fabsf(fp8q_oracle_bf16_to_f32(w[n * ldw + k]));
                    if (a > amax) amax = a;
                }
            float s = (amax > eps ? amax : eps) / 448.0f;
            ws[ib * kb + jb] = s;
            for (int64_t n = n0; n < n1; ++n)
                quant_run(w + n * ldw + k0, k1 - k0, s, wq + n * K + k0);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Variants of the quantizers                                                */
/* ------------------------------------------------------------------------ */

/* Static per-tensor quantization of rows [r0, r1): one given fp32 scale s
 * for the whole tensor (the static quant kernel _static_quant_fp8 named in
 * [PR31340] "Implementation breakdown"), q = cast_e4m3(clamp(x / s)). */
void fp8q_oracle_quant_static(const uint16_t *x, int64_t K, int64_t ldx, float s, uint8_t *xq,
                              int64_t r0, int64_t r1)
{
    for (int64_t r = r0; r < r1; ++r) quant_run(x + r * ldx, K, s, xq + r * K);
}

/* The scale rounded up to a power of two, so that it is exactly an 8-bit
 * exponent (UE8M0; the scale_ue8m0 flag of the group quantizer in [PR27896]
 * "Key source snippets"): the smallest power of two >= s among the normal
 * fp32 numbers, i.e. 2^ceil(log2 s) for a normal s and 2^-126 below that;
 * +inf stays +inf.  frexp gives s = f * 2^e with f in [0.5, 1): s is itself
 * a power of two exactly when f == 0.5. */
static float pow2_ceil(float s)
{
    if (!(s >= FLT_MIN)) return FLT_MIN;
    if (isinf(s)) return s;
    int e;
    double f = frexp((double)s, &e);
    if (f == 0.5) return s;
    return (float)ldexp(1.0, e); /* +inf if e == 128 */
}

/* exp(t) in fp32, fully specified by its sequence of IEEE fp32 operations
 * (no library exp): the range reduction of Cody and Waite ("Software Manual
 * for the Elementary Functions", 1980), done with fused multiply-adds,
 *   n = rint(RN(t * log2 e)),  r = t - n*ln2_hi - n*ln2_lo  (two FMAs),
 * where ln2_hi is ln 2 rounded to fp32 and ln2_lo the fp32 rounding of the
 * remainder, then exp(r) from its Taylor series to degree 7 (coefficients
 * 1/k! rounded to fp32, Horner's rule with FMAs; |r| <= ln2/2 makes the
 * truncation error below 1e-8 relative), times 2^n (exact).  t > 88 gives
 * +inf; t < -32 gives 0 (then exp(t) < 2^-46 cannot change 1 + exp(t) in
 * fp32, the only use made of it). */
static float exp_f32(float t)
{
    if (t > 88.0f) return INFINITY;
    if (t < -32.0f) return 0.0f;
    const float log2e = 0x1.715476p+0f, ln2_hi = 0x1.62e430p-1f, ln2_lo = -0x1.05c610p-29f;
    const float c7 = 0x1.a01a02p-13f, c6 = 0x1.6c16c2p-10f, c5 = 0x1.111112p-7f, c4 = 0x1.555556p-5f,
                c3 = 0x1.555556p-3f, c2 = 0x1.0p-1f;
    float prod = t * log2e;
    float n = rintf(prod);
    float r = fmaf(-n, ln2_hi, t);
    r = fmaf(-n, ln2_lo, r);
    float p = c7;
    p = fmaf(p, r, c6);
    p = fmaf(p, r, c5);
    p = fmaf(p, r, c4);
    p = fmaf(p, r, c3);
    p = fmaf(p, r, c2);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    return p * ldexpf(1.0f, (int)n);
}

/* silu(a) * b in fp32: silu(a) = a / (1 + exp(-a)) (IEEE fp32 add and
 * division, exp as above), then one fp32 multiply -- the fuse_silu_and_mul
 * input of the group quantizer ([PR27896] "Key source snippets"): the
 * quantized row is silu(gate) * up, gate the first and up the second half
 * of the input row, with no rounding to bf16 in between. */
static float silu_mul(float a, float b)
{
    float den = 1.0f + exp_f32(-a);
    float silu = a / den;
    return silu * b;
}

void fp8q_oracle_exp_f32_array(const float *t, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = exp_f32(t[i]);
}

void fp8q_oracle_silu_mul_array(const float *a, const float *b, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = silu_mul(a[i], b[i]);
}

void fp8q_oracle_pow2_ceil_array(const float *s, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = pow2_ceil(s[i]);
}

/* The row-padded per-token-group quantizer with its two options ([PR27896]
 * "Key source snippets": the scale_ue8m0 and fuse_silu_and_mul arguments of
 * sgl_per_token_group_quant_8bit):
 *   silu_and_mul: x rows hold 2K values; the quantized values are
 *                 y[k] = silu(x[k]) * x[K + k] in fp32 (silu_mul above);
 *                 otherwise y[k] = x[k].
 *   ue8m0:        the group scale max(amax|y|, eps) / 448 is rounded up to a
 *                 power of two (pow2_ceil) before use.
 * q = cast_e4m3(clamp(y / s)), y / s an fp32 division; layout as in
 * fp8q_oracle_quant_group_row_padded (x_s[j * m_pad + r]). */
void fp8q_oracle_quant_group_row_padded_ex(const uint16_t *x, int64_t K, int64_t ldx, int64_t g, float eps,
                                           int ue8m0, int silu_and_mul, int64_t m_pad, uint8_t *xq,
                                           float *xs, int64_t r0, int64_t r1)
{
    float *y = (float *)malloc((size_t)g * sizeof(float));
    if (y == NULL) abort();
    int64_t groups = K / g;
    for (int64_t r = r0; r < r1; ++r) {
        const uint16_t *xr = x + r * ldx;
        for (int64_t j = 0; j < groups; ++j) {
            float amax = 0.0f;
            for (int64_t i = 0; i < g; ++i) {
                int64_t k = j * g + i;
                y[i] = silu_and_mul ? silu_mul(fp8q_oracle_bf16_to_f32(xr[k]), fp8q_oracle_bf16_to_f32(xr[K + k]))
                                    : fp8q_oracle_bf16_to_f32(xr[k]);
                float a = fabsf(y[i]);
                if (a > amax) amax = a;
            }
            float s = (amax > eps ? amax : eps) / 448.0f;
            if (ue8m0) s = pow2_ceil(s);
            xs[j * m_pad + r] = s;
            for (int64_t i = 0; i < g; ++i) {
                float v = y[i] / s;
                if (v > 448.0f) v = 448.0f;
                if (v < -448.0f) v = -448.0f;
                xq[r * K + j * g + i] = fp8q_oracle_e4m3_encode(v);
            }
        }
    }
    free(y);
}

/* ------------------------------------------------------------------------ */
/* Scaled GEMMs                                                              */
/* ------------------------------------------------------------------------ */

static void decode_table(double t[256])
{
    for (int c = 0; c < 256; ++c) t[c] = fp8q_oracle_e4m3_decode((uint8_t)c);
}

static uint16_t round_out(double y, int out_fp16)
{
    return out_fp16 ? fp8q_oracle_f64_to_f16(y) : fp8q_oracle_f64_to_bf16(y);
}

/* Channelwise scaled GEMM ([PR34331] "Key source snippets",
 * fp8_scaled_mm(qinput, weight, x_scale, weight_scale, out_dtype, bias)):
 *   y[m, n] = (sum_k dec(a[m, k]) * dec(b[k, n])) * sa[m] * sb[n] (+ bias[n])
 * with the weight logically [K, N] and stored K-contiguous: element (k, n)
 * at b[n * ldb + k].  The sum is exact in double; y is rounded once to the
 * output type.  Rows [r0, r1); out[m * ldo + n]; yd (optional) gets y. */
void fp8q_oracle_gemm_channelwise(const uint8_t *a, int64_t lda, const uint8_t *b, int64_t ldb,
                                  const float *sa, const float *sb, const uint16_t *bias,
                                  int64_t N, int64_t K, int out_fp16, uint16_t *out, int64_t ldo,
                                  double *yd, int64_t r0, int64_t r1)
{
    double t[256];
    decode_table(t);
    double *arow = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    for (int64_t m = r0; m < r1; ++m) {
        for (int64_t k = 0; k < K; ++k) arow[k] = t[a[m * lda + k]];
        for (int64_t n = 0; n < N; ++n) {
            const uint8_t *bc = b + n * ldb;
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) acc += arow[k] * t[bc[k]];
            double y = acc * (double)sa[m] * (double)sb[n];
            if (bias) y += (double)fp8q_oracle_bf16_to_f32(bias[n]);
            out[m * ldo + n] = round_out(y, out_fp16);
            if (yd) yd[m * ldo + n] = y;
        }
    }
    free(arow);
}

/* Blockwise scaled GEMM ([PR27896] "Key source snippets",
 * fp8_blockwise_scaled_mm(q_input, weight.T, x_scale, weight_scale.T)):
 * activations carry one scale per (row, 128-column group) in the
 * column-major layout sa[kb * m_pad + m]; the weight w[N, K] carries one
 * scale per 128 x 128 block, sw[(n / 128) * (K / 128) + kb].
 *   y[m, n] = sum_kb P_kb * sa[m, kb] * sw[n / 128, kb]  (+ bias[n])
 *   P_kb    = sum_{k in block kb} dec(a[m, k]) * dec(w[n, k])   (exact)
 * The bias is added after the GEMM in the reference wrapper; here it joins
 * y before the single rounding.  Rows [r0, r1). */
/* Weight-only FP8 linear (W8A16; the Marlin linear of [PR31340]
 * "Implementation breakdown" and "Key source snippets",
 * apply_fp8_marlin_linear(input, weight, weight_scale, ..., bias): weight-only,
 * no input scale), rows [r0, r1):
 *   out[m, n] = round(sum_k x[m, k] * dec(w[n, k]) * ws[n] + bias[n])
 * x bf16 [M, K] (row stride ldx), w e4m3 [N, K] (row stride ldw), ws fp32 [N]
 * (a per-tensor scale is the case of equal entries).  Evaluated in double:
 * each product of a bf16 and an E4M3 value (8 + 4 significant bits) is
 * exact; the sum's rounding error is at most K * 2^-53 relative to the
 * largest partial sum, ~1e-12 for K <= 16384; one final rounding. */
void fp8q_oracle_gemm_w8a16(const uint16_t *x, int64_t ldx, const uint8_t *w, int64_t ldw, const float *ws,
                            const uint16_t *bias, int64_t N, int64_t K, int out_fp16, uint16_t *out,
                            int64_t ldo, double *yd, int64_t r0, int64_t r1)
{
    double t[256];
    decode_table(t);
    double *xrow = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    for (int64_t m = r0; m < r1; ++m) {
        for (int64_t k = 0; k < K; ++k) xrow[k] = (double)fp8q_oracle_bf16_to_f32(x[m * ldx + k]);
        for (int64_t n = 0; n < N; ++n) {
            const uint8_t *wr = w + n * ldw;
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) acc += xrow[k] * t[wr[k]];
            double y = acc * (double)ws[n];
            if (bias) y += (double)fp8q_oracle_bf16_to_f32(bias[n]);
            out[m * ldo + n] = round_out(y, out_fp16);
            if (yd) yd[m * ldo + n] = y;
        }
    }
    free(xrow);
}

void fp8q_oracle_gemm_blockwise(const uint8_t *a, int64_t lda, const uint8_t *w, int64_t ldw,
                                const float *sa, int64_t m_pad, const float *sw,
                                const uint16_t *bias, int64_t N, int64_t K, int out_fp16,
                                uint16_t *out, int64_t ldo, double *yd, int64_t r0, int64_t r1)
{
    const int64_t B = 128;
    int64_t kblocks = K / B;
    double t[256];
    decode_table(t);
    double *arow = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    for (int64_t m = r0; m < r1; ++m) {
        for (int64_t k = 0; k < K; ++k) arow[k] = t[a[m * lda + k]];
        for (int64_t n = 0; n < N; ++n) {
            const uint8_t *wr = w + n * ldw;
            double y = 0.0;
            for (int64_t kb = 0; kb < kblocks; ++kb) {
                double p = 0.0;
                for (int64_t k = kb * B; k < (kb + 1) * B; ++k) p += arow[k] * t[wr[k]];
                y += p * (double)sa[kb * m_pad + m] * (double)sw[(n / B) * kblocks + kb];
            }
            if (bias) y += (double)fp8q_oracle_bf16_to_f32(bias[n]);
            out[m * ldo + n] = round_out(y, out_fp16);
            if (yd) yd[m * ldo + n] = y;
        }
    }
    free(arow);
}

/* The same two GEMMs at a list of (m, n) positions only: out[i] is the
 * output element at (ms[i], ns[i]).  For spot checks at sizes where the full
 * product would take the oracle too long. */
void fp8q_oracle_gemm_channelwise_at(const uint8_t *a, int64_t lda, const uint8_t *b, int64_t ldb,
                                     const float *sa, const float *sb, const uint16_t *bias,
                                     int64_t K, int out_fp16, const int64_t *ms, const int64_t *ns,
                                     int64_t count, uint16_t *out)
{
    double t[256];
    decode_table(t);
    for (int64_t i = 0; i < count; ++i) {
        int64_t m = ms[i], n = ns[i];
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) acc += t[a[m * lda + k]] * t[b[n * ldb + k]];
        double y = acc * (double)sa[m] * (double)sb[n];
        if (bias) y += (double)fp8q_oracle_bf16_to_f32(bias[n]);
        out[i] = round_out(y, out_fp16);
    }
}

void fp8q_oracle_gemm_blockwise_at(const uint8_t *a, int64_t lda, const uint8_t *w, int64_t ldw,
                                   const float *sa, int64_t m_pad, const float *sw,
                                   const uint16_t *bias, int64_t K, int out_fp16,
                                   const int64_t *ms, const int64_t *ns, int64_t count,
                                   uint16_t *out)
{
    const int64_t B = 128;
    int64_t kblocks = K / B;
    double t[256];
    decode_table(t);
    for (int64_t i = 0; i < count; ++i) {
        int64_t m = ms[i], n = ns[i];
        double y = 0.0;
        for (int64_t kb = 0; kb < kblocks; ++kb) {
            double p = 0.0;
            for (int64_t k = kb * B; k < (kb + 1) * B; ++k) p += t[a[m * lda + k]] * t[w[n * ldw + k]];
            y += p * (double)sa[kb * m_pad + m] * (double)sw[(n / B) * kblocks + kb];
        }
        if (bias) y += (double)fp8q_oracle_bf16_to_f32(bias[n]);
        out[i] = round_out(y, out_fp16);
    }
}
