// quant.cu -- dynamic activation quantization bf16 -> E4M3 (and the 128x128
// block weight quantizer used to prepare blockwise weights).
//
// Rule (all in fp32, IEEE division, no fast-math):
//   s = max(amax(|x| over the group), eps) / 448
//   q = cvt.rn.satfinite.e4m3(x / s)
// The correctly rounded quotient x / s is formed with Markstein's
// FMA-based correction (quotient2() in quant_common.cuh, shared with the
// GEMM's fused quantization) rather than one IEEE division per element.
// Per-token groups are whole rows ("qinput"/"x_scale" of the channelwise
// path, "Tune FP8 GEMM Triton tiles on L40S..." page, key source snippets);
// per-token-group groups are g consecutive columns, written into a
// row-padded buffer with column-major scales ("Remove per-call padding
// overhead of the FP8 blockwise GEMM" page, key source snippets,
// sglang_per_token_group_quant_fp8_row_padded).
//
// These kernels are HBM-bound streams (2 bytes in, 1 byte out per element):
// 16-byte vector loads and stores, warp-shuffle amax reductions, no shared
// memory staging needed.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "device_common.cuh"
#include "internal.h"
#include "quant_common.cuh"

namespace fp8q {
namespace {

// The scale rounded up to a power of two (an exact 8-bit exponent, UE8M0:
// the scale_ue8m0 option of the group quantizer on the row-padding page,
// key source snippets): clear the fp32 mantissa and, if it was not zero,
// step the exponent up; zero and subnormal scales become 2^-126, the
// smallest normal power of two; +inf stays.
__device__ __forceinline__ float pow2_ceil(float s)
{
    uint32_t b = __float_as_uint(s);
    if (b < 0x00800000u) return __uint_as_float(0x00800000u);
    if (b & 0x007FFFFFu) b = (b & 0x7F800000u) + 0x00800000u;
    return __uint_as_float(b);
}

// Quotients RN(y / s) of four fp32 values, for 2^-90 <= s <= 3e38 with
// r = RN(1 / s): Markstein's correction (see quotient2 in quant_common.cuh)
// gives the correctly rounded quotient whenever the remainder y - q0 * s is
// exact, which holds while it is a normal number.  For |y / s| >= 2^-11 the
// remainder is about 2^-24 |y| >= 2^-35 s >= 2^-125: normal.  Below 2^-11
// a quotient off by an ulp still rounds to the same signed zero in E4M3 (the
// smallest code is 2^-9).  Every y of the group is finite here: for finite
// inputs y is finite or an overflow to +-inf, and an infinite y makes the
// group's scale infinite, which takes the IEEE division instead.
__device__ __forceinline__ uint32_t quant4_f32(const float *y, float s, float r)
{
    const float2 a = quotient2(make_float2(y[0], y[1]), s, r);
    const float2 b = quotient2(make_float2(y[2], y[3]), s, r);
    return cvt_e4m3x2(a.x, a.y) | (cvt_e4m3x2(b.x, b.y) << 16);
}

// Programmatic dependent launch: a quantizer first waits for the previous
// kernel in the stream (so every earlier kernel has completed), then lets the
// next kernel launch -- unless its input is written by no kernel that may
// still be running, in which case it lets the next kernel launch at once and
// waits only before its stores (the host then records the previous launch's
// written ranges with its own, so the next kernel's early reads avoid both).
__device__ __forceinline__ void pdl_enter()
{
    pdl_wait();
    pdl_trigger();
}

// ---------------------------------------------------------------------------
// Per-token quantization: one CTA per row, blockDim.x = T (multiple of 32),
// each thread caches up to VPT 16-element chunks in registers so the row is
// read from HBM exactly once.  Rows longer than T*VPT chunks take the
// two-pass kernel below.
// ---------------------------------------------------------------------------
//
// With `early` set (the host found that no library kernel that may still be
// running on this stream writes x), the kernel lets its successor launch at
// once and loads, reduces and quantizes the row in registers before its
// dependency wait, so all of it overlaps the tail of the previous kernel;
// only the stores of the codes and the scale wait.
template <int VPT>
__global__ void __launch_bounds__(1024) quant_per_token_kernel(const __nv_bfloat16 *__restrict__ x, int64_t ldx,
                                                               uint8_t *__restrict__ xq, float *__restrict__ xs,
                                                               int K, float eps, int early)
{
    __shared__ float warp_max[32];
    if (early)
        pdl_trigger();
    else
        pdl_enter();
    const int64_t row = blockIdx.x;
    const int chunks = K >> 4;
    const __nv_bfloat16 *xr = x + row * ldx;
    Chunk16 c[VPT];
    float m = 0.0f;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int ci = threadIdx.x + v * blockDim.x;
        if (ci < chunks) {
            c[v] = load_chunk(xr + (ci << 4));
            m = chunk_amax(c[v], m);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (blockDim.x > 32) {
        if (lane == 0) warp_max[warp] = m;
        __syncthreads();
        m = (lane < (blockDim.x >> 5)) ? warp_max[lane] : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    }
    const float s = scale_of(m, eps);
    // The codes of chunk v replace its first half (its registers are free).
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int ci = threadIdx.x + v * blockDim.x;
        if (ci < chunks) c[v].lo = quant_chunk(c[v], s);
    }
    if (early) pdl_wait();
    if (threadIdx.x == 0) xs[row] = s;
    uint8_t *qr = xq + row * static_cast<int64_t>(K);
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int ci = threadIdx.x + v * blockDim.x;
        if (ci < chunks) *reinterpret_cast<uint4 *>(qr + (ci << 4)) = c[v].lo;
    }
}

__global__ void __launch_bounds__(1024) quant_per_token_two_pass_kernel(const __nv_bfloat16 *__restrict__ x,
                                                                        int64_t ldx, uint8_t *__restrict__ xq,
                                                                        float *__restrict__ xs, int K, float eps)
{
    __shared__ float warp_max[32];
    pdl_enter();
    const int64_t row = blockIdx.x;
    const int chunks = K >> 4;
    const __nv_bfloat16 *xr = x + row * ldx;
    float m = 0.0f;
    for (int ci = threadIdx.x; ci < chunks; ci += blockDim.x) m = chunk_amax(load_chunk(xr + (ci << 4)), m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) warp_max[warp] = m;
    __syncthreads();
    m = (lane < (blockDim.x >> 5)) ? warp_max[lane] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float s = scale_of(m, eps);
    if (threadIdx.x == 0) xs[row] = s;
    uint8_t *qr = xq + row * static_cast<int64_t>(K);
    for (int ci = threadIdx.x; ci < chunks; ci += blockDim.x)
        *reinterpret_cast<uint4 *>(qr + (ci << 4)) = quant_chunk(load_chunk(xr + (ci << 4)), s);
}

// ---------------------------------------------------------------------------
// Per-token-group quantization into the row-padded buffer.  TPG = g / 16
// threads own one group (16 elements each); the amax is reduced with XOR
// shuffles inside aligned TPG-lane segments.  Consecutive threads walk a row
// left to right, so loads and stores are fully coalesced; the scale of
// (row r, group j) goes to xs[j * m_pad + r].
// ---------------------------------------------------------------------------
//
// Options (the scale_ue8m0 and fuse_silu_and_mul arguments of the group
// quantizer on the row-padding page): UE8M0 rounds each scale up to a power
// of two; SILU reads rows of 2K values and quantizes y = silu(x[k]) *
// x[K + k] (fp32): exp, silu's add and product and the quotients by the
// group scale run on fp32 pairs (the kernel is bound by its instruction
// issue, not by HBM).
// ---------------------------------------------------------------------------
template <int TPG, bool UE8M0, bool SILU>
__global__ void __launch_bounds__(256) quant_group_kernel(const __nv_bfloat16 *__restrict__ x, int64_t ldx,
                                                          uint8_t *__restrict__ xq, float *__restrict__ xs,
                                                          int64_t M, int K, int64_t m_pad, float eps, int early)
{
    // With `early` (no library kernel that may still be running on this
    // stream writes x), the kernel lets its successor launch at once, and
    // each thread's first chunk is loaded and quantized before the
    // dependency wait, which then comes right before its first store.
    bool waited = !early;
    if (early)
        pdl_trigger();
    else
        pdl_enter();
    const int chunks_per_row = K >> 4;
    const int64_t total = M * chunks_per_row;
    // (row, chunk) of chunk index t, advanced by the grid stride without a
    // division per step.
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t stride_rows = stride / chunks_per_row;
    const int stride_ci = static_cast<int>(stride - stride_rows * chunks_per_row);
    int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    int64_t row = t / chunks_per_row;
    int ci = static_cast<int>(t - row * chunks_per_row);
    for (; t - (threadIdx.x & 31) < total;  // whole warps stay in the loop for the shuffles
         t += stride, row += stride_rows, ci += stride_ci) {
        if (ci >= chunks_per_row) {
            ci -= chunks_per_row;
            ++row;
        }
        const bool active = t < total;
        Chunk16 c;
        float y[SILU ? 16 : 1];
        float m = 0.0f;
        if (active) {
            c = load_chunk(x + row * ldx + (ci << 4));
            if constexpr (SILU) {
                const Chunk16 u = load_chunk(x + row * ldx + K + (ci << 4));
                const uint32_t gw[8] = {c.lo.x, c.lo.y, c.lo.z, c.lo.w, c.hi.x, c.hi.y, c.hi.z, c.hi.w};
                const uint32_t uw[8] = {u.lo.x, u.lo.y, u.lo.z, u.lo.w, u.hi.x, u.hi.y, u.hi.z, u.hi.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float2 y2 = silu_mul2(make_float2(bf_lo(gw[i]), bf_hi(gw[i])),
                                                make_float2(bf_lo(uw[i]), bf_hi(uw[i])));
                    y[2 * i] = y2.x;
                    y[2 * i + 1] = y2.y;
                    m = fmaxf(m, fmaxf(fabsf(y2.x), fabsf(y2.y)));
                }
            } else {
                m = chunk_amax(c, 0.0f);
            }
        }
#pragma unroll
        for (int o = TPG >> 1; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (active) {
            float s = scale_of(m, eps);
            if (UE8M0) s = pow2_ceil(s);
            uint4 q;
            if constexpr (SILU) {
                uint32_t w[4];
                if (s >= 0x1p-90f && s <= 3.0e38f) {
                    const float r = 1.0f / s;
#pragma unroll
                    for (int i = 0; i < 4; ++i) w[i] = quant4_f32(y + 4 * i, s, r);
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        w[i] = cvt_e4m3x2(__fdiv_rn(y[4 * i], s), __fdiv_rn(y[4 * i + 1], s)) |
                               (cvt_e4m3x2(__fdiv_rn(y[4 * i + 2], s), __fdiv_rn(y[4 * i + 3], s)) << 16);
                }
                q = make_uint4(w[0], w[1], w[2], w[3]);
            } else {
                q = quant_chunk(c, s);
            }
            if (!waited) {
                pdl_wait();
                waited = true;
            }
            *reinterpret_cast<uint4 *>(xq + row * static_cast<int64_t>(K) + (ci << 4)) = q;
            if ((ci & (TPG - 1)) == 0) xs[static_cast<int64_t>(ci / TPG) * m_pad + row] = s;
        }
    }
    if (!waited) pdl_wait();   // threads without a chunk
}

// ---------------------------------------------------------------------------
// Per-token quantization of many rows: one CTA per row, the row copied whole
// into shared memory by one bulk copy (cp.async.bulk, completion counted in
// bytes on an mbarrier) issued by thread 0.  The CTA holds none of its loads
// in registers, so an SM runs as many rows at once as its shared memory holds
// (24 rows of 4096 values) -- the register-cached kernel above fits 17.  The
// threads then take the row's 8-element units tid, tid + T, ... (16-byte
// shared loads, consecutive threads on consecutive words: conflict-free):
// the amax (bf16 pairs), a CTA reduction, then the codes (8-byte stores,
// coalesced).  The wait is bounded; on a timeout thread 0 still waits
// (bounded) for the copy before the CTA exits.
// ---------------------------------------------------------------------------
constexpr int kBulkMaxK = 16384;  // 32 KB rows: within the default dynamic shared memory

__global__ void __launch_bounds__(256) quant_per_token_bulk_kernel(const __nv_bfloat16 *__restrict__ x, int64_t ldx,
                                                                   uint8_t *__restrict__ xq, float *__restrict__ xs,
                                                                   int K, float eps, unsigned *status)
{
    extern __shared__ __align__(128) uint8_t row_smem[];
    __shared__ uint64_t bar;
    __shared__ float warp_max[8];
    __shared__ int abort_flag;
    const int tid = static_cast<int>(threadIdx.x), T = static_cast<int>(blockDim.x);
    const int lane = tid & 31;
    if (tid == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_enter();
    const int64_t row = blockIdx.x;
    const uint32_t bytes = static_cast<uint32_t>(K) * 2u;
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar, bytes);
        bulk_load_global_hint(row_smem, x + row * ldx, bytes, &bar, policy_evict_first());
    }
    if (!__syncthreads_and(mbar_wait(&bar, 0, &abort_flag, status))) {
        // The copy has not landed: it must before the CTA may exit.
        if (tid == 0) mbar_wait_drain(&bar, 0, status);
        return;
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(row_smem);
    const int units = K >> 3;
    __nv_bfloat162 acc = __float2bfloat162_rn(0.0f);
#pragma unroll 4
    for (int u = tid; u < units; u += T) acc = unit_amax2(src[u], acc);
    float m = fmaxf(__low2float(acc), __high2float(acc));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (T > 32) {
        if (lane == 0) warp_max[tid >> 5] = m;
        __syncthreads();
        m = lane < (T >> 5) ? warp_max[lane] : 0.0f;
        // A full butterfly, so that every lane ends with the row's max.
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    }
    const float sc = scale_of(m, eps);
    if (tid == 0) xs[row] = sc;
    const bool recip = scale_has_reciprocal(sc);
    const float r = recip ? 1.0f / sc : 0.0f;
    uint2 *dst = reinterpret_cast<uint2 *>(xq + row * static_cast<int64_t>(K));
#pragma unroll 4
    for (int u = tid; u < units; u += T) dst[u] = quant_unit8(src[u], sc, r, recip);
}

// ---------------------------------------------------------------------------
// Static per-tensor quantization (one precomputed scale, read from device
// memory): a grid-stride stream over the 16-element chunks of x; the first
// chunk of each row also writes the repeated per-token scale if asked.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) quant_static_kernel(const __nv_bfloat16 *__restrict__ x, int64_t ldx,
                                                           uint8_t *__restrict__ xq, const float *__restrict__ scale,
                                                           float *__restrict__ xs_rep, int64_t M, int K)
{
    pdl_enter();
    const float s = __ldg(scale);
    const int chunks_per_row = K >> 4;
    const int64_t total = M * chunks_per_row;
    for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < total;
         t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t row = t / chunks_per_row;
        const int ci = static_cast<int>(t - row * chunks_per_row);
        *reinterpret_cast<uint4 *>(xq + row * static_cast<int64_t>(K) + (ci << 4)) =
            quant_chunk(load_chunk(x + row * ldx + (ci << 4)), s);
        if (xs_rep != nullptr && ci == 0) xs_rep[row] = s;
    }
}

// ---------------------------------------------------------------------------
// 128 x 128 block weight quantization: one CTA (256 threads) per block.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) quant_weight_block128_kernel(const __nv_bfloat16 *__restrict__ w,
                                                                    uint8_t *__restrict__ wq,
                                                                    float *__restrict__ ws, int64_t K, float eps)
{
    __shared__ float warp_max[8];
    pdl_enter();
    const int64_t bn = blockIdx.y, bk = blockIdx.x;
    // 128 rows x 8 chunks of 16; thread t handles chunks t, t + 256, ...
    Chunk16 c[4];
    float m = 0.0f;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const int idx = threadIdx.x + v * 256;
        const int r = idx >> 3, cc = idx & 7;
        c[v] = load_chunk(w + (bn * 128 + r) * K + bk * 128 + cc * 16);
        m = chunk_amax(c[v], m);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = m;
    __syncthreads();
    m = warp_max[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) m = fmaxf(m, warp_max[i]);
    const float s = scale_of(m, eps);
    if (threadIdx.x == 0) ws[bn * (K >> 7) + bk] = s;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const int idx = threadIdx.x + v * 256;
        const int r = idx >> 3, cc = idx & 7;
        *reinterpret_cast<uint4 *>(wq + (bn * 128 + r) * K + bk * 128 + cc * 16) = quant_chunk(c[v], s);
    }
}

// Launch with programmatic stream serialization so the kernel's launch
// overlaps the tail of the previous kernel in the stream (each kernel waits
// for it with griddepcontrol.wait before touching global memory).
template <typename... Params, typename... Args>
cudaError_t launch_pdl_smem(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                            Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}

template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, cudaStream_t st, Args... args)
{
    return launch_pdl_smem(kernel, grid, block, 0, st, args...);
}

// Threads for a bulk row of K values: about 8 units each, whole warps, 32 to
// 256 (64 for rows of 4096).
cudaError_t launch_per_token_bulk(const void *x, int64_t M, int64_t K, int64_t ldx, void *xq, float *xs, float eps,
                                  unsigned *status, cudaStream_t st)
{
    int threads = (static_cast<int>(K >> 3) / 8 + 31) / 32 * 32;
    if (threads < 32) threads = 32;
    if (threads > 256) threads = 256;
    return launch_pdl_smem(quant_per_token_bulk_kernel, dim3(static_cast<unsigned>(M)), dim3(threads),
                           static_cast<size_t>(K) * 2, st, static_cast<const __nv_bfloat16 *>(x), ldx,
                           static_cast<uint8_t *>(xq), xs, static_cast<int>(K), eps, status);
}

template <int VPT>
cudaError_t launch_per_token(const void *x, int64_t M, int K, int64_t ldx, void *xq, float *xs, float eps, int threads,
                             bool early, cudaStream_t st)
{
    return launch_pdl(quant_per_token_kernel<VPT>, dim3(static_cast<unsigned>(M)), dim3(threads), st,
                      static_cast<const __nv_bfloat16 *>(x), ldx, static_cast<uint8_t *>(xq), xs, K, eps,
                      early ? 1 : 0);
}

}  // namespace

// Row counts from which per-token quantization is bandwidth-bound rather
// than latency-bound (several rows per SM), and from which the rows an SM
// keeps in flight decide its speed: the bulk kernel, measured over inputs
// larger than L2, 15.5 against 20.5 us at 8192 x 4096 and 9.5 against 10.6 us
// at 4096 x 4096, but 7.1 against 6.4 us at 2048 rows, where the register-
// cached kernel already holds every row in flight at once.
constexpr int64_t kManyRows = 1024;
constexpr int64_t kBulkRows = 4096;

cudaError_t launch_quant_per_token(const void *x, int64_t M, int64_t K, int64_t ldx, void *xq, float *xs, float eps,
                                   unsigned *status, cudaStream_t st, bool *early_trigger)
{
    if (early_trigger != nullptr) *early_trigger = false;
    if (M >= kBulkRows && K <= kBulkMaxK) return launch_per_token_bulk(x, M, K, ldx, xq, xs, eps, status, st);
    const int chunks = static_cast<int>(K >> 4);
    // Decode-size M (latency-bound, one CTA per row): one 16-element chunk
    // per thread where possible, the shortest dependent chain.  Many rows
    // (bandwidth-bound): four chunks per thread, so each thread keeps 128
    // bytes of loads in flight.  Whole warps, at most 1024 threads; rows
    // longer than 4 chunks per thread take the two-pass kernel.
    const int per_thread = M >= kManyRows ? 4 : 1;
    int threads = (chunks + 32 * per_thread - 1) / (32 * per_thread) * 32;
    if (threads > 1024) threads = 1024;
    const int vpt = (chunks + threads - 1) / threads;
    // The rows may be read before the dependency wait unless a library
    // kernel that may still be running on this stream writes them.
    const size_t xbytes = (static_cast<size_t>(M - 1) * static_cast<size_t>(ldx) + static_cast<size_t>(K)) * 2u;
    const bool early = !last_launch_writes_overlap(st, x, xbytes);
    if (early_trigger != nullptr) *early_trigger = early && vpt <= 4;
    switch (vpt) {
        case 1: return launch_per_token<1>(x, M, static_cast<int>(K), ldx, xq, xs, eps, threads, early, st);
        case 2: return launch_per_token<2>(x, M, static_cast<int>(K), ldx, xq, xs, eps, threads, early, st);
        case 3: return launch_per_token<3>(x, M, static_cast<int>(K), ldx, xq, xs, eps, threads, early, st);
        case 4: return launch_per_token<4>(x, M, static_cast<int>(K), ldx, xq, xs, eps, threads, early, st);
        default:
            return launch_pdl(quant_per_token_two_pass_kernel, dim3(static_cast<unsigned>(M)), dim3(1024), st,
                              static_cast<const __nv_bfloat16 *>(x), ldx, static_cast<uint8_t *>(xq), xs,
                              static_cast<int>(K), eps);
    }
}

namespace {

// Grid of a grid-stride quantizer over M * K / 16 chunks (256 threads).
dim3 stream_grid(int64_t M, int64_t K, int num_sms)
{
    const int64_t total = M * (K >> 4);
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms > 0 ? num_sms : 148) * 64;
    if (blocks > cap) blocks = cap;
    return dim3(static_cast<unsigned>(blocks));
}

template <bool UE8M0, bool SILU>
cudaError_t launch_group(const void *x, int64_t M, int64_t K, int64_t ldx, int group, void *xq, float *xs,
                         int64_t m_pad, float eps, int num_sms, cudaStream_t st, bool *early_trigger)
{
    const auto *xb = static_cast<const __nv_bfloat16 *>(x);
    auto *q = static_cast<uint8_t *>(xq);
    const dim3 g = stream_grid(M, K, num_sms), b(256);
    const int k = static_cast<int>(K);
    // The rows (2K values each with the silu input) may be read before the
    // dependency wait unless a library kernel that may still be running
    // writes them.
    const size_t xbytes =
        (static_cast<size_t>(M - 1) * static_cast<size_t>(ldx) + static_cast<size_t>(SILU ? 2 * K : K)) * 2u;
    const int e = last_launch_writes_overlap(st, x, xbytes) ? 0 : 1;
    if (early_trigger != nullptr) *early_trigger = e != 0;
    switch (group) {
        case 16: return launch_pdl(quant_group_kernel<1, UE8M0, SILU>, g, b, st, xb, ldx, q, xs, M, k, m_pad, eps, e);
        case 32: return launch_pdl(quant_group_kernel<2, UE8M0, SILU>, g, b, st, xb, ldx, q, xs, M, k, m_pad, eps, e);
        case 64: return launch_pdl(quant_group_kernel<4, UE8M0, SILU>, g, b, st, xb, ldx, q, xs, M, k, m_pad, eps, e);
        default: return launch_pdl(quant_group_kernel<8, UE8M0, SILU>, g, b, st, xb, ldx, q, xs, M, k, m_pad, eps, e);
    }
}

}  // namespace

cudaError_t launch_quant_group(const void *x, int64_t M, int64_t K, int64_t ldx, int group, void *xq, float *xs,
                               int64_t m_pad, float eps, int num_sms, cudaStream_t st, bool ue8m0, bool silu_and_mul,
                               bool *early_trigger)
{
    bool et = false;
    cudaError_t e;
    if (silu_and_mul)
        e = ue8m0 ? launch_group<true, true>(x, M, K, ldx, group, xq, xs, m_pad, eps, num_sms, st, &et)
                  : launch_group<false, true>(x, M, K, ldx, group, xq, xs, m_pad, eps, num_sms, st, &et);
    else
        e = ue8m0 ? launch_group<true, false>(x, M, K, ldx, group, xq, xs, m_pad, eps, num_sms, st, &et)
                  : launch_group<false, false>(x, M, K, ldx, group, xq, xs, m_pad, eps, num_sms, st, &et);
    if (early_trigger != nullptr) *early_trigger = et;
    return e;
}

cudaError_t launch_quant_static(const void *x, int64_t M, int64_t K, int64_t ldx, const float *scale, void *xq,
                                float *xs_rep, int num_sms, cudaStream_t st)
{
    return launch_pdl(quant_static_kernel, stream_grid(M, K, num_sms), dim3(256), st,
                      static_cast<const __nv_bfloat16 *>(x), ldx, static_cast<uint8_t *>(xq), scale, xs_rep, M,
                      static_cast<int>(K));
}

cudaError_t launch_quant_weight_block128(const void *w, int64_t N, int64_t K, void *wq, float *ws, float eps,
                                         cudaStream_t st)
{
    dim3 grid(static_cast<unsigned>(K / 128), static_cast<unsigned>(N / 128));
    return launch_pdl(quant_weight_block128_kernel, grid, dim3(256), st, static_cast<const __nv_bfloat16 *>(w),
                      static_cast<uint8_t *>(wq), ws, K, eps);
}

}  // namespace fp8q
