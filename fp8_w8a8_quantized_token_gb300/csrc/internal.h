// internal.h -- declarations shared by the library's translation units
// (host side only; no CUDA device code here).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fp8q.h"

namespace fp8q {

// ---- quantizers (quant.cu) ------------------------------------------------
// `status`: the device status word, where the many-row kernel's bounded
// wait records a timeout.
// `early_trigger` (may be null) is set when the kernel lets its successor
// start before its own dependency wait (the record must then keep the
// previous launch's ranges).
cudaError_t launch_quant_per_token(const void *x, int64_t M, int64_t K, int64_t ldx, void *xq, float *xs, float eps,
                                   unsigned *status, cudaStream_t st, bool *early_trigger = nullptr);
cudaError_t launch_quant_group(const void *x, int64_t M, int64_t K, int64_t ldx, int group, void *xq, float *xs,
                               int64_t m_pad, float eps, int num_sms, cudaStream_t st, bool ue8m0 = false,
                               bool silu_and_mul = false, bool *early_trigger = nullptr);
cudaError_t launch_quant_static(const void *x, int64_t M, int64_t K, int64_t ldx, const float *scale, void *xq,
                                float *xs_rep, int num_sms, cudaStream_t st);
cudaError_t launch_quant_weight_block128(const void *w, int64_t N, int64_t K, void *wq, float *ws, float eps,
                                         cudaStream_t st);

// ---- GEMM (gemm_*.cu) -------------------------------------------------------
// A GEMM launch as the planner decided it.
struct GemmLaunch {
    bool swap_ab;      // true: MMA A = 128 weight rows, MMA N = tokens
    int mma_n;         // MMA N extent (tile width along the B operand)
    int split;         // K-split count = cluster size
    int grid;          // CTAs
    int stages;        // pipeline depth the instantiation uses
    bool pair;         // non-swapped channelwise, split 1: 2-CTA clusters on adjacent token tiles
    bool two_sm;       // the pair computes 256-token tiles with 2-CTA MMAs (always with pair)
    bool stream_k;     // swapped tiles: equal shares of (tile, K block) pairs per CTA, split 1
    bool wide;         // non-swapped channelwise: stages of two K blocks (fp8q_plan::kb_per_stage 2)
};

struct GemmProblem {
    int64_t M, N, K;
    int64_t m_pad;          // blockwise: leading dimension of the scale columns
    const void *a;          // e4m3 activations, row stride K (fused_quant: bf16, row stride lda)
    int64_t lda;            // fused_quant: row stride of the bf16 activations (elements)
    const void *w;          // e4m3 weights [N, K] with row stride ldw
    int64_t ldw;
    const float *a_scale;   // channelwise [M]; blockwise column-major [K/128][m_pad]
    const float *w_scale;   // channelwise [N]; blockwise [N/128][K/128]
    const void *bias;       // bf16 [N] or null
    void *out;              // [M, N]
    bool out_fp16;
    bool blockwise;
    bool preload;           // weights may be read before the dependency wait
    bool fused_quant;       // blockwise: a is bf16, quantized inside the GEMM (group 128, eps)
    bool w16;               // channelwise weight-only FP8: a is bf16 (row stride lda), no a_scale
    float eps;              // fused_quant: amax floor of the group scales
    void *ws;               // split-K workspace (16-byte aligned) or null
    size_t ws_bytes;        // its size; smaller than the schedule needs = not used
};

// Bytes of split-K workspace a schedule uses (0 when K is not split or the
// partial tiles are smaller than 128 x 128 floats): one slot of 128 x mma_n
// fp32 partial sums per CTA.
size_t plan_workspace_bytes(int64_t M, int64_t N, int swap_ab, int mma_n, int split_k);

// Workspace of a stream-K launch of `grid` CTAs: one slot of 128 x mma_n
// floats per CTA, then one 32-bit flag per CTA (zero between launches).
size_t stream_k_workspace_bytes(int grid, int mma_n);

// The K-split schedule of a stream-K plan's tiles (the generic rule's
// split: 2, 4 or 8 while the CTAs fill at most half the SMs).
void plan_without_stream_k(int64_t M, int64_t N, int64_t K, int blockwise, int num_sms, fp8q_plan *pl);

// Launchers return cudaSuccess or the launch error; a tensor map the driver
// rejects is reported as cudaErrorInvalidValue.

cudaError_t launch_gemm_channelwise(const GemmProblem &p, const GemmLaunch &l, unsigned *status, cudaStream_t st);
cudaError_t launch_gemm_blockwise(const GemmProblem &p, const GemmLaunch &l, unsigned *status, cudaStream_t st);

// Pipeline depth of the instantiation serving (swap_ab, mma_n): the
// shared-memory ring holds `stages` slots of 16 KB (A) + mma_n*128 B (B).
// The 16- and 32-token decode tiles keep their footprint near 100 KB so two
// CTAs fit on one SM: a layer's GEMM can then start (prologue, L2 weight
// prefetch) on SMs still running the previous layer's tail.
constexpr int stages_for(bool swap_ab, int mma_n)
{
    return swap_ab ? (mma_n == 16 ? 5 : mma_n == 32 ? 4 : mma_n == 64 ? 7 : 4)
                   : (mma_n == 256 ? 4 : mma_n == 128 ? 6 : 8);
}

// Ring depth of the stream-K instantiations (16- and 32-token tiles).  A
// stream-K grid has at most one CTA per SM, so the ring can take the shared
// memory two split-K CTAs would share: 10 slots of 16 KB + 2 KB, 9 of
// 16 KB + 4 KB.  Measured on gate_up at M = 1: 21.5 us with the 5-slot ring
// of the 16-token split-K instantiation, 19.0 us with 8 slots.
constexpr int stream_k_stages(int mma_n) { return mma_n == 16 ? 10 : 9; }

// Ring depth of the fused-quantization instantiation (blockwise, 16-token
// tiles): 4 slots of 16 KB + 2 KB plus a 4-slot bf16 staging ring of 4 KB
// keep it near 100 KB, so two CTAs still fit on one SM.
constexpr int kFusedQuantStages = 4;
// (32-token tiles: 3 slots of 16 KB + 4 KB and a 3-slot staging ring of 8 KB
// keep the CTA near 105 KB as well.)
constexpr int kFusedQuantStages32 = 3;
// Weight-only FP8 for at most this many tokens runs as matrix-vector
// products on the CUDA cores (w8a16_gemv.cu), above it on the tensor cores
// (with three or four tokens the CUDA-core kernel measured slower).
constexpr int kW16GemvMaxM = 2;
cudaError_t launch_w8a16_gemv(const void *x, int64_t ldx, const void *w, int64_t ldw, const float *w_scale,
                              const void *bias, void *out, int64_t M, int64_t N, int64_t K, bool out_fp16,
                              cudaStream_t st);
// True while a schedule override (fp8q_set_plan_override / FP8Q_PLAN) is set.
bool plan_override_active();
// The channelwise and blockwise linears for one token with K <= 12288 run
// as one launch with the activation quantization fused (linear_gemv.cu),
// unless a schedule override is set.  Each warp of the matrix-vector CTA
// owns ceil(K / 4096) 512-byte chunks of a row per group and requests them
// together.  Measured on GB300 this is faster than the quantizer +
// tensor-core GEMM at K = 3072, 4096, 7168 and 12288 (channelwise: for
// small layers); with two tokens it was slower.
inline int gemv_chunks_per_warp(int64_t K) { return static_cast<int>((K + 4095) / 4096); }
// Channelwise: only layers of at most 4096 x 4096 weights.  Once the
// quantizer lets the GEMM launch early, the two kernels are faster on
// larger layers (qkv 6144 x 4096: 7.3 against 8.1 us; down, gate_up).
inline bool linear_gemv_fits(int64_t M, int64_t N, int64_t K)
{
    return M == 1 && K <= 12288 && N * K <= 4096 * 4096;
}
inline bool linear_blk_gemv_fits(int64_t M, int64_t K) { return M == 1 && K <= 12288; }
cudaError_t launch_linear_blk_gemv(const void *x, const void *w, const float *w_scale, const void *bias, void *out,
                                   void *xq, float *xs, int64_t m_pad, int64_t N, int64_t K, float eps, bool out_fp16,
                                   cudaStream_t st);
cudaError_t launch_linear_pt_gemv(const void *x, const void *w, int64_t ldw, const float *w_scale, const void *bias,
                                  void *out, void *xq, float *xs, int64_t M, int64_t N, int64_t K, float eps,
                                  bool out_fp16, cudaStream_t st);
// Ring stages of the double-K-block (WIDE) narrow channelwise tiles: stages
// of 32 KB of activations + BN x 256 bytes of weights, about 190 KB.
constexpr int wide_stages(int mma_n) { return mma_n == 128 ? 3 : mma_n == 64 ? 4 : 5; }

// Depth of the MMA ring of the weight-only FP8 (W16) instantiations: per
// stage a bf16 A tile in tensor memory (64 columns) and the token tile's bf16
// activations in shared memory; the E4M3 weight and bf16 activation tiles
// stream through a deeper landing ring of their own (gemm_kernel.cuh).
constexpr int kW16Stages = 3;

// Ring depth of the 2-CTA MMA instantiation (each slot: 16 KB of tokens +
// 16 KB, the CTA's half, of weight rows).
constexpr int kTwoSmStages = 6;

// True if an instantiation exists for (swap_ab, mma_n).
constexpr bool gemm_shape_supported(bool swap_ab, int mma_n)
{
    return swap_ab ? (mma_n == 16 || mma_n == 32 || mma_n == 64 || mma_n == 128)
                   : (mma_n == 32 || mma_n == 64 || mma_n == 128 || mma_n == 256);
}

// ---- tensor maps (host_util.cu) ------------------------------------------------
// 2-D tensor map over a row-major matrix of `rows` x `cols` elements with a
// row stride of `row_bytes`, box = box_cols x box_rows, the given shared-
// memory swizzle.  Returns false if the driver rejects it.
bool make_tmap_2d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, uint64_t cols, uint64_t rows,
                  uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swizzle);

// ---- device status word (host_util.cu) --------------------------------------
unsigned *device_status_ptr();   // of the current device, or null
// Per-CTA phase timestamps of a trace build (-DFP8Q_TRACE) and, through
// *stages, the per-ring-stage stamps of the launch's CTA 0; null otherwise.
unsigned long long *trace_buffer(unsigned long long **stages);
// Ring stages of CTA 0 whose stamps a trace build keeps.
constexpr int kTraceStages = 128;
// Weight K blocks each GEMM CTA prefetches into L2 before its dependency
// wait: 16 for swapped (decode) tiles -- blockwise ones only while the grid
// is at most 1.5 CTAs per SM -- and none for non-swapped tiles;
// FP8Q_PREFETCH_KB overrides the rule at start-up (0 disables).  Measured on
// GB300 over rotating weight copies (more than L2), two interleaved runs
// each: the prefetch shortens o_proj decode from 6.72 to 6.22 us (128 CTAs,
// 8 K blocks each) and blockwise 3072 x 12288 decode from 11.1 to 10.55 us
// (192 CTAs), but lengthens blockwise 4096 x 7168 decode (256 CTAs, 9.08 ->
// 9.25 us) and every non-swapped size by 1-6 % (o_proj M = 512: 12.56 ->
// 12.85 us; down M = 256: 19.9 -> 21.2 us).
int prefetch_kblocks(bool swapped, bool blockwise, int grid);
// E4M3 operand [rows, K] (K % 128 == 0, row stride row_bytes) as a 3-D
// tensor (128 bytes, rows, K / 128) whose boxes of 128 bytes x box_rows x 2
// hold two consecutive 128-wide K blocks (each 128-byte swizzled, one after
// the other): the double-K-block stages of the non-swapped channelwise
// tiles.  A box starting at the last K block of an odd count reads the
// missing second block as zeros.
bool make_tmap_3d_kblocks(CUtensorMap *map, const void *base, uint64_t K, uint64_t rows, uint64_t row_bytes,
                          uint32_t box_rows);
// Split-K partial sums through the caller's workspace (global memory)
// instead of distributed shared memory: off unless FP8Q_WORKSPACE_EXCHANGE=1
// at start-up.  On the GB300s measured, reading partials that other SMs of
// the cluster have just written through global memory moved 10-30 GB/s per
// SM, below the distributed-shared-memory exchange at every schedule, so by
// default the library asks for no workspace and ignores one passed to it.
bool workspace_exchange_enabled();

// Per-stream record of the byte ranges that the library kernels which may
// still be running when the next one starts write.  With programmatic
// dependent launch a kernel triggers its dependents after its own
// dependency wait, so normally only the most recent launch can still be
// running, and its ranges (up to three) are recorded.  A quantizer whose
// input no earlier kernel on the stream is writing triggers at its start
// instead (keep_previous): the launch before it may then still run as well,
// and its ranges are kept in the record too.  A kernel reads before its own
// dependency wait (a GEMM its weights, a quantizer its input) only what
// overlaps none of the recorded ranges.
void note_launch_writes(cudaStream_t st, const void *base, size_t bytes, const void *base2 = nullptr,
                        size_t bytes2 = 0, const void *base3 = nullptr, size_t bytes3 = 0,
                        bool keep_previous = false);
bool last_launch_writes_overlap(cudaStream_t st, const void *base, size_t bytes);
int current_device_sms();        // SM count of the current device (cached)

}  // namespace fp8q

namespace fp8q {
// Copies the current device's status word to *value (synchronizing `st`);
// reset clears it afterwards.
cudaError_t read_status_word(unsigned *value, bool reset, cudaStream_t st);
}  // namespace fp8q
