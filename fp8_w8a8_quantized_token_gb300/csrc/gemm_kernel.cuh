// gemm_kernel.cuh -- the scaled FP8 (E4M3 x E4M3 -> fp32) GEMM for sm_103a.
//
// Computes, for the channelwise scheme ("Tune FP8 GEMM Triton tiles on L40S
// and enable by default" page, key source snippets: fp8_scaled_mm)
//     out[m,n] = cvt( acc[m,n] * a_scale[m] * w_scale[n] (+ bias[n]) ),
//     acc[m,n] = sum_k a[m,k] * w[n,k]
// and for the blockwise scheme ("Remove per-call padding overhead of the FP8
// blockwise GEMM" page, key source snippets: fp8_blockwise_scaled_mm)
//     out[m,n] = cvt( sum_kb P_kb[m,n] * a_scale[kb*m_pad + m]
//                                      * w_scale[(n/128)*(K/128) + kb] (+ bias[n]) )
// where P_kb is the product over the 128 k of block kb.
//
// Structure (one CTA, warp-specialised):
//   warp 0        TMA producer: streams 128-byte-wide K slices of the A and
//                 B operand tiles (and, blockwise, the tile's activation
//                 scales of that K block) into a STAGES-deep shared-memory
//                 ring, 128-byte swizzled.
//   warp 1        TMEM allocator + MMA issuer: one thread issues four
//                 tcgen05.mma.kind::f8f6f4 (K = 32 each) per ring slot into
//                 a TMEM accumulator (M = 128 lanes x N = BN fp32 columns)
//                 and commits completion to mbarriers.
//   warps 2..     epilogue: tcgen05.ld the accumulator, apply the scales
//                 (blockwise: after every K block, "promotion" into fp32
//                 registers), add the bias, convert and store.
// TMEM holds two accumulator slots so MMA on the next tile (channelwise) or
// the next K block (blockwise) overlaps the epilogue of the current one.
//
// Orientation.  The MMA's M side is always 128 rows of the A operand.
//   SWAP = true  (decode-size M): A = 128 weight rows, B = BN tokens;
//                 TMEM lane = output column n, TMEM column = token m.
//   SWAP = false (prefill M):      A = 128 tokens, B = BN weight rows;
//                 TMEM lane = token m, TMEM column = output column n.
//
// 2-CTA MMA (TWO_SM, non-swapped channelwise, split 1).  Two CTAs of a
// 2-CTA cluster ("a pair") take the token tiles 2t and 2t+1 against the
// same BN weight rows and compute the 256-token x BN tile with
// tcgen05.mma.cta_group::2 (M = 256) issued by the even CTA: each CTA loads
// (plain TMA into its own shared memory) only its own 128 tokens and its
// half of the BN weight rows, so every weight byte leaves L2 once per pair
// and neither CTA holds a duplicate copy.  All of a slot's loads complete on
// the even CTA's full barrier, and the even CTA's commits arrive on both
// CTAs' empty and accumulator barriers.  Each CTA's TMEM holds its own 128
// accumulator rows; both epilogues release the even CTA's accumulator slot.
//
// Split-K.  split > 1 launches thread-block clusters of `split` CTAs that
// share one output tile and take consecutive ranges of K blocks.  Each CTA
// stages its fp32 partial tile in its own (then idle) shared-memory ring;
// the tile's outputs are divided among the ranks, and each rank sums its
// share over all ranks' partials in rank order (deterministic).  The
// partials of the other ranks reach the owner in one of two ways:
//   * a caller-provided global workspace (GemmArgs::ws): each CTA writes the
//     parts of its partial tile that other ranks own into its own slot
//     (coalesced stores that stay in L2), one cluster barrier publishes
//     them, and each owner reads its share of every slot;
//   * no workspace: through distributed shared memory (the non-swapped
//     orientation pulls its share from every CTA after a cluster barrier,
//     the swapped orientation pushes each rank's rows into that rank's
//     receive buffer with bulk copies).
// Both ways add the same values in the same order, so they give identical
// results.
//
// Stream-K (swapped channelwise or blockwise tiles, p.stream_k).  The
// (tile, K block) pairs are numbered tile-major, T = num_tiles * num_kb of
// them, and CTA c of G takes the pairs [c*T/G, (c+1)*T/G): every CTA streams
// the same number of weight blocks whatever the tile count.  A CTA's range
// is cut at tile boundaries into work units (tile, K blocks [kb0, kb1)); a
// unit covering the whole tile is stored as usual.  Only a CTA's first unit
// can start inside a tile: it writes its fp32 partial tile (raw MMA sums;
// blockwise: the promoted sums) to its workspace slot and publishes it with
// a release store of its flag.  The unit holding the tile's first K block
// (the last unit of its CTA, which therefore reaches the tile after the
// other CTAs have published theirs) waits for the flags of the following
// CTAs whose ranges start inside the tile (acquire loads, bounded), adds
// their partials in increasing K order (a fixed order: deterministic),
// clears the flags for the next launch and stores the tile.  Waits only go
// to higher CTA indices, so they cannot form a cycle.
//
// Every mbarrier wait is bounded (device_common.cuh); a wait that runs out
// records a timeout in the status word and all roles wind down, waiting
// (bounded) for their in-flight TMA copies and MMAs before TMEM is freed.
#pragma once

#include "device_common.cuh"
#include "internal.h"
#include "quant_common.cuh"

namespace fp8q {

struct GemmArgs {
    int M, N, K;
    int num_kb;            // ceil(K / 128)
    int m_tiles, n_tiles;  // tile counts along tokens and output columns
    int num_tiles;
    int split;             // CTAs per cluster along K
    int group;             // tile rasterisation group
    int raster_b;          // 1: groups of B-operand tiles sweep the A tiles (else the reverse)
    int pair;              // 1: 2-CTA MMA pairs (TWO_SM): num_tiles counts tile pairs
    const float *a_scale;
    const float *w_scale;
    const __nv_bfloat16 *bias;
    void *out;
    long long ldo;
    unsigned *status;
    unsigned long long *trace;  // per-CTA phase timestamps (trace builds only), or null
    int prefetch_kb;            // weight K blocks per CTA prefetched into L2 before the dependency wait
    int preload;                // 1: load the first tile's weight slices before the dependency wait
    float eps;                  // fused quantization: the amax floor of the group scales
    const __nv_bfloat16 *x;     // fused quantization: bf16 activations [M, K]
    long long ldx;              //   and their row stride (elements)
    float *ws;                  // split-K workspace: split slots of 128 x BN floats per cluster, or null;
                                //   stream-K: one slot of 128 x BN floats per CTA
    int stream_k;               // 1: stream-K (swapped tiles, one CTA per cluster, see below)
    unsigned *sk_flags;         // stream-K: one flag per CTA after the slots, 1 = its partial is published
    unsigned long long *trace_stages;  // trace builds: CTA 0's per-stage stamps (null otherwise)
};

// Phase timestamps of a trace build (-DFP8Q_TRACE): kTraceSlots 64-bit
// %globaltimer values per CTA, written by one designated thread per phase.
constexpr int kTraceSlots = 16;
enum TracePhase {
    kTrEntry = 0, kTrPrologue, kTrPdlWait, kTrFirstTma, kTrFirstMma, kTrLastCommit, kTrEpiFull, kTrEpiDone,
    kTrCluster1, kTrReduced, kTrCluster2, kTrExit, kTrPreloaded, kTrTmemAlloc, kTrSmid = 14, kTrRank = 15
};
#ifdef FP8Q_TRACE
#define FP8Q_TRACE_AT(p, phase)                                                                   \
    do {                                                                                          \
        if ((p).trace != nullptr && blockIdx.x < 4096)                                            \
            (p).trace[blockIdx.x * kTraceSlots + (phase)] = globaltimer_ns();                     \
    } while (0)
// Per-ring-stage stamps of CTA 0 (stage k in issue order, k < kTraceStages):
// event 0 loads issued, 1 MMA issuer 0 saw the stage full, 2 its commit
// issued, 3 the producer began waiting for the stage to be empty.
#define FP8Q_TRACE_STAGE(p, event, k)                                                             \
    do {                                                                                          \
        if ((p).trace_stages != nullptr && blockIdx.x == 0 && (k) < kTraceStages)                 \
            (p).trace_stages[(k) * 4 + (event)] = globaltimer_ns();                               \
    } while (0)
#else
#define FP8Q_TRACE_STAGE(p, event, k) \
    do {                              \
    } while (0)
#define FP8Q_TRACE_AT(p, phase) \
    do {                        \
    } while (0)
#endif

template <bool SWAP, int BN, int STAGES, bool BLOCKWISE, bool TWO_SM = false, bool FQ = false, bool W16 = false,
          bool WIDE = false>
struct GemmCfg {
    static constexpr int kEpiWarps = BN > 128 ? 8 : 4;
    static constexpr int kColGroups = kEpiWarps / 4;
    static constexpr int kCols = BN / kColGroups;  // TMEM columns per epilogue thread
    // MMA-issuing warps.  Measured on GB300: one issuing thread completes a
    // 128 x N x 32 MMA chain no faster than about one MMA per 27 ns whatever
    // N (up to 64), while the tensor pipe needs only about N/256 of 66 ns
    // for it; a second issuing warp with its own accumulator overlaps the
    // first (about 1.4x at N = 16; no gain at N >= 128, where the pipe is
    // the limit).  Channelwise tiles narrower than 256 columns therefore
    // spread each K block's four MMAs over 2 warps, each accumulating into
    // its own TMEM columns; the epilogue adds the two accumulators.  (More
    // issuers would add warps: 2 CTAs of 7 warps still fit one SM's register
    // file, which lets the next launch's CTAs load their weights while this
    // launch's CTAs finish.)
    static constexpr int kIssuers = (BLOCKWISE || TWO_SM || BN >= 256) ? 1 : 2;
    // Stream-K: swapped E4M3 tiles of 16 and 32 tokens (not the fused-
    // quantization or weight-only variants, whose extra warps walk tiles on
    // their own; wider tiles hold rows of 64 or 128 floats per thread, and the
    // hand-over code would cost them registers they do not have).
    static constexpr bool kStreamK = SWAP && BN <= 32 && !TWO_SM && !FQ && !W16;
    static constexpr int kSlotCols = kIssuers * BN;  // TMEM columns per accumulator slot
    // Register split (blockwise 256-column tiles): each epilogue thread
    // promotes 128 accumulator columns every K block, in rounds of (TMEM
    // load, wait, packed FMAs) whose latencies add up; with 10 warps, three
    // share a sub-partition and cap a thread at 168 registers, which allows
    // only 16 columns per round (8 rounds per K block, longer than the
    // block's MMA).  Instead the CTA runs 12 warps: warpgroup 0 = producer,
    // MMA issuer and two idle warps; warpgroups 1 and 2 = the eight epilogue
    // warps.  Launched at kLaunchRegs registers per thread, warpgroup 0 gives
    // registers back (setmaxnreg.dec to kLowRegs) and the epilogue warpgroups
    // take them (setmaxnreg.inc to kHighRegs), enough for 64 columns per
    // round.  kLowRegs * 128 + kHighRegs * 256 == kLaunchRegs * kThreads, and
    // the host checks the kernel's register count before it launches.
    static constexpr bool kRegSplit = BLOCKWISE && !SWAP && BN == 256 && !TWO_SM && !FQ && !W16;
    static constexpr int kIdleWarps = kRegSplit ? 2 : 0;
    static constexpr int kLaunchRegs = 168, kLowRegs = 72, kHighRegs = 216;
    static constexpr int kEpiWarp0 = 1 + kIssuers + kIdleWarps;   // first epilogue warp
    // FQ: two warps after the epilogue warps quantize the activation tiles.
    static constexpr int kQuantWarps = FQ ? 2 : 0;
    static constexpr int kQuantWarp0 = kEpiWarp0 + kEpiWarps;
    // W16 (weight-only FP8, bf16 activations; swapped channelwise tiles):
    // eight warps after the epilogue warps (two per TMEM lane quarter, one
    // per 64-wide K half of a block) convert each landed E4M3 weight tile to
    // bf16 (exact) into tensor memory, the A operand of kind::f16 MMAs.
    static constexpr int kConvWarps = W16 ? 8 : 0;
    static constexpr int kConvWarp0 = kQuantWarp0 + kQuantWarps;
    static constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps + kQuantWarps + kConvWarps);
    // CTAs per SM the register allocation must allow.  The fused-quantization
    // tiles run clusters of up to 8 CTAs along K: with one CTA per SM, few
    // such clusters fit in a GPC at once (the 32-token tile at 139 registers
    // took 48 us for blockwise 4096 x 7168 at M = 32, against 11.5 us for the
    // two-kernel path), so they are held to two CTAs per SM.
    static constexpr int kMinBlocks = FQ ? 2 : 1;
    static_assert(!kRegSplit || (kThreads == 384 && kEpiWarp0 == 4 && kEpiWarps == 8 &&
                                 kLowRegs * 128 + kHighRegs * 256 == kLaunchRegs * kThreads),
                  "register split: warpgroup 0 low, warpgroups 1-2 high, same total as at launch");
    // WIDE (non-swapped channelwise single-CTA tiles, K a multiple of 128,
    // no K split): each ring stage holds two consecutive 128-wide K blocks,
    // loaded by one 3-D TMA box per operand.  Measured on GB300, the TMA
    // issue of one thread costs ~85 ns per box whatever its size (16 or
    // 32 KB) plus ~70 ns per stage, which paced the 128 x 64 tiles at
    // ~290 ns per K block with or without their MMAs; two blocks per box
    // halve both.
    static constexpr int kSub = WIDE ? 2 : 1;            // K blocks per stage
    // K steps of one stage: 4 MMAs of K = 32 per K block (E4M3) or, W16, 8
    // of K = 16 (bf16).
    static constexpr int kKSteps = W16 ? 8 : 4 * kSub;
    static constexpr int kEpiThreads = 32 * kEpiWarps;
    static constexpr int kTokTile = SWAP ? BN : 128;     // tokens per tile
    static constexpr int kColTile = SWAP ? 128 : BN;     // output columns per tile
    // A operand slot: 128 rows x 128 K of E4M3.  (W16: none; the bf16 A
    // tiles are in tensor memory, kATmemCols columns per ring stage from
    // column kATmemCol0, after the two accumulator slots.)
    static constexpr uint32_t kABytes = W16 ? 0u : 128u * 128u * kSub;
    // W16: a landing ring of slots holding one K block's E4M3 weight tile
    // (16 KB) and its bf16 activation tile (two 64-column halves of BN x 128
    // bytes).  The converting warps empty a slot as soon as they have turned
    // the weights into the A tile and copied the activations into the B
    // tile of an MMA ring stage, so the landing slots never wait for MMAs.
    static constexpr uint32_t kLBytes = W16 ? 128u * 128u : 0u;
    static constexpr uint32_t kXBBytes = W16 ? static_cast<uint32_t>(BN) * 256u : 0u;
    static constexpr uint32_t kLSlotBytes = kLBytes + kXBBytes;
    static constexpr int kLStages = W16 ? (BN == 16 ? 8 : 7) : 0;
    // TWO_SM: each CTA of the pair holds BN/2 weight rows.  W16: the bf16
    // activation tile copied out of the landing slot.
    static constexpr uint32_t kBBytes = W16 ? kXBBytes : static_cast<uint32_t>(TWO_SM ? BN / 2 : BN) * 128u * kSub;
    static constexpr uint32_t kSABytes = BLOCKWISE ? static_cast<uint32_t>(kTokTile) * 4u : 0u;  // TMA box
    // Scale slots are 128-byte aligned (TMA destination alignment).
    static constexpr uint32_t kSASlot = BLOCKWISE ? (kSABytes + 127u) / 128u * 128u : 0u;
    static constexpr int kSASlotFloats = static_cast<int>(kSASlot / 4u);
    // Bytes one ring slot's full barrier waits for (TWO_SM: both CTAs' loads).
    // Fused quantization (FQ; blockwise, swapped 16- or 32-token tiles): the
    // producer loads only the weight slices; two quantizing warps copy the
    // bf16 activation tiles (BN rows x 128 columns) into a staging ring of
    // their own and turn them into the ring's B tiles and scale slots.
    static constexpr int kXStages = FQ ? STAGES : 0;
    static constexpr uint32_t kXBytes = FQ ? static_cast<uint32_t>(BN) * 256u : 0u;
    static constexpr uint32_t kStageTx = TWO_SM ? 2u * (kABytes + kBBytes)
                                                : (FQ ? kABytes : (W16 ? kLSlotBytes : kABytes + kBBytes + kSABytes));
    // Two accumulator slots (+ W16: the bf16 A tiles of the ring stages, 128
    // K values = 64 columns each), allocated as a power of two >= 32 columns.
    static constexpr uint32_t kATmemCol0 = 2u * kSlotCols;
    static constexpr uint32_t kATmemCols = 64u;
    static constexpr uint32_t kTmemNeed = kATmemCol0 + (W16 ? STAGES * kATmemCols : 0u);
    static constexpr uint32_t kTmemCols = kTmemNeed <= 32 ? 32u : kTmemNeed <= 64 ? 64u
                                        : kTmemNeed <= 128 ? 128u : kTmemNeed <= 256 ? 256u : 512u;
    static constexpr uint32_t kOffA = 0;
    static constexpr uint32_t kOffB = kOffA + STAGES * kABytes;
    static constexpr uint32_t kOffSA = kOffB + STAGES * kBBytes;
    // Split-K with the swapped (decode) orientation pushes partial rows into
    // the owning CTA's receive buffer: slots for every source rank, each of
    // up to 4*ceil(32/split) rows of BN floats (at most 144 rows in total).
    static constexpr bool kPush = SWAP;
    // Row stride (floats) of the partial tiles exchanged by the push
    // reduction: padded by 4 so float4 accesses of consecutive rows by
    // consecutive lanes hit distinct shared-memory banks.
    static constexpr int kPartStride = BN + 4;
    static constexpr uint32_t kRecvBytes = kPush ? 144u * kPartStride * 4u : 0u;
    static constexpr uint32_t kOffRecv = kOffSA + STAGES * kSASlot;
    static constexpr uint32_t kOffX = (kOffRecv + kRecvBytes + 127u) / 128u * 128u;
    static constexpr uint32_t kOffL = (kOffX + kXStages * kXBytes + 1023u) / 1024u * 1024u;  // W16 landing ring
    static constexpr uint32_t kOffBar = kOffL + kLStages * kLSlotBytes;
    // Split-K exchange through the global workspace: only for partial tiles
    // of 64 KB and more (non-swapped 256-column tiles, swapped 128-token
    // tiles); smaller ones exchange faster in distributed shared memory.
    // The owner's remote partial rows land (bulk copies, padded rows) in the
    // idle ring after the partial tile, double-buffered in chunks, each chunk
    // completing on its own single-use barrier.
    static constexpr bool kWsExchange = !FQ && !W16 && (!SWAP || BN >= 128);
    static constexpr int kWsBars = 8;
    static constexpr uint32_t kOffLand = (128u * kPartStride * 4u + 127u) / 128u * 128u;
    static constexpr uint32_t kLandBytes = kOffX > kOffLand ? kOffX - kOffLand : 0u;
    // full, empty, tfull[2], tempty[2], drain, recv (+ W16: lfull, lempty[kLStages]), workspace chunks
    static constexpr uint32_t kNumBars = 2 * STAGES + 6 + 2 * kLStages + kWsBars;
    static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
    static constexpr uint32_t kOffCol = (kOffMisc + 16 + 15) / 16 * 16;  // staged column scale, bias
    // Non-swapped tiles store their output through one 2 KB staging buffer
    // per epilogue warp (32 rows x 32 columns of 2-byte values) and TMA.
    static constexpr bool kTmaStore = !SWAP;
    static constexpr uint32_t kStageBufBytes = 2048;
    static constexpr uint32_t kOffStage = (kOffCol + 2u * BN * 4u + 1023u) / 1024u * 1024u;
    static constexpr uint32_t kSmemBytes =
        (kTmaStore ? kOffStage + kEpiWarps * kStageBufBytes : kOffCol + 2u * BN * 4u) + 1024u;  // + alignment slack
    static constexpr uint32_t kRedBytes = 128u * (BN + 4) * 4u;  // padded partial tile
    static constexpr uint32_t kIdesc = W16 ? idesc_bf16_f32<128, BN>() : idesc_e4m3_f32<TWO_SM ? 256 : 128, BN>();
    static_assert(!TWO_SM || (!SWAP && !BLOCKWISE && BN == 256), "2-CTA MMA: non-swapped channelwise 256");
    static_assert(kRedBytes <= kOffSA, "the split-K partial tile must fit in the stage ring");
    static_assert(kSmemBytes <= 232448, "shared memory budget exceeded");
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N for M = 128");
    static_assert(kCols % 32 == 0 || kCols == 16, "epilogue column chunking");
    static_assert(2 * kSlotCols <= 512, "TMEM columns");
    static_assert(!FQ || (BLOCKWISE && SWAP && (BN == 16 || BN == 32) && !TWO_SM),
                  "fused quantization: blockwise 16- and 32-token tiles");
    static_assert(!W16 || (!BLOCKWISE && SWAP && !TWO_SM && !FQ && BN <= 32), "W16: swapped channelwise tiles");
    static_assert(!WIDE || (!SWAP && !BLOCKWISE && !TWO_SM && !FQ && !W16), "WIDE: non-swapped channelwise tiles");
    static_assert(kTmemNeed <= 512, "tensor memory budget exceeded");
};

__device__ __forceinline__ uint64_t policy_evict_normal()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Tile index -> (A-operand tile, B-operand tile) with grouped rasterisation:
// `group` consecutive A tiles sweep all B tiles together so concurrently
// running CTAs share operands in L2.
__device__ __forceinline__ void tile_coords(int tile, int a_tiles, int b_tiles, int group, int &a_t, int &b_t)
{
    const int per_group = group * b_tiles;
    const int g = tile / per_group;
    const int first = g * group;
    const int gsize = min(group, a_tiles - first);
    const int idx = tile - g * per_group;
    a_t = first + idx % gsize;
    b_t = idx / gsize;
}

// The kernel's tile order: groups of `group` A tiles (or B tiles when
// raster_b) sweep all tiles of the other operand.
__device__ __forceinline__ void tile_order(int tile, int a_tiles, int b_tiles, int group, int raster_b, int &a_t,
                                           int &b_t)
{
    if (raster_b) tile_coords(tile, b_tiles, a_tiles, group, b_t, a_t);
    else tile_coords(tile, a_tiles, b_tiles, group, a_t, b_t);
}

template <typename OutT>
__device__ __forceinline__ void store_out(OutT *out, long long idx, float v)
{
    out[idx] = to_out<OutT>(v);
}

// Two outputs converted (round to nearest even) and packed into one 32-bit
// word, lo in the low half: one paired conversion instruction.
template <typename OutT>
__device__ __forceinline__ uint32_t pack_out2(float lo, float hi);
template <>
__device__ __forceinline__ uint32_t pack_out2<__nv_bfloat16>(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}
template <>
__device__ __forceinline__ uint32_t pack_out2<__half>(float lo, float hi)
{
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// Channelwise output of 32 consecutive columns of one row: y = acc * a_scale
// * w_scale + bias, as (acc * a_scale) rounded, then one fma -- the scalar
// order -- two columns per packed instruction; scales and bias read four at a
// time from shared memory (16-byte aligned).
template <typename OutT>
__device__ __forceinline__ void convert32_channelwise(const float *acc, float row_scale, const float *col_scale,
                                                      const float *col_bias, uint32_t (&w)[16])
{
    const float2 rs = make_float2(row_scale, row_scale);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float4 sc = *reinterpret_cast<const float4 *>(col_scale + 4 * q);
        const float4 bi = *reinterpret_cast<const float4 *>(col_bias + 4 * q);
        const float2 p0 = __fmul2_rn(make_float2(acc[4 * q], acc[4 * q + 1]), rs);
        const float2 p1 = __fmul2_rn(make_float2(acc[4 * q + 2], acc[4 * q + 3]), rs);
        const float2 y0 = __ffma2_rn(p0, make_float2(sc.x, sc.y), make_float2(bi.x, bi.y));
        const float2 y1 = __ffma2_rn(p1, make_float2(sc.z, sc.w), make_float2(bi.z, bi.w));
        w[2 * q] = pack_out2<OutT>(y0.x, y0.y);
        w[2 * q + 1] = pack_out2<OutT>(y1.x, y1.y);
    }
}

// One warp stores a 32-row x 32-column box of 2-byte outputs (lane = row,
// w = its 32 packed values) through its 2 KB staging buffer: 64-byte rows,
// 64-byte TMA swizzle -- 16-byte unit u of row r sits at unit
// u ^ ((r >> 1) & 3), so the eight rows a quarter-warp writes hit distinct
// banks -- then lane 0 stores the box at (column x, row y) with TMA, which
// clips rows and columns outside the tensor.  The previous box stored from
// the buffer must have been read out before it is overwritten.
__device__ __forceinline__ void store_box_tma(const CUtensorMap *tm_out, uint8_t *sbuf, int lane,
                                              const uint32_t (&w)[16], int x, int y, bool any_inside)
{
    if (lane == 0) bulk_wait_read();
    __syncwarp();
#pragma unroll
    for (int u = 0; u < 4; ++u)
        *reinterpret_cast<uint4 *>(sbuf + lane * 64 + 16 * (u ^ ((lane >> 1) & 3))) =
            make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && any_inside) {
        tma_store_2d(tm_out, sbuf, x, y);
        bulk_commit();
    }
}

// Split-K reduction through the global workspace (every thread of the CTA
// calls it; the cluster barrier inside needs all of them).  The partial
// tile of this CTA is in shared memory, row r (TMEM lane: a token of a
// non-swapped tile, an output column of a swapped one) at r * kPartStride
// floats, its BN columns contiguous.  Rank q of the cluster owns the rows
// [rows * q / split, rows * (q + 1) / split) of the tile's valid rows.
//   1. Every rank writes the rows it does not own into its own slot of the
//      workspace (one slot of 128 x BN floats, rows dense), one bulk copy
//      per row, and waits for the copies to complete.
//   2. A cluster barrier publishes the slots.
//   3. The owner bulk-loads its rows from every other rank's slot, in
//      chunks of rows, double-buffered in the idle ring after its partial
//      tile (padded rows, so both item orders read shared memory without
//      bank conflicts), adds each item over the ranks in rank order and
//      stores the outputs; the slot lines it has loaded are dead and are
//      discarded from L2 (never written back to HBM).
// Items are 4-column groups, numbered in the order the owner stores its
// outputs: non-swapped (r, c4) with c4 fastest (consecutive threads,
// consecutive output columns of one token), swapped (c4, r) with r fastest
// (consecutive threads, consecutive output columns n0 + r).
// Called once per CTA and kept out of line: its registers do not add to
// the main loop's.
template <typename C, typename OutT, bool BLOCKWISE, bool SWAP>
__device__ __noinline__ void reduce_split_workspace(const GemmArgs &p, uint8_t *smem, const float *sColScale,
                                                    uint64_t *ws_bar, int rank, int cluster_id, int warp,
                                                    volatile int *abort, int m0, int n0)
{
    constexpr int SP = C::kPartStride;
    constexpr int BN = C::kPartStride - 4;   // columns of the partial tile (the MMA N extent)
    constexpr int G = BN / 4;
    constexpr uint32_t kRowBytes = BN * 4u;
    constexpr long long kSlotFloats = 128LL * BN;
    const float *sRed = reinterpret_cast<const float *>(smem);
    float *land = reinterpret_cast<float *>(smem + C::kOffLand);
    const int split = p.split;
    const bool epi = warp >= C::kEpiWarp0 && warp < C::kEpiWarp0 + C::kEpiWarps;
    const bool lead_warp = warp == C::kEpiWarp0;   // issues the bulk copies
    const int etid = threadIdx.x - 32 * C::kEpiWarp0;
    const int lane = threadIdx.x & 31;
    // Valid rows of the partial tile and this rank's share of them.
    const int rows = SWAP ? min(128, p.N - n0) : min(128, p.M - m0);
    const int lo = rows * rank / split, hi = rows * (rank + 1) / split;
    // Chunk rows: two buffers of (split - 1) x cr padded rows fit the
    // landing area (the host checks that the chunks fit kWsBars barriers).
    const int cr = static_cast<int>(C::kLandBytes / (2u * static_cast<uint32_t>(split - 1) * SP * 4u));
    const int nchunks = hi > lo ? (hi - lo + cr - 1) / cr : 0;
    float *slots = p.ws + static_cast<long long>(cluster_id) * split * kSlotFloats;
    if (epi) {
        // This thread's partial-tile writes, before the bulk copies read them.
        fence_proxy_async_smem();
        named_barrier_sync(1, C::kEpiThreads);
        if (lead_warp && !*abort) {
            float *mine = slots + static_cast<long long>(rank) * kSlotFloats;
            for (int r = lane; r < rows; r += 32)
                if (r < lo || r >= hi) bulk_store_global(mine + r * BN, sRed + r * SP, kRowBytes);
            bulk_commit();
            bulk_wait_all();
            fence_proxy_async_global();
        }
    }
    // Publishes every rank's slot to the cluster (release / acquire).
    cluster_sync();
    if (threadIdx.x == 32 * C::kEpiWarp0) FP8Q_TRACE_AT(p, kTrCluster1);
    if (!epi || *abort) return;
    auto issue = [&](int c) {   // the lead warp, all lanes
        const int r0 = lo + c * cr, nr = min(cr, hi - r0);
        float *buf = land + (c & 1) * (split - 1) * cr * SP;
        if (lane == 0) mbar_arrive_expect_tx(&ws_bar[c], static_cast<uint32_t>((split - 1) * nr) * kRowBytes);
        __syncwarp();
        for (int t = lane; t < (split - 1) * nr; t += 32) {
            const int j = t / nr, rr = t - j * nr;
            const int q = j < rank ? j : j + 1;
            bulk_load_global(buf + (j * cr + rr) * SP, slots + q * kSlotFloats + static_cast<long long>(r0 + rr) * BN,
                             kRowBytes, &ws_bar[c]);
        }
    };
    if (lead_warp) {
        fence_proxy_async_global();   // after the barrier's acquire, before the bulk reads
        for (int c = 0; c < 2 && c < nchunks; ++c) issue(c);
    }
    const bool may_discard = (reinterpret_cast<uintptr_t>(p.ws) & 127u) == 0;
    OutT *out = static_cast<OutT *>(p.out);
    for (int c = 0; c < nchunks; ++c) {
        const bool got = mbar_wait(&ws_bar[c], 0, abort, p.status);
        const bool ok = named_barrier_and(1, C::kEpiThreads, got);
        const int r0 = lo + c * cr, nr = min(cr, hi - r0);
        const float *buf = land + (c & 1) * (split - 1) * cr * SP;
        if (ok) {
            for (int i = etid; i < nr * G; i += C::kEpiThreads) {
                int rr, c4;
                if (SWAP) { c4 = i / nr; rr = i - c4 * nr; }
                else { rr = i / G; c4 = i - rr * G; }
                const int r = r0 + rr;
                float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int q = 0; q < split; ++q) {
                    const float *src = q == rank ? sRed + r * SP : buf + ((q < rank ? q : q - 1) * cr + rr) * SP;
                    const float4 v = *reinterpret_cast<const float4 *>(src + 4 * c4);
                    sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
                }
                const float sv[4] = {sum.x, sum.y, sum.z, sum.w};
                if (SWAP) {
                    // Output column n0 + r; tokens m0 + 4 c4 .. + 3 (scales
                    // staged in sColScale by the epilogue).
                    const int n = n0 + r;
                    const float wsc = BLOCKWISE ? 1.0f : __ldg(p.w_scale + n);
                    const float bv = p.bias != nullptr ? __bfloat162float(p.bias[n]) : 0.0f;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int m = m0 + c4 * 4 + e;
                        if (m < p.M) {
                            const float y = BLOCKWISE ? sv[e] + bv : fmaf(sv[e] * wsc, sColScale[c4 * 4 + e], bv);
                            out[static_cast<long long>(m) * p.ldo + n] = to_out<OutT>(y);
                        }
                    }
                } else {
                    // Token m0 + r; output columns n0 + 4 c4 .. + 3.
                    const int m = m0 + r, n = n0 + 4 * c4;
                    if (n < p.N) {
                        const float am = BLOCKWISE ? 1.0f : __ldg(p.a_scale + m);
                        float y[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const bool in = n + e < p.N;
                            const float bv = (p.bias != nullptr && in) ? __bfloat162float(p.bias[n + e]) : 0.0f;
                            y[e] = BLOCKWISE ? sv[e] + bv : fmaf(sv[e] * am, in ? __ldg(p.w_scale + n + e) : 0.0f, bv);
                        }
                        OutT *o = out + static_cast<long long>(m) * p.ldo + n;
                        if (n + 4 <= p.N) {
                            *reinterpret_cast<uint2 *>(o) =
                                make_uint2(pack_out2<OutT>(y[0], y[1]), pack_out2<OutT>(y[2], y[3]));
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                if (n + e < p.N) o[e] = to_out<OutT>(y[e]);
                        }
                    }
                }
            }
        }
        // This thread's reads of the buffer, before the next bulk copies
        // overwrite it.
        fence_proxy_async_smem();
        named_barrier_sync(1, C::kEpiThreads);
        if (lead_warp && ok) {
            // The chunk's rows in the other ranks' slots are dead.
            if (may_discard) {
                constexpr int kLinesPerRow = static_cast<int>(kRowBytes / 128u);
                for (int t = lane; t < (split - 1) * nr * kLinesPerRow; t += 32) {
                    const int j = t / (nr * kLinesPerRow), l = t - j * (nr * kLinesPerRow);
                    const int q = j < rank ? j : j + 1;
                    discard_l2_line(reinterpret_cast<const uint8_t *>(slots + q * kSlotFloats +
                                                                      static_cast<long long>(r0) * BN) +
                                    128 * l);
                }
            }
            if (c + 2 < nchunks) issue(c + 2);
        }
    }
    if (threadIdx.x == 32 * C::kEpiWarp0) FP8Q_TRACE_AT(p, kTrReduced);
}

template <bool SWAP, int BN, int STAGES, bool BLOCKWISE, typename OutT, bool TWO_SM = false, bool FQ = false,
          bool W16 = false, bool WIDE = false>
__global__ void __launch_bounds__(GemmCfg<SWAP, BN, STAGES, BLOCKWISE, TWO_SM, FQ, W16, WIDE>::kThreads,
                                  GemmCfg<SWAP, BN, STAGES, BLOCKWISE, TWO_SM, FQ, W16, WIDE>::kMinBlocks)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                    const __grid_constant__ CUtensorMap tm_sa, const __grid_constant__ CUtensorMap tm_out,
                    const GemmArgs p)
{
    using C = GemmCfg<SWAP, BN, STAGES, BLOCKWISE, TWO_SM, FQ, W16, WIDE>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sA = smem + C::kOffA;
    uint8_t *sB = smem + C::kOffB;
    float *sSA = reinterpret_cast<float *>(smem + C::kOffSA);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    uint64_t *empty = full + STAGES;
    uint64_t *tfull = empty + STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint64_t *recv_full = drain + 1;
    uint8_t *sX = smem + C::kOffX;              // FQ: bf16 activation tiles
    uint8_t *sL = smem + C::kOffL;              // W16: E4M3 weight landing slots
    uint64_t *lfull = recv_full + 1;            // W16: landing slot filled
    uint64_t *lempty = lfull + C::kLStages;     // W16: landing slot read by the converting warps
    uint64_t *ws_bar = lempty + C::kLStages;    // split-K workspace exchange: chunk landed
    constexpr int kLS = C::kLStages > 0 ? C::kLStages : 1;  // (non-W16 builds never use the landing ring)
    float *sRecv = reinterpret_cast<float *>(smem + C::kOffRecv);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
    float *sColScale = reinterpret_cast<float *>(smem + C::kOffCol);
    float *sColBias = sColScale + BN;
    // Split-K partial tile, reusing the (then idle) ring: [BN][128] for the
    // pull reduction, [128][BN] (rows contiguous) for the push reduction.
    float *sRed = reinterpret_cast<float *>(smem);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = p.split;
    const bool pair = TWO_SM;                 // (then non-swapped, split == 1)
    const int csize = pair ? 2 : split;       // CTAs per cluster
    const int rank = csize > 1 ? static_cast<int>(cluster_ctarank()) : 0;
    const int krank = pair ? 0 : rank;        // position along K
    const int cluster_id = blockIdx.x / csize;
    const int num_clusters = gridDim.x / csize;
    const int kb_begin = static_cast<int>(static_cast<long long>(p.num_kb) * krank / split);
    const int kb_end = static_cast<int>(static_cast<long long>(p.num_kb) * (krank + 1) / split);
    const int nkb = kb_end - kb_begin;
    // Paired: the A-tile index walks token-tile pairs; this CTA's token tile
    // is 2 * pair_index + rank.
    const int a_tiles = SWAP ? p.n_tiles : (pair ? (p.m_tiles + 1) / 2 : p.m_tiles);
    const int b_tiles = SWAP ? p.m_tiles : p.n_tiles;
    auto coords = [&](int tile, int &a_t, int &b_t) {
        tile_order(tile, a_tiles, b_tiles, p.group, p.raster_b, a_t, b_t);
        if (pair) a_t = 2 * a_t + rank;
    };
    // Paired: this CTA's half of the weight rows (its ring holds only that
    // half).
    constexpr int kHalfRows = BN / 2;
    const int w_half_row = pair ? rank * kHalfRows : 0;
    const bool leader = rank == 0;  // TWO_SM: the CTA that issues the MMAs
    // TWO_SM: a ring slot's full barrier in the even CTA (shared::cluster).
    auto lead_full = [&](int stage) { return dsmem_map(smem_u32(&full[stage]), 0u); };
    // Work units (tile, K blocks [kb0, kb1)), walked in the same order by
    // every role: the cluster's tiles over this rank's K range, or (stream-K)
    // this CTA's range of (tile, K block) pairs cut at tile boundaries.
    const bool sk = C::kStreamK && p.stream_k != 0;
    const long long sk_total = static_cast<long long>(p.num_tiles) * p.num_kb;
    const long long sk_g0 = sk ? sk_total * blockIdx.x / gridDim.x : 0;
    const long long sk_g1 = sk ? sk_total * (blockIdx.x + 1) / gridDim.x : 0;
    const long long unit_first = sk ? sk_g0 : static_cast<long long>(cluster_id);
    auto next_unit = [&](long long &cur, int &tile, int &kb0, int &kb1) -> bool {
        if (sk) {
            if (cur >= sk_g1) return false;
            tile = static_cast<int>(cur / p.num_kb);
            kb0 = static_cast<int>(cur - static_cast<long long>(tile) * p.num_kb);
            const long long left = sk_g1 - cur;
            kb1 = left < p.num_kb - kb0 ? kb0 + static_cast<int>(left) : p.num_kb;
            cur += kb1 - kb0;
            return true;
        }
        if (cur >= p.num_tiles) return false;
        tile = static_cast<int>(cur);
        kb0 = kb_begin;
        kb1 = kb_end;
        cur += num_clusters;
        return true;
    };

    // Prologue.  Thread 0 initialises the barriers while warp 1 allocates the
    // TMEM accumulators; one block barrier publishes both.
    if (threadIdx.x == 0) {
        FP8Q_TRACE_AT(p, kTrEntry);
#ifdef FP8Q_TRACE
        if (p.trace != nullptr && blockIdx.x < 4096) {
            unsigned smid;
            asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
            p.trace[blockIdx.x * kTraceSlots + kTrSmid] = smid;
            p.trace[blockIdx.x * kTraceSlots + kTrRank] = static_cast<unsigned long long>(rank);
        }
#endif
        tma_prefetch_map(&tm_a);
        tma_prefetch_map(&tm_b);
        if (BLOCKWISE) tma_prefetch_map(&tm_sa);
        if (C::kTmaStore) tma_prefetch_map(&tm_out);
        for (int s = 0; s < STAGES; ++s) {
            // FQ: the quantizing warps' arrivals publish the B tile; W16: the
            // converting warps' arrivals alone publish the stage (its bf16 A
            // tile in tensor memory and its activation B tile).
            mbar_init(&full[s], W16 ? C::kConvWarps : 1 + C::kQuantWarps);
            mbar_init(&empty[s], (BLOCKWISE ? C::kEpiWarps : 0) + C::kIssuers);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], C::kIssuers);
            mbar_init(&tempty[i], TWO_SM ? 2 * C::kEpiWarps : C::kEpiWarps);
        }
        mbar_init(drain, C::kIssuers);
        mbar_init(recv_full, 1);
        for (int j = 0; j < C::kLStages; ++j) {
            mbar_init(&lfull[j], 1);
            mbar_init(&lempty[j], C::kConvWarps);
        }
        for (int c = 0; c < C::kWsBars; ++c) mbar_init(&ws_bar[c], 1);

        *abort = 0;
        fence_mbar_init();
        if (C::kPush && split > 1 && p.ws == nullptr) {
            // Expect the partial rows this CTA owns from every other rank
            // (armed before the cluster barrier below, so before any push).
            const int my_rows = 4 * (32 * (rank + 1) / split) - 4 * (32 * rank / split);
            mbar_arrive_expect_tx(recv_full, static_cast<uint32_t>((split - 1) * my_rows * C::kPartStride * 4));
        }
    }
    if (warp == 1) {
        if (TWO_SM) {
            tmem_alloc_pair(tmem_holder, C::kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_holder, C::kTmemCols);
            tmem_relinquish();
        }
        if (lane == 0) FP8Q_TRACE_AT(p, kTrTmemAlloc);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    // Barriers must be initialised before the early weight loads below (in
    // both CTAs of a pair: each loads into, or signals, the other).
    if (pair) cluster_sync();
    // Push reduction: every CTA's receive barrier must be initialised and
    // armed before any CTA of the cluster may push into it.  Arrive now,
    // wait just before the dependency wait (the latency overlaps the rest of
    // the prologue).
    const bool push = C::kPush && split > 1 && p.ws == nullptr;   // DSMEM push reduction
    if (push) cluster_arrive_relaxed();
    // Weight slices of the first tile issued before the dependency wait.
    int npre = 0;
    if (warp == 0 && lane == 0) {
        // The kernels that may still run now are the immediate
        // predecessor and, when that is a quantizer that let this kernel
        // launch before its own dependency wait, the one before it; the
        // host clears p.preload when any of them writes the weights.  Otherwise the first tile's weight
        // slices stream into the ring right away and the activation slices
        // follow after pdl_wait().  Further weight slices of the first tile
        // are prefetched into L2 (always safe: L2 is the coherence point).
        long long cur0 = unit_first;
        int t0, u0_kb0, u0_kb1;
        if (next_unit(cur0, t0, u0_kb0, u0_kb1)) {
            const int u0_nkb = u0_kb1 - u0_kb0;
            int a_t, b_t;
            coords(t0, a_t, b_t);
            const CUtensorMap *wmap = SWAP ? &tm_a : &tm_b;
            const int wrow = SWAP ? a_t * 128 : b_t * BN;
            // (W16: the E4M3 weight slices land in their own slots.)
            uint8_t *wbuf = W16 ? sL : (SWAP ? sA : sB);
            const uint32_t wbytes = W16 ? C::kLSlotBytes : (SWAP ? C::kABytes : C::kBBytes);
            uint64_t *wbar = W16 ? lfull : full;
            const int ring = W16 ? C::kLStages : STAGES;
            const uint64_t pol_w = SWAP ? policy_evict_first() : policy_evict_normal();
            // (WIDE: stages of two K blocks.)
            const int u0_nst = (u0_nkb + C::kSub - 1) / C::kSub;
            npre = p.preload ? (u0_nst < ring ? u0_nst : ring) : 0;
            for (int i = 0; i < npre; ++i) {
                if (TWO_SM) {
                    if (leader) mbar_arrive_expect_tx(&full[i], C::kStageTx);
                    tma_load_2d_pair(wbuf + i * wbytes, wmap, lead_full(i), (u0_kb0 + i) * 128, wrow + w_half_row,
                                     pol_w);
                    continue;
                }
                mbar_arrive_expect_tx(&wbar[i], C::kStageTx);
                if constexpr (WIDE)
                    tma_load_3d(wbuf + i * wbytes, wmap, &wbar[i], 0, wrow, u0_kb0 + 2 * i, pol_w);
                else
                    tma_load_2d(wbuf + i * wbytes, wmap, &wbar[i], (u0_kb0 + i) * 128, wrow, pol_w);
            }
            const int pf = WIDE ? 0 : (u0_nkb < p.prefetch_kb ? u0_nkb : p.prefetch_kb);
            for (int i = npre; i < pf; ++i) tma_prefetch_l2_2d(wmap, (u0_kb0 + i) * 128, wrow + w_half_row);
            if (sk) {
                // Stream-K: a CTA's first unit may be a few K blocks only
                // (the tail of a tile); the ring and the L2 prefetch go on
                // into the following units, in the order the producer
                // issues them (issued < npre: weight slice already loaded).
                int n = u0_nkb;   // blocks walked so far
                auto more = [&]() { return (p.preload && npre == n && npre < ring) || n < p.prefetch_kb; };
                int tn, kn0, kn1;
                while (more() && next_unit(cur0, tn, kn0, kn1)) {
                    coords(tn, a_t, b_t);
                    const int wr = a_t * 128;   // (swapped tiles: the weights are the A operand)
                    for (int kb = kn0; kb < kn1 && more(); ++kb, ++n) {
                        if (p.preload && npre == n && npre < ring) {
                            mbar_arrive_expect_tx(&wbar[npre], C::kStageTx);
                            tma_load_2d(wbuf + npre * wbytes, wmap, &wbar[npre], kb * 128, wr, pol_w);
                            ++npre;
                        } else if (n < p.prefetch_kb) {
                            tma_prefetch_l2_2d(wmap, kb * 128, wr);
                        }
                    }
                }
            }
        }
        FP8Q_TRACE_AT(p, kTrPreloaded);
    }
    if (push) cluster_wait();
    // The producer's cache policies, made before the dependency wait.
    uint64_t pol_a = 0, pol_b = 0;
    if (warp == 0 && lane == 0) {
        pol_a = SWAP ? policy_evict_first() : policy_evict_normal();
        pol_b = SWAP ? policy_evict_last() : policy_evict_normal();
    }
    if (threadIdx.x == 0) FP8Q_TRACE_AT(p, kTrPrologue);
    // Everything below may read the previous kernel's output (activations,
    // scales) or overwrite buffers it reads (out).
    pdl_wait();
    pdl_trigger();
    if (threadIdx.x == 0) FP8Q_TRACE_AT(p, kTrPdlWait);
    if constexpr (C::kRegSplit) {
        if (warp < 4) setmaxnreg_dec<C::kLowRegs>();
        else setmaxnreg_inc<C::kHighRegs>();
    }

    if (warp == 0) {
        // ------------------------------------------------------------------
        // TMA producer
        // ------------------------------------------------------------------
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            long long issued = 0;
            long long cur = unit_first;
            int tile, ukb0, ukb1;
            while (next_unit(cur, tile, ukb0, ukb1)) {
                int a_t, b_t;
                coords(tile, a_t, b_t);
                const int m_tile = SWAP ? b_t : a_t;
                const int a_row = a_t * 128;
                const int b_row = b_t * BN;
                bool ok = true;
                for (int kb = ukb0; kb < ukb1; kb += C::kSub) {
                    if (issued == 0) FP8Q_TRACE_AT(p, kTrFirstTma);
                    if (TWO_SM) {
                        if (issued >= npre) {
                            if (!mbar_wait(&empty[stage], phase ^ 1u, abort, p.status)) { ok = false; break; }
                            if (leader) mbar_arrive_expect_tx(&full[stage], C::kStageTx);
                            tma_load_2d_pair(sB + stage * C::kBBytes, &tm_b, lead_full(stage), kb * 128,
                                             b_row + w_half_row, pol_b);
                        }
                        tma_load_2d_pair(sA + stage * C::kABytes, &tm_a, lead_full(stage), kb * 128, a_row, pol_a);
                    } else if (W16) {
                        // Block `issued` into landing slot j: its E4M3 weight
                        // tile (already in flight if preloaded) and its bf16
                        // activation tile as two 64-column halves, both for
                        // the converting warps.
                        const int j = static_cast<int>(issued % kLS);
                        uint8_t *slot = sL + j * C::kLSlotBytes;
                        if (issued >= npre) {
                            const uint32_t lph = static_cast<uint32_t>((issued / kLS) & 1);
                            if (!mbar_wait(&lempty[j], lph ^ 1u, abort, p.status)) { ok = false; break; }
                            mbar_arrive_expect_tx(&lfull[j], C::kStageTx);
                            tma_load_2d(slot, &tm_a, &lfull[j], kb * 128, a_row, pol_a);
                        }
#pragma unroll
                        for (int h = 0; h < 2; ++h)
                            tma_load_2d(slot + C::kLBytes + h * (BN * 128), &tm_b, &lfull[j], kb * 128 + 64 * h, b_row,
                                        pol_b);
                    } else if (issued < npre) {
                        // Weight slice already in flight; barrier armed.
                        if (FQ) {
                            // (the activation tile is the epilogue warps' work)
                        } else if (SWAP)
                            tma_load_2d(sB + stage * C::kBBytes, &tm_b, &full[stage], kb * 128, b_row, pol_b);
                        else if (WIDE)
                            tma_load_3d(sA + stage * C::kABytes, &tm_a, &full[stage], 0, a_row, kb, pol_a);
                        else
                            tma_load_2d(sA + stage * C::kABytes, &tm_a, &full[stage], kb * 128, a_row, pol_a);
                    } else {
                        FP8Q_TRACE_STAGE(p, 3, issued);
                        if (!mbar_wait(&empty[stage], phase ^ 1u, abort, p.status)) { ok = false; break; }
                        mbar_arrive_expect_tx(&full[stage], C::kStageTx);
                        if constexpr (WIDE) {
                            tma_load_3d(sA + stage * C::kABytes, &tm_a, &full[stage], 0, a_row, kb, pol_a);
                            tma_load_3d(sB + stage * C::kBBytes, &tm_b, &full[stage], 0, b_row, kb, pol_b);
                        } else {
                            tma_load_2d(sA + stage * C::kABytes, &tm_a, &full[stage], kb * 128, a_row, pol_a);
                            if (!FQ)
                                tma_load_2d(sB + stage * C::kBBytes, &tm_b, &full[stage], kb * 128, b_row, pol_b);
                        }
                    }
                    if (BLOCKWISE && !FQ)
                        tma_load_2d(sSA + stage * C::kSASlotFloats, &tm_sa, &full[stage], m_tile * C::kTokTile, kb,
                                    pol_b);
                    FP8Q_TRACE_STAGE(p, 0, issued);
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
            }
            // Drain: the last STAGES copies must have landed before the CTA
            // may exit (they complete in the normal flow long before this).
            // Preloaded weight slices whose stage never got its activation
            // slice (an early abort) are waited for as well: their barrier
            // phase cannot complete, so the wait only ends on the timeout.
            if (issued < npre) issued = npre;
            const long long first = issued > STAGES ? issued - STAGES : 0;
            // (TWO_SM: only the even CTA's full barriers are used.)
            // (W16: the copies go to the landing ring.)
            if (W16) {
                const long long lfirst = issued > kLS ? issued - kLS : 0;
                for (long long j = lfirst; j < issued; ++j)
                    mbar_wait_drain(&lfull[j % kLS], static_cast<uint32_t>((j / kLS) & 1), p.status);
            } else if (!TWO_SM || leader) {
                for (long long j = first; j < issued; ++j)
                    mbar_wait_drain(&full[j % STAGES], static_cast<uint32_t>((j / STAGES) & 1), p.status);
            }
            // Paired: the partner's MMA commits arrive on this CTA's empty
            // barriers; every one of them must have landed before exit.
            if (pair)
                for (long long j = first; j < issued; ++j)
                    mbar_wait_drain(&empty[j % STAGES], static_cast<uint32_t>((j / STAGES) & 1), p.status);
        }
    } else if (warp <= C::kIssuers) {
        // ------------------------------------------------------------------
        // MMA issuers (one thread per issuing warp; issuer j takes the K
        // steps k of every K block with k % kIssuers == j)
        // ------------------------------------------------------------------
        const int issuer = warp - 1;
        if (lane == 0 && (!TWO_SM || leader)) {
            uint32_t stage = 0, phase = 0, slot = 0, tphase = 0;
            long long n_stages = 0;   // stages consumed (trace stamps)
            bool ok = true;
            bool first_unit = true;
            long long cur = unit_first;
            int tile, ukb0, ukb1;
            while (ok && next_unit(cur, tile, ukb0, ukb1)) {
                if (!BLOCKWISE) {
                    if (!mbar_wait(&tempty[slot], tphase ^ 1u, abort, p.status)) { ok = false; break; }
                    tc_fence_after();
                }
                const int unkb = (ukb1 - ukb0 + C::kSub - 1) / C::kSub;   // ring stages of this unit
                for (int i = 0; i < unkb; ++i) {
                    if (BLOCKWISE) {
                        if (!mbar_wait(&tempty[slot], tphase ^ 1u, abort, p.status)) { ok = false; break; }
                        tc_fence_after();
                    }
                    if (!mbar_wait(&full[stage], phase, abort, p.status)) { ok = false; break; }
                    tc_fence_after();
                    if (issuer == 0) FP8Q_TRACE_STAGE(p, 1, n_stages);
                    if (first_unit && i == 0 && issuer == 0) FP8Q_TRACE_AT(p, kTrFirstMma);
                    const uint32_t a_addr = smem_u32(sA + stage * C::kABytes);
                    const uint32_t b_addr = smem_u32(sB + stage * C::kBBytes);
                    const uint32_t d = tmem_base + slot * C::kSlotCols + static_cast<uint32_t>(issuer * BN);
#pragma unroll
                    for (int k = 0; k < C::kKSteps; ++k) {
                        if (C::kIssuers > 1 && k % C::kIssuers != issuer) continue;
                        const uint32_t acc = BLOCKWISE ? (k > 0) : (i > 0 || k >= C::kIssuers);
                        if (TWO_SM) {
                            umma_e4m3_pair(d, umma_desc_sw128(a_addr + k * 32), umma_desc_sw128(b_addr + k * 32),
                                           C::kIdesc, acc);
                        } else if (W16) {
                            // K step k (16 bf16): TMEM columns 8k .. 8k + 7 of
                            // the stage's A tile; 32 bytes in 64-column half
                            // k / 4 of the B slot.
                            const uint32_t at = tmem_base + C::kATmemCol0 + stage * C::kATmemCols +
                                                static_cast<uint32_t>(k * 8);
                            const uint32_t bo = static_cast<uint32_t>((k >> 2) * (BN * 128) + (k & 3) * 32);
                            umma_bf16_tmem_a(d, at, umma_desc_sw128(b_addr + bo), C::kIdesc, acc);
                        } else {
                            // (WIDE: K step k reads 32 bytes of K block k / 4 of the stage.)
                            const uint32_t ao = static_cast<uint32_t>((k >> 2) * (128 * 128) + (k & 3) * 32);
                            const uint32_t bo = static_cast<uint32_t>((k >> 2) * (BN * 128) + (k & 3) * 32);
                            umma_e4m3(d, umma_desc_sw128(a_addr + ao), umma_desc_sw128(b_addr + bo), C::kIdesc,
                                      acc);
                        }
                    }
                    if (TWO_SM) umma_commit_pair_mc(&empty[stage], 3);
                    else umma_commit(&empty[stage]);
                    if (issuer == 0) FP8Q_TRACE_STAGE(p, 2, n_stages);
                    ++n_stages;
                    if (BLOCKWISE) {
                        umma_commit(&tfull[slot]);
                        slot ^= 1u;
                        if (slot == 0) tphase ^= 1u;
                    }
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                if (!BLOCKWISE) {
                    if (TWO_SM) umma_commit_pair_mc(&tfull[slot], 3);
                    else umma_commit(&tfull[slot]);
                    slot ^= 1u;
                    if (slot == 0) tphase ^= 1u;
                }
                first_unit = false;
            }
            if (issuer == 0) FP8Q_TRACE_AT(p, kTrLastCommit);
            // Every MMA this thread issued has finished before TMEM is freed.
            if (TWO_SM) umma_commit_pair(drain);
            else umma_commit(drain);
            mbar_wait_drain(drain, 0, p.status);
            // TWO_SM: the other CTA's epilogue releases arrive on this CTA's
            // accumulator barriers; all of them must have landed before exit.
            if (TWO_SM)
                for (int i = 0; i < 2; ++i) {
                    mbar_wait_drain(&tempty[slot], tphase ^ 1u, p.status);
                    slot ^= 1u;
                    if (slot == 0) tphase ^= 1u;
                }
        }
        __syncwarp();
    } else if (FQ && warp >= C::kQuantWarp0) {
        // ------------------------------------------------------------------
        // Quantizing warps (FQ): this CTA's K blocks g = 0, 1, ... (its tiles
        // in order, nkb blocks each).  Each thread owns BN/8 16-element chunks
        // of every block (rows t0, t0 + 8, ..., chunk c) and copies them itself
        // into staging slot g % kXStages with cp.async (16-byte global ->
        // shared copies, zero-filled past row M; not the TMA unit, whose
        // queue holds the weight tiles), kXStages blocks ahead, one commit
        // group per block.  Once ring stage g % STAGES is free (the empty
        // barrier the producer waits on: the block STAGES earlier was
        // consumed by its MMA and promoted), it quantizes them with the
        // standalone quantizer's arithmetic (quant_common.cuh) -- the row's
        // group scale from the 8 lanes holding that row -- writes the E4M3
        // codes into the 128-byte-swizzled B tile (16-byte unit c of row t
        // at c ^ (t & 7), as the TMA would) and the scale into the stage's
        // scale slot, and publishes the tile (proxy fence, arrive on full).
        // Each thread reads only the bytes it copied: no barrier between the
        // two warps.
        // ------------------------------------------------------------------
        if constexpr (FQ) {
            const int qt = threadIdx.x - 32 * C::kQuantWarp0;  // 0 .. 63
            const int t0 = qt >> 3, c = qt & 7;                 // rows t0, t0 + 8, ..., chunk c
            constexpr int kRowsPer = BN / 8;                    // rows of the tile per thread
            const long long total =
                cluster_id < p.num_tiles
                    ? static_cast<long long>((p.num_tiles - 1 - cluster_id) / num_clusters + 1) * nkb
                    : 0;
            // Copy this thread's part of block g into its staging slot (an
            // empty commit group past the last block keeps the count uniform).
            auto copy_x = [&](long long g) {
                if (g < total) {
                    int a_q, b_q;
                    coords(cluster_id + static_cast<int>(g / nkb) * num_clusters, a_q, b_q);
                    const int k0 = (kb_begin + static_cast<int>(g % nkb)) * 128 + c * 16;
                    uint8_t *slot = sX + static_cast<int>(g % C::kXStages) * C::kXBytes;
#pragma unroll
                    for (int h = 0; h < kRowsPer; ++h) {
                        const int t = t0 + 8 * h;
                        const int m = b_q * BN + t;
                        const bool in = m < p.M;
                        const __nv_bfloat16 *src = p.x + (in ? static_cast<long long>(m) * p.ldx + k0 : 0);
                        const uint32_t dst = smem_u32(slot + t * 256 + c * 32);
                        cp_async_16(dst, src, in ? 16u : 0u);
                        cp_async_16(dst + 16, src + 8, in ? 16u : 0u);
                    }
                }
                cp_async_commit();
            };
            for (int u = 0; u < C::kXStages; ++u) copy_x(u);
            uint32_t stage = 0, phase = 0;
            for (long long g = 0; g < total; ++g) {
                cp_async_wait_group<C::kXStages - 1>();   // block g's copies have landed
                const bool got = mbar_wait(&empty[stage], phase ^ 1u, abort, p.status);
                if (!__all_sync(0xffffffffu, got)) break;
                const uint8_t *xs = sX + static_cast<int>(g % C::kXStages) * C::kXBytes;
                uint8_t *bt = sB + stage * C::kBBytes;
                float *sa = sSA + stage * C::kSASlotFloats;
#pragma unroll
                for (int h = 0; h < kRowsPer; ++h) {
                    const int t = t0 + 8 * h;
                    const Chunk16 v = load_chunk_smem(xs + t * 256 + c * 32);
                    float m = chunk_amax(v, 0.0f);
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                    const float sc = scale_of(m, p.eps);
                    *reinterpret_cast<uint4 *>(bt + t * 128 + ((c ^ (t & 7)) << 4)) = quant_chunk(v, sc);
                    if (c == 0) sa[t] = sc;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&full[stage]);
                copy_x(g + C::kXStages);                 // refill the slot just read (by this thread)
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
            cp_async_wait_all();   // no copy may still be writing when the CTA exits
        }
        __syncwarp();
    } else if (W16 && warp >= C::kConvWarp0) {
        // ------------------------------------------------------------------
        // Converting warps (W16): once block g's tiles have landed (slot
        // g % kLStages of the landing ring) and the A tile of its ring stage
        // has been read by the MMAs STAGES blocks earlier, convert the E4M3
        // weight tile (128 rows x 128 bytes, 128-byte swizzled by the TMA:
        // logical 16-byte unit L of row m at position L ^ (m & 7)) to bf16 --
        // exact: every E4M3 value is a bf16 value -- into that stage's A tile
        // in tensor memory.  Weight row m is TMEM lane m, so warp w (lanes
        // 32 (w % 4) ..) converts rows 32 (w % 4) + lane, the first four
        // warps K 0..63 of the block, the next four K 64..127: each thread
        // one row's 64 bytes into 32 columns.  The bf16 activation tile is
        // copied unchanged into the stage's B slot (both 1024-byte aligned,
        // so the swizzle carries over), and the landing slot is free again.
        // ------------------------------------------------------------------
        if constexpr (W16) {
            static_assert(C::kConvWarps == 8, "two warps per TMEM lane quarter");
            const int ct = threadIdx.x - 32 * C::kConvWarp0;  // 0 .. 32 * kConvWarps - 1
            const int quarter = warp & 3;                      // TMEM lanes this warp may access
            const int khalf = (warp - C::kConvWarp0) >> 2;     // K half of the block
            const int m = quarter * 32 + lane;                 // weight row of the tile = TMEM lane
            constexpr int kXUnits = static_cast<int>(C::kXBBytes / 16u) / (32 * C::kConvWarps);  // activation units
            static_assert(static_cast<int>(C::kXBBytes / 16u) % (32 * C::kConvWarps) == 0, "activation units");
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + C::kATmemCol0 +
                                   static_cast<uint32_t>(khalf * 32);
            const long long total =
                cluster_id < p.num_tiles
                    ? static_cast<long long>((p.num_tiles - 1 - cluster_id) / num_clusters + 1) * nkb
                    : 0;
            uint32_t stage = 0, phase = 0;
            for (long long g = 0; g < total; ++g) {
                const int j = static_cast<int>(g % kLS);
                bool got = mbar_wait(&lfull[j], static_cast<uint32_t>((g / kLS) & 1), abort, p.status);
                got = got && mbar_wait(&empty[stage], phase ^ 1u, abort, p.status);   // A tile read by its MMAs
                if (!__all_sync(0xffffffffu, got)) break;
                tc_fence_after();
                const uint8_t *ls = sL + j * C::kLSlotBytes;
                uint4 vin[4], xin[kXUnits];
                // Units 4 khalf .. 4 khalf + 3 of row m: the eight rows of a
                // store phase hit eight distinct positions (no bank conflict).
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    vin[i] = *reinterpret_cast<const uint4 *>(ls + m * 128 + (((4 * khalf + i) ^ (m & 7)) << 4));
#pragma unroll
                for (int q = 0; q < kXUnits; ++q)
                    xin[q] = *reinterpret_cast<const uint4 *>(ls + C::kLBytes + (ct + q * 32 * C::kConvWarps) * 16);
#pragma unroll
                for (int q = 0; q < kXUnits; ++q)
                    *reinterpret_cast<uint4 *>(sB + stage * C::kBBytes + (ct + q * 32 * C::kConvWarps) * 16) = xin[q];
                // Column 8 i + 2 e (+ 1) holds K 16 i + 4 e .. + 1 (+ 2 .. + 3)
                // of this half: two bf16 per column, the lower K in the low half.
                uint32_t o[32];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t wv[4] = {vin[i].x, vin[i].y, vin[i].z, vin[i].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        o[8 * i + 2 * e] = e4m3x2_to_bf16x2(static_cast<uint16_t>(wv[e] & 0xFFFFu));
                        o[8 * i + 2 * e + 1] = e4m3x2_to_bf16x2(static_cast<uint16_t>(wv[e] >> 16));
                    }
                }
                tmem_st32(t_row + stage * C::kATmemCols, o);
                tmem_st_wait();
                tc_fence_before();
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&full[stage]);
                    mbar_arrive(&lempty[j]);   // both tiles are out of the landing slot
                }
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
        __syncwarp();
    } else if (warp < C::kEpiWarp0) {
        // Idle warps of the register split's warpgroup 0.
    } else {
        // ------------------------------------------------------------------
        // Epilogue warps
        // ------------------------------------------------------------------
        const int ew = warp - C::kEpiWarp0;
        const int quarter = warp & 3;          // TMEM lanes this warp may access
        const int cgroup = ew >> 2;            // column group
        const int row = quarter * 32 + lane;   // TMEM lane = accumulator row
        const int col0 = cgroup * C::kCols;
        const int etid = threadIdx.x - 32 * C::kEpiWarp0;
        OutT *out = static_cast<OutT *>(p.out);
        uint32_t slot = 0, tphase = 0, estage = 0, ephase = 0;

        long long cur = unit_first;
        int tile, ukb0, ukb1;
        while (next_unit(cur, tile, ukb0, ukb1)) {
            int a_t, b_t;
            coords(tile, a_t, b_t);
            const int m0 = (SWAP ? b_t : a_t) * C::kTokTile;
            const int n0 = (SWAP ? a_t : b_t) * C::kColTile;
            // Row-wise (per thread) values.
            const int rm = SWAP ? 0 : m0 + row;       // token of this row (non-swapped)
            const int rn = SWAP ? n0 + row : 0;       // output column of this row (swapped)
            float row_scale = 0.0f, row_bias = 0.0f;
            if (!BLOCKWISE) {
                if (SWAP) row_scale = rn < p.N ? __ldg(p.w_scale + rn) : 0.0f;
                else row_scale = rm < p.M ? __ldg(p.a_scale + rm) : 0.0f;
            }
            if (SWAP && p.bias != nullptr && rn < p.N) row_bias = __bfloat162float(p.bias[rn]);

            // Column-wise values staged in shared memory.
            named_barrier_sync(1, C::kEpiThreads);
            for (int c = etid; c < BN; c += C::kEpiThreads) {
                if (SWAP) {
                    const int m = m0 + c;
                    // (W16: no activation scale)
                    sColScale[c] = (!BLOCKWISE && m < p.M) ? (W16 ? 1.0f : __ldg(p.a_scale + m)) : 0.0f;
                    sColBias[c] = 0.0f;
                } else {
                    const int n = n0 + c;
                    sColScale[c] = (!BLOCKWISE && n < p.N) ? __ldg(p.w_scale + n) : 0.0f;
                    sColBias[c] = (p.bias != nullptr && n < p.N) ? __bfloat162float(p.bias[n]) : 0.0f;
                }
            }
            named_barrier_sync(1, C::kEpiThreads);

            float acc[C::kCols];
            bool ok = true;
            if (BLOCKWISE) {
                // TMEM columns per wait: 16 where the accumulator row is long
                // (keeps the 128-float row and the loop state in registers),
                // 64 with the register split.
                constexpr int kPromoteCols = C::kRegSplit ? 64 : C::kCols >= 128 ? 16 : 32;
#pragma unroll
                for (int j = 0; j < C::kCols; ++j) acc[j] = 0.0f;
                const int wblk = SWAP ? a_t : (n0 + col0) >> 7;  // 128-row weight block of these columns
                const float *sw_row = p.w_scale + static_cast<long long>(wblk) * p.num_kb;
                for (int kb = ukb0; kb < ukb1; ++kb) {
                    // Warp-uniform outcome: the __syncwarp below needs every lane.
                    bool got = mbar_wait(&full[estage], ephase, abort, p.status);
                    got = got && mbar_wait(&tfull[slot], tphase, abort, p.status);
                    if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                    tc_fence_after();
                    const float swk = __ldg(sw_row + kb);
                    const float *sa = sSA + estage * C::kSASlotFloats;
                    const float srow = SWAP ? 0.0f : sa[row] * swk;
                    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + slot * C::kSlotCols + col0;
                    // Promotion, two columns per packed FMA (each lane a
                    // correctly rounded fmaf).
#pragma unroll
                    for (int c = 0; c < C::kCols; c += kPromoteCols) {
                        uint32_t r[kPromoteCols];
#pragma unroll
                        for (int h = 0; h < kPromoteCols; h += 16)
                            if (c + h < C::kCols) tmem_ld16(taddr + c + h, *reinterpret_cast<uint32_t(*)[16]>(r + h));
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < kPromoteCols && c + j < C::kCols; j += 2) {
                            const float2 s2 = SWAP ? make_float2(sa[col0 + c + j] * swk, sa[col0 + c + j + 1] * swk)
                                                   : make_float2(srow, srow);
                            const float2 t = __ffma2_rn(make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])),
                                                        s2, make_float2(acc[c + j], acc[c + j + 1]));
                            acc[c + j] = t.x;
                            acc[c + j + 1] = t.y;
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&tempty[slot]);
                        mbar_arrive(&empty[estage]);
                    }
                    slot ^= 1u;
                    if (slot == 0) tphase ^= 1u;
                    if (++estage == STAGES) { estage = 0; ephase ^= 1u; }
                }
            } else {
                ok = __all_sync(0xffffffffu, mbar_wait(&tfull[slot], tphase, abort, p.status));
                if (ok) {
                    tc_fence_after();
                    if (ew == 0 && lane == 0) FP8Q_TRACE_AT(p, kTrEpiFull);
                    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + slot * C::kSlotCols + col0;
                    // Non-swapped channelwise tiles go straight from TMEM to
                    // the output (or, split along K, to the partial tile);
                    // swapped tiles keep the whole row in registers for the
                    // stores or the split-K exchange below.
                    if constexpr (!SWAP) {
                        // 32 accumulator columns at a time: TMEM -> scale,
                        // bias, convert -> staging buffer -> TMA store; split
                        // along K: TMEM -> this row of the partial tile, kept
                        // row-major with padded rows in the ring (idle: every
                        // copy was consumed and every MMA has completed).
                        uint8_t *sbuf = smem + C::kOffStage + static_cast<uint32_t>(ew) * C::kStageBufBytes;
                        const int ybox = m0 + quarter * 32;
                        const bool partial = !TWO_SM && split > 1;
#pragma unroll 1
                        for (int ch = 0; ch < C::kCols / 32; ++ch) {
                            uint32_t r[32];
                            tmem_ld16(taddr + ch * 32, *reinterpret_cast<uint32_t(*)[16]>(r));
                            tmem_ld16(taddr + ch * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(r + 16));
                            if constexpr (C::kIssuers > 1) {
                                // Tiles narrower than 256 columns: the second
                                // issuer's accumulator (BN columns on), added
                                // in issuer order.
                                uint32_t r2[32];
                                tmem_ld16(taddr + BN + ch * 32, *reinterpret_cast<uint32_t(*)[16]>(r2));
                                tmem_ld16(taddr + BN + ch * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(r2 + 16));
                                tmem_ld_wait();
#pragma unroll
                                for (int j = 0; j < 32; ++j)
                                    r[j] = __float_as_uint(__uint_as_float(r[j]) + __uint_as_float(r2[j]));
                            } else {
                                tmem_ld_wait();
                            }
                            const int cb = col0 + ch * 32;
                            if (partial) {
                                float *dst = sRed + row * C::kPartStride + cb;
#pragma unroll
                                for (int j = 0; j < 32; j += 4)
                                    *reinterpret_cast<float4 *>(dst + j) =
                                        make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                                                    __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
                            } else {
                                uint32_t w[16];
                                convert32_channelwise<OutT>(reinterpret_cast<const float *>(r), row_scale,
                                                            sColScale + cb, sColBias + cb, w);
                                store_box_tma(&tm_out, sbuf, lane, w, n0 + cb, ybox, ybox < p.M && n0 + cb < p.N);
                            }
                        }
                    } else {
                        if constexpr (C::kIssuers == 1) {
                            // All column loads in flight at once, then one wait.
                            uint32_t r[C::kCols];
#pragma unroll
                            for (int c = 0; c < C::kCols; c += 16)
                                tmem_ld16(taddr + c, *reinterpret_cast<uint32_t(*)[16]>(r + c));
                            tmem_ld_wait();
#pragma unroll
                            for (int j = 0; j < C::kCols; ++j) acc[j] = __uint_as_float(r[j]);
                        } else {
                            // Up to 32 columns of every issuer's accumulator
                            // in flight, then one wait; added in issuer order.
                            constexpr int kChunk = C::kCols < 32 ? C::kCols : 32;
#pragma unroll
                            for (int c = 0; c < C::kCols; c += kChunk) {
                                uint32_t r[C::kIssuers][kChunk];
#pragma unroll
                                for (int a = 0; a < C::kIssuers; ++a)
#pragma unroll
                                    for (int h = 0; h < kChunk; h += 16)
                                        tmem_ld16(taddr + a * BN + c + h, *reinterpret_cast<uint32_t(*)[16]>(r[a] + h));
                                tmem_ld_wait();
#pragma unroll
                                for (int j = 0; j < kChunk; ++j) {
                                    float v = __uint_as_float(r[0][j]);
#pragma unroll
                                    for (int a = 1; a < C::kIssuers; ++a) v += __uint_as_float(r[a][j]);
                                    acc[c + j] = v;
                                }
                            }
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if (TWO_SM && !leader) mbar_arrive_cluster(dsmem_map(smem_u32(&tempty[slot]), 0u));
                        else mbar_arrive(&tempty[slot]);
                    }
                    slot ^= 1u;
                    if (slot == 0) tphase ^= 1u;
                }
            }
            // No early exit from the tile loop: every epilogue thread must
            // reach the same named barriers, so all of them take the same
            // decision (after a timeout every further wait fails at once
            // and the output below is skipped).
            if (!named_barrier_and(1, C::kEpiThreads, ok && !*abort)) continue;

            if (sk && (ukb0 > 0 || ukb1 < p.num_kb)) {
                // Stream-K unit that is part of a tile (only swapped tiles:
                // the whole row is in registers, kCols == BN).
                if constexpr (C::kStreamK) {
                    if (ukb0 > 0) {
                        // The CTA's leading unit: publish the partial tile
                        // (row-major [128][BN] in this CTA's slot).
                        float *dst = p.ws + static_cast<size_t>(blockIdx.x) * (128u * BN) + row * BN + col0;
#pragma unroll
                        for (int j = 0; j < C::kCols; j += 4)
                            *reinterpret_cast<float4 *>(dst + j) = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
                        // The barrier orders every thread's stores before
                        // thread 0's fence and release store (cumulative).
                        named_barrier_sync(1, C::kEpiThreads);
                        if (etid == 0) {
                            __threadfence();
                            st_release_gpu_u32(p.sk_flags + blockIdx.x, 1u);
                            FP8Q_TRACE_AT(p, kTrCluster1);   // stream-K: partial published
                        }
                        continue;
                    }
                    // The unit holding the tile's first K block: add the
                    // partials of the CTAs whose ranges start inside the
                    // tile (the sources), in increasing K order.  Epilogue
                    // thread q waits for source q's flag, so all the waits
                    // overlap; the barrier then orders every thread's reads
                    // after those acquires.
                    const long long tile_end = static_cast<long long>(tile + 1) * p.num_kb;
                    int nsrc = 0;
                    while (blockIdx.x + 1 + nsrc < gridDim.x &&
                           sk_total * (blockIdx.x + 1 + nsrc) / gridDim.x < tile_end)
                        ++nsrc;
                    bool seen = true;
                    for (int q = etid; q < nsrc; q += C::kEpiThreads)
                        seen = seen && flag_wait_acquire(p.sk_flags + blockIdx.x + 1 + q, abort, p.status);
                    const bool got = named_barrier_and(1, C::kEpiThreads, seen);
                    if (etid == 0) FP8Q_TRACE_AT(p, kTrReduced);   // stream-K: sources' flags seen
                    if (got) {
                        // (One source at a time: loading several sources' rows
                        // before adding them overlaps their L2 round trips,
                        // but the registers it takes would cost the decode
                        // kernels their second CTA per SM.)
                        const float *src = p.ws + static_cast<size_t>(blockIdx.x + 1) * (128u * BN) + row * BN + col0;
#pragma unroll 1
                        for (int q = 0; q < nsrc; ++q, src += 128 * BN) {
#pragma unroll
                            for (int j = 0; j < C::kCols; j += 4) {
                                const float4 v = __ldcg(reinterpret_cast<const float4 *>(src + j));
                                acc[j] += v.x;
                                acc[j + 1] += v.y;
                                acc[j + 2] += v.z;
                                acc[j + 3] += v.w;
                            }
                        }
                        // Every thread has read the partials: clear their
                        // flags for the next launch.
                        named_barrier_sync(1, C::kEpiThreads);
                        for (int q = etid; q < nsrc; q += C::kEpiThreads)
                            st_relaxed_gpu_u32(p.sk_flags + blockIdx.x + 1 + q, 0u);
                        if (etid == 0) FP8Q_TRACE_AT(p, kTrCluster2);   // stream-K: partials added
                    }
                    if (!got) continue;
                }
            }

            if (!SWAP && !BLOCKWISE) {
                // Stored (or published as a partial tile) above.
            } else if (split == 1) {
                // Scale, add bias, convert, store.
                if (SWAP) {
                    if (rn < p.N) {
#pragma unroll
                        for (int j = 0; j < C::kCols; ++j) {
                            const int m = m0 + col0 + j;
                            if (m < p.M) {
                                const float y = BLOCKWISE ? acc[j] + row_bias
                                                          : fmaf(acc[j] * row_scale, sColScale[col0 + j], row_bias);
                                store_out(out, static_cast<long long>(m) * p.ldo + rn, y);
                            }
                        }
                    }
                } else if (C::kTmaStore) {
                    // From the promoted row in registers, 32 columns at a time.
                    if constexpr (BLOCKWISE) {
                        uint8_t *sbuf = smem + C::kOffStage + static_cast<uint32_t>(ew) * C::kStageBufBytes;
                        const int ybox = m0 + quarter * 32;
#pragma unroll
                        for (int ch = 0; ch < C::kCols / 32; ++ch) {
                            const int cb = col0 + ch * 32;
                            uint32_t w[16];
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const int j = ch * 32 + 2 * e, c = cb + 2 * e;
                                w[e] = BLOCKWISE
                                           ? pack_out2<OutT>(acc[j] + sColBias[c], acc[j + 1] + sColBias[c + 1])
                                           : pack_out2<OutT>(fmaf(acc[j] * row_scale, sColScale[c], sColBias[c]),
                                                             fmaf(acc[j + 1] * row_scale, sColScale[c + 1],
                                                                  sColBias[c + 1]));
                            }
                            store_box_tma(&tm_out, sbuf, lane, w, n0 + cb, ybox, ybox < p.M && n0 + cb < p.N);
                        }
                    }
                } else if (rm < p.M) {
                    OutT *orow = out + static_cast<long long>(rm) * p.ldo;
#pragma unroll
                    for (int j = 0; j < C::kCols; j += 8) {
                        const int n = n0 + col0 + j;
                        float y[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int c = col0 + j + e;
                            y[e] = BLOCKWISE ? acc[j + e] + sColBias[c]
                                             : fmaf(acc[j + e] * row_scale, sColScale[c], sColBias[c]);
                        }
                        if (n + 8 <= p.N) {
                            uint4 v;
                            uint32_t *vw = reinterpret_cast<uint32_t *>(&v);
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const OutT lo = to_out<OutT>(y[2 * e]), hi = to_out<OutT>(y[2 * e + 1]);
                                vw[e] = static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(&lo)) |
                                        (static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(&hi)) << 16);
                            }
                            *reinterpret_cast<uint4 *>(orow + n) = v;
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                if (n + e < p.N) orow[n + e] = to_out<OutT>(y[e]);
                        }
                    }
                }
            } else if (push) {
                // Split-K, push: stage the partial tile row-major in the idle
                // ring, push each other rank's rows into its receive buffer
                // (bulk DSMEM copies completing on its mbarrier), then the
                // epilogue warps together add up the rows this CTA owns, over
                // the ranks in increasing order (a fixed order: the result is
                // deterministic).
                constexpr int SP = C::kPartStride;
                named_barrier_sync(1, C::kEpiThreads);
#pragma unroll
                for (int j = 0; j < C::kCols; j += 4)
                    *reinterpret_cast<float4 *>(sRed + row * SP + col0 + j) =
                        make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
                fence_proxy_async_smem();
                named_barrier_sync(1, C::kEpiThreads);
                const int slot_rows = 4 * ((32 + split - 1) / split);
                if (etid == 0) {
                    for (int q = 0; q < split; ++q) {
                        if (q == rank) continue;
                        const int q_lo = 4 * (32 * q / split), q_hi = 4 * (32 * (q + 1) / split);
                        const uint32_t src = smem_u32(sRed + q_lo * SP);
                        const uint32_t dst = dsmem_map(smem_u32(sRecv + rank * slot_rows * SP), q);
                        dsmem_bulk_push(dst, src, static_cast<uint32_t>((q_hi - q_lo) * SP * 4),
                                        dsmem_map(smem_u32(recv_full), q));
                    }
                    bulk_commit();
                }
                const int my_lo = 4 * (32 * rank / split), my_hi = 4 * (32 * (rank + 1) / split);
                const int my_rows = my_hi - my_lo;
                if (mbar_wait(recv_full, 0, abort, p.status)) {
                    // Items (owned row r, 4-column group c4), rows fastest so a
                    // warp's stores of one column group are contiguous in n.
                    for (int item = etid; item < my_rows * (BN / 4); item += C::kEpiThreads) {
                        const int c4 = item / my_rows;
                        const int r = my_lo + (item - c4 * my_rows);
                        float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
                        for (int q = 0; q < split; ++q) {
                            const float *src = q == rank ? sRed + r * SP
                                                         : sRecv + (q * slot_rows + (r - my_lo)) * SP;
                            const float4 v = *reinterpret_cast<const float4 *>(src + c4 * 4);
                            sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
                        }
                        const int n = n0 + r;
                        if (n < p.N) {
                            const float ws = BLOCKWISE ? 1.0f : __ldg(p.w_scale + n);
                            const float bv = p.bias != nullptr ? __bfloat162float(p.bias[n]) : 0.0f;
                            const float sv[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int m = m0 + c4 * 4 + e;
                                if (m < p.M) {
                                    const float y = BLOCKWISE ? sv[e] + bv : fmaf(sv[e] * ws, sColScale[c4 * 4 + e], bv);
                                    store_out(out, static_cast<long long>(m) * p.ldo + n, y);
                                }
                            }
                        }
                    }
                }
                // The pushed rows must have left this CTA's shared memory
                // before it may exit.
                if (etid == 0) bulk_wait_read();
            } else {
                // Split-K, pull or workspace: publish this CTA's partial tile
                // row-major with padded rows (the ring is idle: every copy was
                // consumed and every MMA has completed).
                constexpr int SP = C::kPartStride;
                named_barrier_sync(1, C::kEpiThreads);
#pragma unroll
                for (int j = 0; j < C::kCols; j += 4)
                    *reinterpret_cast<float4 *>(sRed + row * SP + col0 + j) =
                        make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
            }
            if (ew == 0 && lane == 0) FP8Q_TRACE_AT(p, kTrEpiDone);
        }
        // The staging buffers must have been read out by the TMA unit before
        // the CTA exits (the stores themselves complete with the grid).
        if (C::kTmaStore && lane == 0) bulk_wait_read();

    }

    bool exchanged = false;   // split-K partials reduced through the workspace
    if constexpr (C::kWsExchange) {
        if (split > 1 && p.ws != nullptr) {
            // (split > 1: one tile per cluster, tile index = cluster index)
            int a_t, b_t;
            coords(cluster_id, a_t, b_t);
            reduce_split_workspace<C, OutT, BLOCKWISE, SWAP>(p, smem, sColScale, ws_bar, rank, cluster_id, warp,
                                                             abort, (SWAP ? b_t : a_t) * C::kTokTile,
                                                             (SWAP ? a_t : b_t) * C::kColTile);
            exchanged = true;
        }
    }
    if constexpr (!C::kPush) {
        if (split > 1 && !exchanged) {
            cluster_sync();
            if (threadIdx.x == 32 * C::kEpiWarp0) FP8Q_TRACE_AT(p, kTrCluster1);
            if (warp >= C::kEpiWarp0 && !*abort) {
                // Reduce the tile's valid rows over the cluster in rank
                // order.  Items are (row, 4-column group) with the columns
                // fastest, so a warp's DSMEM reads and its 8-byte output
                // stores are contiguous; each rank takes an equal share of
                // the items (a share of the columns when the tile holds few
                // tokens).
                constexpr int SP = C::kPartStride;
                constexpr int G = BN / 4;
                const int etid = threadIdx.x - 32 * C::kEpiWarp0;
                int a_t, b_t;
                coords(cluster_id, a_t, b_t);
                const int m0 = a_t * C::kTokTile;
                const int n0 = b_t * C::kColTile;
                const int rows = p.M - m0 < C::kTokTile ? p.M - m0 : C::kTokTile;
                const int items = rows * G;
                const int i_lo = static_cast<int>(static_cast<long long>(items) * rank / split);
                const int i_hi = static_cast<int>(static_cast<long long>(items) * (rank + 1) / split);
                OutT *out = static_cast<OutT *>(p.out);
                const uint32_t red_base = smem_u32(sRed);
                for (int item = i_lo + etid; item < i_hi; item += C::kEpiThreads) {
                    const int r = item / G;
                    const int c4 = item - r * G;
                    const int m = m0 + r, n = n0 + 4 * c4;
                    if (n >= p.N) continue;
                    const uint32_t off = static_cast<uint32_t>((r * SP + c4 * 4) * 4);
                    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int q = 0; q < split; ++q) {
                        const float4 v = dsmem_ld_f4(dsmem_map(red_base + off, static_cast<uint32_t>(q)));
                        sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
                    }
                    const float sv[4] = {sum.x, sum.y, sum.z, sum.w};
                    const float am = BLOCKWISE ? 1.0f : __ldg(p.a_scale + m);
                    float y[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const bool in = n + e < p.N;
                        const float bv = (p.bias != nullptr && in) ? __bfloat162float(p.bias[n + e]) : 0.0f;
                        y[e] = BLOCKWISE ? sv[e] + bv : fmaf(sv[e] * am, in ? __ldg(p.w_scale + n + e) : 0.0f, bv);
                    }
                    OutT *o = out + static_cast<long long>(m) * p.ldo + n;
                    if (n + 4 <= p.N) {
                        *reinterpret_cast<uint2 *>(o) = make_uint2(pack_out2<OutT>(y[0], y[1]), pack_out2<OutT>(y[2], y[3]));
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (n + e < p.N) o[e] = to_out<OutT>(y[e]);
                    }
                }
            }
            if (threadIdx.x == 32 * C::kEpiWarp0) FP8Q_TRACE_AT(p, kTrReduced);
            cluster_sync();
            if (threadIdx.x == 32 * C::kEpiWarp0) FP8Q_TRACE_AT(p, kTrCluster2);
        }
    }

    tc_fence_before();
    __syncthreads();
    // Paired: neither CTA may exit while the other can still load into its
    // shared memory (the odd CTA's loads signal the even CTA's barriers) or
    // arrive on its barriers.
    if (pair) cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        if (TWO_SM) tmem_dealloc_pair(tmem_base, C::kTmemCols);
        else tmem_dealloc(tmem_base, C::kTmemCols);
        if (lane == 0) FP8Q_TRACE_AT(p, kTrExit);
    }
}

}  // namespace fp8q
