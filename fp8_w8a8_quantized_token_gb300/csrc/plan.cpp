// plan.cpp -- GEMM schedule selection (host only).
//
// A compiled-in table keyed by (N, K, scheme) holds the schedules that
// tune.py's sweep on GB300 found fastest at a set of M values; a problem
// takes the entry of the nearest M, ties going to the smaller M (the
// nearest-M rule of get_w8a8_channelwise_fp8_config on the "Tune FP8 GEMM
// Triton tiles on L40S and enable by default" page, key source snippets,
// whose keys are scanned in ascending order), except that a smaller-M row
// whose token tile M outgrows is passed over for a larger-M row (the
// schedules here fix the token tile, the page's configs only block sizes).
// Shapes without a table entry
// use the generic rule.  fp8q_set_plan_override (or FP8Q_PLAN="swap,mma_n,
// split" at start-up) forces a schedule for tests and sweeps; FP8Q_LOG=1
// prints each new choice once to stderr.
#include <stdio.h>
#include <stdlib.h>

#include <atomic>
#include <mutex>
#include <set>
#include <tuple>

#include "../../include/fp8q.h"
#include "internal.h"

namespace fp8q {
namespace {

struct TableEntry {
    int64_t N, K;
    int blockwise;
    int64_t M;
    int swap_ab, mma_n, split;
};

// Rows "{N, K, blockwise, M, swap_ab, mma_n, split}," from the sweep
// (split 0: stream-K).
const TableEntry kTable[] = {
#include "tile_table.inc"
    {0, 0, 0, 0, 0, 0, 0}};
const int kTableSize = static_cast<int>(sizeof(kTable) / sizeof(kTable[0])) - 1;

int next_pow2(int64_t v)
{
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

// Generic rule (shapes without table rows), following what the sweep found
// on the measured shapes: up to 64 tokens the weights take the MMA's
// 128-row side and the tokens its N side (smallest MMA N >= M); up to 512
// tokens 128-token swapped tiles; beyond that 128 x 256 tiles.  If the tiles
// cannot fill the GPU, K is split across a cluster of 2, 4 or 8 CTAs (odd
// cluster sizes measured slower).
void generic_rule(int64_t M, int64_t N, int64_t K, int num_sms, fp8q_plan *pl)
{
    if (M <= 64) {
        pl->swap_ab = 1;
        pl->mma_n = next_pow2(M < 16 ? 16 : M);
    } else if (M <= 512) {
        pl->swap_ab = 1;
        pl->mma_n = 128;
    } else {
        pl->swap_ab = 0;
        pl->mma_n = 256;
    }
    const int tile_m = pl->swap_ab ? pl->mma_n : 128;
    const int tile_n = pl->swap_ab ? 128 : pl->mma_n;
    const int64_t tiles = ((M + tile_m - 1) / tile_m) * ((N + tile_n - 1) / tile_n);
    int split = 1;
    while (split < 8 && tiles * split * 2 <= num_sms) split *= 2;
    pl->split_k = split;
}

// Process-wide schedule override (fp8q_set_plan_override), initialised
// from FP8Q_PLAN="swap,mma_n,split".
std::atomic<int> g_ovr_swap{-2}, g_ovr_n{0}, g_ovr_split{0};

bool override_plan(fp8q_plan *pl)
{
    if (g_ovr_swap.load() == -2) {
        int swap = -1, mma_n = 0, split = 0;
        const char *s = getenv("FP8Q_PLAN");
        if (s == nullptr || sscanf(s, "%d,%d,%d", &swap, &mma_n, &split) != 3 ||
            !gemm_shape_supported(swap != 0, mma_n))
            swap = -1;
        g_ovr_n.store(mma_n);
        g_ovr_split.store(split);
        int expected = -2;
        g_ovr_swap.compare_exchange_strong(expected, swap);
    }
    const int swap = g_ovr_swap.load();
    if (swap < 0) return false;
    pl->swap_ab = swap;
    pl->mma_n = g_ovr_n.load();
    pl->split_k = g_ovr_split.load();
    return true;
}

// Token tiles of a row's schedule at M tokens.
int64_t token_tiles(const TableEntry &e, int64_t M)
{
    const int64_t tile_m = e.swap_ab ? e.mma_n : 128;
    return (M + tile_m - 1) / tile_m;
}

bool table_plan(int64_t M, int64_t N, int64_t K, int blockwise, fp8q_plan *pl)
{
    // A row swept at a smaller M is not taken where M needs more token tiles
    // than that row's M did (every weight tile would be read once more per
    // extra token tile) while a row at a larger M exists: blockwise 4096 x
    // 7168 at M = 17 ran 18.5 us on the M = 16 row's 16-token tiles and
    // 11.5 us on the M = 32 row's 32-token tile.
    bool larger = false;
    for (int i = 0; i < kTableSize; ++i) {
        const TableEntry &e = kTable[i];
        if (e.N == N && e.K == K && e.blockwise == blockwise && e.M >= M) larger = true;
    }
    const TableEntry *best = nullptr;
    int64_t best_d = 0;
    for (int i = 0; i < kTableSize; ++i) {
        const TableEntry &e = kTable[i];
        if (e.N != N || e.K != K || e.blockwise != blockwise) continue;
        if (larger && e.M < M && token_tiles(e, M) > token_tiles(e, e.M)) continue;
        const int64_t d = e.M > M ? e.M - M : M - e.M;
        if (best == nullptr || d < best_d || (d == best_d && e.M < best->M)) {
            best = &e;
            best_d = d;
        }
    }
    if (best == nullptr || !gemm_shape_supported(best->swap_ab != 0, best->mma_n)) return false;
    pl->swap_ab = best->swap_ab;
    pl->mma_n = best->mma_n;
    pl->split_k = best->split;
    return true;
}

}  // namespace

bool plan_override_active()
{
    fp8q_plan pl = {};
    return override_plan(&pl);
}

size_t plan_workspace_bytes(int64_t M, int64_t N, int swap_ab, int mma_n, int split_k)
{
    // Only partial tiles of 64 KB and more (128 x 128 floats) go through the
    // workspace, and only when the workspace exchange is enabled.
    if (split_k <= 1 || (swap_ab && mma_n < 128) || !workspace_exchange_enabled()) return 0;
    const int64_t tile_m = swap_ab ? mma_n : 128, tile_n = swap_ab ? 128 : mma_n;
    const int64_t tiles = ((M + tile_m - 1) / tile_m) * ((N + tile_n - 1) / tile_n);
    return static_cast<size_t>(tiles) * static_cast<size_t>(split_k) * 128u * static_cast<size_t>(mma_n) * 4u;
}

size_t stream_k_workspace_bytes(int grid, int mma_n)
{
    return static_cast<size_t>(grid) * (128u * static_cast<size_t>(mma_n) * 4u + 4u);
}

// Tile sizes, grid and persistence for a chosen (swap_ab, mma_n, split_k);
// split_k 0 with swapped tiles asks for stream-K.
void plan_finish(int64_t M, int64_t N, int64_t K, int blockwise, int num_sms, fp8q_plan *pl)
{
    pl->kb_per_stage = 1;
    pl->tile_m = pl->swap_ab ? pl->mma_n : 128;
    pl->tile_n = pl->swap_ab ? 128 : pl->mma_n;
    const int64_t tiles = ((M + pl->tile_m - 1) / pl->tile_m) * ((N + pl->tile_n - 1) / pl->tile_n);
    const int64_t num_kb = (K + 127) / 128;
    if (pl->swap_ab && pl->mma_n <= 32 && pl->split_k == 0) {
        // Stream-K: at most one CTA per SM (every CTA must be resident for
        // the partial hand-over) and at least one K block per CTA.
        const int64_t total = tiles * num_kb;
        const int64_t sms = num_sms > 0 ? num_sms : 1;
        pl->stream_k = 1;
        pl->split_k = 1;
        pl->pair = 0;
        pl->two_sm = 0;
        pl->grid = static_cast<int32_t>(total < sms ? total : sms);
        pl->persistent = 1;
        pl->stages = stream_k_stages(pl->mma_n);
        return;
    }
    pl->stream_k = 0;
    int64_t split = pl->split_k;
    if (split > 8) split = 8;
    if (split > num_kb) split = num_kb;
    if (split < 1) split = 1;
    pl->split_k = static_cast<int32_t>(split);
    // Channelwise 256-column tiles on adjacent token tiles run as CTA pairs
    // with 2-CTA MMAs (256 tokens x 256 columns per pair, each CTA loading
    // half of the weight rows) whenever there are two token tiles to pair.
    // Blockwise tiles stay single: their per-K-block promotion hands each
    // accumulator slot back to the MMA every K block, which a 2-CTA MMA would
    // couple across both CTAs' epilogues.  FP8Q_NO_PAIR=1 turns pairs off.
    static const bool no_pair = getenv("FP8Q_NO_PAIR") != nullptr && getenv("FP8Q_NO_PAIR")[0] == '1';
    const int64_t m_tiles = (M + pl->tile_m - 1) / pl->tile_m;
    pl->pair = (!pl->swap_ab && !blockwise && pl->mma_n == 256 && split == 1 && m_tiles >= 2 && !no_pair) ? 1 : 0;
    if (pl->pair) {
        const int64_t pairs = ((m_tiles + 1) / 2) * ((N + pl->tile_n - 1) / pl->tile_n);
        const int64_t max_pairs = num_sms / 2 > 0 ? num_sms / 2 : 1;
        pl->grid = static_cast<int32_t>(2 * (pairs < max_pairs ? pairs : max_pairs));
        pl->persistent = pairs > max_pairs ? 1 : 0;
    } else if (split > 1) {
        pl->grid = static_cast<int32_t>(tiles * split);
        pl->persistent = 0;
    } else {
        pl->grid = static_cast<int32_t>(tiles < num_sms ? tiles : num_sms);
        pl->persistent = tiles > num_sms ? 1 : 0;
    }
    pl->two_sm = pl->pair;
    pl->stages = pl->two_sm ? kTwoSmStages : stages_for(pl->swap_ab != 0, pl->mma_n);
    // Narrow channelwise tiles over whole K blocks, K not split: stages of
    // two K blocks.
    if (!blockwise && !pl->swap_ab && !pl->pair && pl->split_k == 1 && K % 128 == 0 && pl->mma_n <= 128) {
        pl->kb_per_stage = 2;
        pl->stages = wide_stages(pl->mma_n);
    }
}

void plan_without_stream_k(int64_t M, int64_t N, int64_t K, int blockwise, int num_sms, fp8q_plan *pl)
{
    const int64_t tiles = ((M + pl->tile_m - 1) / pl->tile_m) * ((N + pl->tile_n - 1) / pl->tile_n);
    int split = 1;
    while (split < 8 && tiles * split * 2 <= num_sms) split *= 2;
    pl->split_k = split;
    plan_finish(M, N, K, blockwise, num_sms, pl);
}

}  // namespace fp8q

extern "C" fp8q_status fp8q_gemm_plan(int64_t M, int64_t N, int64_t K, int32_t blockwise, int32_t num_sms,
                                      fp8q_plan *plan)
{
    using namespace fp8q;
    if (plan == nullptr || M < 0 || N <= 0 || K <= 0) return FP8Q_ERR_INVALID_ARG;
    if (num_sms <= 0) {
        num_sms = current_device_sms();
        if (num_sms <= 0) return FP8Q_ERR_CUDA;
    }
    fp8q_plan pl = {};
    if (override_plan(&pl)) {
        pl.from_table = 0;
    } else if (table_plan(M, N, K, blockwise ? 1 : 0, &pl)) {
        pl.from_table = 1;
    } else {
        generic_rule(M, N, K, num_sms, &pl);
        pl.from_table = 0;
    }
    plan_finish(M, N, K, blockwise ? 1 : 0, num_sms, &pl);
    static const bool log = getenv("FP8Q_LOG") != nullptr && getenv("FP8Q_LOG")[0] == '1';
    if (log) {
        static std::mutex mu;
        static std::set<std::tuple<int64_t, int64_t, int64_t, int>> seen;
        std::lock_guard<std::mutex> g(mu);
        if (seen.insert(std::make_tuple(M, N, K, blockwise)).second)
            fprintf(stderr, "fp8q plan M=%lld N=%lld K=%lld %s: swap_ab=%d mma_n=%d split_k=%d pair=%d stream_k=%d "
                    "grid=%d%s\n",
                    static_cast<long long>(M), static_cast<long long>(N), static_cast<long long>(K),
                    blockwise ? "blockwise" : "channelwise", pl.swap_ab, pl.mma_n, pl.split_k, pl.pair, pl.stream_k,
                    pl.grid, pl.from_table ? " (table)" : "");
    }
    *plan = pl;
    return FP8Q_OK;
}

extern "C" size_t fp8q_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t blockwise)
{
    using namespace fp8q;
    fp8q_plan pl;
    if (M <= 0 || fp8q_gemm_plan(M, N, K, blockwise, 0, &pl) != FP8Q_OK) return 0;
    if (pl.stream_k) return stream_k_workspace_bytes(pl.grid, pl.mma_n);
    return plan_workspace_bytes(M, N, pl.swap_ab, pl.mma_n, pl.split_k);
}

extern "C" fp8q_status fp8q_set_plan_override(int32_t swap_ab, int32_t mma_n, int32_t split_k)
{
    using namespace fp8q;
    if (swap_ab < 0) {
        g_ovr_swap.store(-1);
        return FP8Q_OK;
    }
    if (swap_ab > 1 || !gemm_shape_supported(swap_ab != 0, mma_n) || split_k < 0 ||
        (split_k == 0 && (swap_ab != 1 || mma_n > 32)))
        return FP8Q_ERR_INVALID_ARG;
    g_ovr_n.store(mma_n);
    g_ovr_split.store(split_k);
    g_ovr_swap.store(swap_ab);
    return FP8Q_OK;
}
