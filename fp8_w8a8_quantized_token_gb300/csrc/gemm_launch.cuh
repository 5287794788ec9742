// gemm_launch.cuh -- host-side launch of one fp8_gemm_kernel instantiation:
// tensor maps, kernel attributes, cluster launch.
#pragma once

#include <cuda_runtime.h>

#include <atomic>

#include "gemm_kernel.cuh"
#include "internal.h"

namespace fp8q {

constexpr int kMaxDevices = 64;

template <bool SWAP, int BN, int STAGES, bool BLOCKWISE, typename OutT, bool TWO_SM = false, bool FQ = false,
          bool W16 = false, bool WIDE = false>
cudaError_t launch_gemm_inst(const GemmProblem &pr, const GemmLaunch &l, unsigned *status, cudaStream_t st)
{
    using C = GemmCfg<SWAP, BN, STAGES, BLOCKWISE, TWO_SM, FQ, W16, WIDE>;
    auto kernel = fp8_gemm_kernel<SWAP, BN, STAGES, BLOCKWISE, OutT, TWO_SM, FQ, W16, WIDE>;
    // Double-K-block stages: whole 128-wide K blocks, one CTA per tile along K.
    if (WIDE && (pr.K % 128 != 0 || l.split != 1)) return cudaErrorInvalidValue;

    static std::atomic<uint64_t> attr_done[kMaxDevices / 64 + 1];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done[dev >> 6].load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::kSmemBytes));
        if (e != cudaSuccess) return e;
        if constexpr (C::kRegSplit) {
            // The register split hands exactly the launch allocation between
            // the warpgroups; with any other per-thread count its
            // setmaxnreg.inc could never be satisfied, so refuse to launch.
            cudaFuncAttributes fa;
            e = cudaFuncGetAttributes(&fa, kernel);
            if (e != cudaSuccess) return e;
            if (fa.numRegs != C::kLaunchRegs) return cudaErrorInvalidKernelImage;
        }
        attr_done[dev >> 6].fetch_or(bit, std::memory_order_acq_rel);
    }

    // Operand maps: e4m3 rows of K bytes, boxes of 128 (K) x rows.
    CUtensorMap tm_w, tm_x, tm_sa;
    const int tok_box = C::kTokTile;
    const bool pair = TWO_SM;   // 2-CTA MMA pairs (non-swapped channelwise, split 1)
    // Paired tiles: each CTA loads half of the weight rows of the tile.
    const int wrow_box = SWAP ? 128 : (pair ? BN / 2 : BN);
    if (WIDE) {
        if (!make_tmap_3d_kblocks(&tm_w, pr.w, static_cast<uint64_t>(pr.K), static_cast<uint64_t>(pr.N),
                                  static_cast<uint64_t>(pr.ldw), static_cast<uint32_t>(wrow_box)))
            return cudaErrorInvalidValue;
    } else if (!make_tmap_2d(&tm_w, pr.w, CU_TENSOR_MAP_DATA_TYPE_UINT8, static_cast<uint64_t>(pr.K),
                             static_cast<uint64_t>(pr.N), static_cast<uint64_t>(pr.ldw), 128, wrow_box,
                             CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    // FQ: the bf16 activations are copied by the kernel's quantizing warps
    // (GemmArgs::x); the activation map slot holds the weight map, unused.
    // W16: bf16 activations [M, K] with row stride lda, boxes of 64 columns
    // (128 bytes) x the tile's tokens, 128-byte swizzle: two per K block.
    if (FQ)
        tm_x = tm_w;
    else if (WIDE) {
        if (!make_tmap_3d_kblocks(&tm_x, pr.a, static_cast<uint64_t>(pr.K), static_cast<uint64_t>(pr.M),
                                  static_cast<uint64_t>(pr.K), static_cast<uint32_t>(tok_box)))
            return cudaErrorInvalidValue;
    } else if (W16) {
        if (!make_tmap_2d(&tm_x, pr.a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<uint64_t>(pr.K),
                          static_cast<uint64_t>(pr.M), static_cast<uint64_t>(pr.lda) * 2u, 64, tok_box,
                          CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    } else if (!make_tmap_2d(&tm_x, pr.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, static_cast<uint64_t>(pr.K),
                           static_cast<uint64_t>(pr.M), static_cast<uint64_t>(pr.K), 128, tok_box,
                           CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    // Output (non-swapped tiles): 2-byte values [M, N], row stride N, boxes
    // of 32 x 32 with the 64-byte swizzle of the epilogue's staging buffers.
    CUtensorMap tm_out = tm_x;
    if (C::kTmaStore &&
        !make_tmap_2d(&tm_out, pr.out, CU_TENSOR_MAP_DATA_TYPE_UINT16, static_cast<uint64_t>(pr.N),
                      static_cast<uint64_t>(pr.M), static_cast<uint64_t>(pr.N) * 2u, 32, 32,
                      CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    if (BLOCKWISE && !FQ) {
        // Column-major activation scales: K/128 columns of m_pad floats; only
        // the first M entries of each column are real (the rest read as 0).
        if (!make_tmap_2d(&tm_sa, pr.a_scale, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, static_cast<uint64_t>(pr.M),
                          static_cast<uint64_t>(pr.K / 128), static_cast<uint64_t>(pr.m_pad) * 4u, tok_box, 1,
                          CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    } else {
        tm_sa = tm_x;  // unused
    }

    GemmArgs a;
    a.M = static_cast<int>(pr.M);
    a.N = static_cast<int>(pr.N);
    a.K = static_cast<int>(pr.K);
    a.num_kb = static_cast<int>((pr.K + 127) / 128);
    a.m_tiles = static_cast<int>((pr.M + C::kTokTile - 1) / C::kTokTile);
    a.n_tiles = static_cast<int>((pr.N + C::kColTile - 1) / C::kColTile);
    a.pair = pair ? 1 : 0;
    a.num_tiles = (pair ? (a.m_tiles + 1) / 2 : a.m_tiles) * a.n_tiles;
    a.split = pair ? 1 : l.split;
    // Non-swapped tiles with more weight tiles than token tiles group the
    // weight tiles (each weight tile is then fetched by few concurrent CTAs
    // while the smaller activation matrix stays in L2).
    a.raster_b = (!SWAP && pr.N > pr.M) ? 1 : 0;
    a.group = SWAP ? a.n_tiles : 8;
    if (a.group < 1) a.group = 1;
    a.a_scale = pr.a_scale;
    a.w_scale = pr.w_scale;
    a.bias = static_cast<const __nv_bfloat16 *>(pr.bias);
    a.out = pr.out;
    a.ldo = pr.N;
    a.status = status;
    a.trace = trace_buffer(&a.trace_stages);
    a.prefetch_kb = prefetch_kblocks(SWAP, BLOCKWISE, l.grid);
    a.preload = pr.preload ? 1 : 0;
    a.eps = pr.eps;
    a.x = FQ ? static_cast<const __nv_bfloat16 *>(pr.a) : nullptr;
    a.ldx = pr.lda;
    // Split-K partials go through the workspace when the instantiation
    // exchanges that way and the caller gave a workspace large enough for
    // this schedule (one 128 x BN slot per CTA); the owner's rows arrive in
    // at most kWsBars chunks.
    const size_t ws_need = static_cast<size_t>(a.num_tiles) * static_cast<size_t>(a.split) * 128u * BN * 4u;
    bool use_ws = C::kWsExchange && a.split > 1 && pr.ws != nullptr && pr.ws_bytes >= ws_need &&
                  workspace_exchange_enabled();
    if (use_ws) {
        const uint32_t cr = C::kLandBytes / (2u * static_cast<uint32_t>(a.split - 1) * C::kPartStride * 4u);
        const uint32_t owned = (128u + static_cast<uint32_t>(a.split) - 1u) / static_cast<uint32_t>(a.split);
        use_ws = cr >= 1 && (owned + cr - 1) / cr <= static_cast<uint32_t>(C::kWsBars);
    }
    a.ws = use_ws ? static_cast<float *>(pr.ws) : nullptr;
    // Stream-K (the caller checked the workspace size): slots, then flags.
    a.stream_k = 0;
    a.sk_flags = nullptr;
    if (l.stream_k) {
        if (!C::kStreamK || l.split != 1 || pr.ws == nullptr) return cudaErrorInvalidValue;
        a.stream_k = 1;
        a.ws = static_cast<float *>(pr.ws);
        a.sk_flags = reinterpret_cast<unsigned *>(static_cast<char *>(pr.ws) +
                                                  static_cast<size_t>(l.grid) * 128u * BN * 4u);
    }

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(l.grid));
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    const int csize = pair ? 2 : l.split;
    if (csize > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = static_cast<unsigned>(csize);
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    // A operand: the 128-row side of the MMA; B operand: the BN-row side.
    const CUtensorMap &tm_a = SWAP ? tm_w : tm_x;
    const CUtensorMap &tm_b = SWAP ? tm_x : tm_w;
    return cudaLaunchKernelEx(&cfg, kernel, tm_a, tm_b, tm_sa, tm_out, a);
}

}  // namespace fp8q
