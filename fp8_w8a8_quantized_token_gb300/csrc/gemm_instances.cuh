// gemm_instances.cuh -- the instantiations a translation unit provides:
// swapped (decode) tiles of 16/32/64/128 tokens (16 and 32 also as stream-K
// instantiations with a deeper ring) and non-swapped tiles of
// 128 tokens x 256 output columns (prefill; 2-CTA pairs for channelwise)
// or 128 / 64 / 32 columns (mid-size M), bf16 or fp16 output.
#pragma once

#include "gemm_launch.cuh"

namespace fp8q {

template <bool BLOCKWISE, typename OutT>
cudaError_t dispatch_gemm(const GemmProblem &p, const GemmLaunch &l, unsigned *status, cudaStream_t st)
{
    if (p.w16) {
        // Weight-only FP8 (bf16 activations): swapped 16- or 32-token tiles.
        if constexpr (!BLOCKWISE) {
            if (l.swap_ab && l.mma_n == 16)
                return launch_gemm_inst<true, 16, kW16Stages, false, OutT, false, false, true>(p, l, status, st);
            if (l.swap_ab && l.mma_n == 32)
                return launch_gemm_inst<true, 32, kW16Stages, false, OutT, false, false, true>(p, l, status, st);
        }
        return cudaErrorInvalidValue;
    }
    if (p.fused_quant) {
        // Quantization fused into the GEMM: blockwise 16- and 32-token decode tiles.
        if constexpr (BLOCKWISE)
            if (l.swap_ab && l.mma_n == 16)
                return launch_gemm_inst<true, 16, kFusedQuantStages, true, OutT, false, true>(p, l, status, st);
        if constexpr (BLOCKWISE)
            if (l.swap_ab && l.mma_n == 32)
                return launch_gemm_inst<true, 32, kFusedQuantStages32, true, OutT, false, true>(p, l, status, st);
        return cudaErrorInvalidValue;
    }
    if (l.swap_ab && l.stream_k) {
        // Stream-K: one CTA per SM at most, a deeper ring.
        if (l.mma_n == 16)
            return launch_gemm_inst<true, 16, stream_k_stages(16), BLOCKWISE, OutT>(p, l, status, st);
        if (l.mma_n == 32)
            return launch_gemm_inst<true, 32, stream_k_stages(32), BLOCKWISE, OutT>(p, l, status, st);
        return cudaErrorInvalidValue;
    }
    if (l.swap_ab) {
        switch (l.mma_n) {
            case 16: return launch_gemm_inst<true, 16, stages_for(true, 16), BLOCKWISE, OutT>(p, l, status, st);
            case 32: return launch_gemm_inst<true, 32, stages_for(true, 32), BLOCKWISE, OutT>(p, l, status, st);
            case 64: return launch_gemm_inst<true, 64, stages_for(true, 64), BLOCKWISE, OutT>(p, l, status, st);
            case 128: return launch_gemm_inst<true, 128, stages_for(true, 128), BLOCKWISE, OutT>(p, l, status, st);
            default: return cudaErrorInvalidValue;
        }
    }
    if constexpr (!BLOCKWISE) {
        // Narrow channelwise tiles over whole 128-wide K blocks, K not split:
        // stages of two K blocks.
        if (l.wide) {
            switch (l.mma_n) {
                case 128: return launch_gemm_inst<false, 128, wide_stages(128), false, OutT, false, false, false, true>(p, l, status, st);
                case 64: return launch_gemm_inst<false, 64, wide_stages(64), false, OutT, false, false, false, true>(p, l, status, st);
                case 32: return launch_gemm_inst<false, 32, wide_stages(32), false, OutT, false, false, false, true>(p, l, status, st);
                default: break;
            }
        }
    }
    switch (l.mma_n) {
        case 256:
            if constexpr (!BLOCKWISE)
                if (l.pair && l.two_sm)
                    return launch_gemm_inst<false, 256, kTwoSmStages, false, OutT, true>(p, l, status, st);
            return launch_gemm_inst<false, 256, stages_for(false, 256), BLOCKWISE, OutT>(p, l, status, st);
        // Narrow weight tiles: mid-size M with one tile per CTA and no K split.
        case 128: return launch_gemm_inst<false, 128, stages_for(false, 128), BLOCKWISE, OutT>(p, l, status, st);
        case 64: return launch_gemm_inst<false, 64, stages_for(false, 64), BLOCKWISE, OutT>(p, l, status, st);
        case 32: return launch_gemm_inst<false, 32, stages_for(false, 32), BLOCKWISE, OutT>(p, l, status, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fp8q
