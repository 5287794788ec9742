// gemm_channelwise.cu -- per-token x per-channel scaled FP8 GEMM instances.
#include "gemm_instances.cuh"

namespace fp8q {

cudaError_t launch_gemm_channelwise(const GemmProblem &p, const GemmLaunch &l, unsigned *status, cudaStream_t st)
{
    return p.out_fp16 ? dispatch_gemm<false, __half>(p, l, status, st)
                      : dispatch_gemm<false, __nv_bfloat16>(p, l, status, st);
}

}  // namespace fp8q
