// gemm_blockwise.cu -- 1x128 x 128x128 blockwise scaled FP8 GEMM instances.
#include "gemm_instances.cuh"

namespace fp8q {

cudaError_t launch_gemm_blockwise(const GemmProblem &p, const GemmLaunch &l, unsigned *status, cudaStream_t st)
{
    return p.out_fp16 ? dispatch_gemm<true, __half>(p, l, status, st)
                      : dispatch_gemm<true, __nv_bfloat16>(p, l, status, st);
}

}  // namespace fp8q
