// selftest.cu -- fp8q_selftest_wait_timeout: a diagnostics kernel whose
// pipeline wait can never complete, to show that the library's bounded
// waits report a stalled pipeline (FP8Q_ERR_TIMEOUT in the device status
// word) and return instead of hanging the GPU.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fp8q.h"
#include "device_common.cuh"
#include "internal.h"

namespace fp8q {
namespace {

// One warp: thread 0 initialises an mbarrier that expects one arrival, which
// nothing ever makes, and waits for its first phase with the same bounded
// wait the GEMM's pipeline uses.  After kWaitTimeoutNs the wait records the
// timeout in *status and the kernel returns.
__global__ void __launch_bounds__(32) stalled_wait_kernel(unsigned *status)
{
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, &abort_flag, status);
    __syncwarp();
}

}  // namespace
}  // namespace fp8q

extern "C" fp8q_status fp8q_selftest_wait_timeout(void *stream)
{
    using namespace fp8q;
    unsigned *status = device_status_ptr();
    if (status == nullptr) return FP8Q_ERR_CUDA;
    stalled_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status);
    return cudaGetLastError() == cudaSuccess ? FP8Q_OK : FP8Q_ERR_CUDA;
}
