// selftest.cu -- diagnostics entry points:
//   fp8q_selftest_wait_timeout: a kernel whose pipeline wait can never
//     complete, to show that the library's bounded waits report a stalled
//     pipeline (FP8Q_ERR_TIMEOUT in the device status word) and return
//     instead of hanging the GPU;
//   fp8q_selftest_silu_mul: the fused group quantizer's silu(a) * b
//     evaluated elementwise, so its fp32 results can be compared bit for bit.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fp8q.h"
#include "device_common.cuh"
#include "internal.h"
#include "quant_common.cuh"

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

// out[i] = silu(a[i]) * b[i] with the quantizer's device function, two
// elements per thread.
__global__ void __launch_bounds__(256) silu_mul_kernel(const float *__restrict__ a, const float *__restrict__ b,
                                                       float *__restrict__ out, int64_t n)
{
    const int64_t i = 2 * (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x);
    if (i >= n) return;
    const bool two = i + 1 < n;
    const float2 r = silu_mul2(make_float2(a[i], two ? a[i + 1] : 0.0f), make_float2(b[i], two ? b[i + 1] : 0.0f));
    out[i] = r.x;
    if (two) out[i + 1] = r.y;
}

}  // namespace
}  // namespace fp8q

extern "C" fp8q_status fp8q_selftest_silu_mul(const float *a, const float *b, float *out, int64_t n, void *stream)
{
    using namespace fp8q;
    if (n < 0 || n > (int64_t{1} << 40)) return FP8Q_ERR_INVALID_ARG;
    if (n == 0) return FP8Q_OK;
    if (a == nullptr || b == nullptr || out == nullptr) return FP8Q_ERR_INVALID_ARG;
    const int64_t threads = (n + 1) / 2;
    const int64_t blocks = (threads + 255) / 256;
    if (blocks > 0x7FFFFFFF) return FP8Q_ERR_INVALID_ARG;
    silu_mul_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(a, b, out, n);
    return cudaGetLastError() == cudaSuccess ? FP8Q_OK : FP8Q_ERR_CUDA;
}

extern "C" fp8q_status fp8q_selftest_wait_timeout(void *stream)
{
    using namespace fp8q;
    unsigned *status = device_status_ptr();
    if (status == nullptr) return FP8Q_ERR_CUDA;
    stalled_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status);
    return cudaGetLastError() == cudaSuccess ? FP8Q_OK : FP8Q_ERR_CUDA;
}
