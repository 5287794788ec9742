// noalloc.cu -- fp8q_linear_channelwise_noalloc: the channelwise linear layer
// (per-token quantization, then the scaled GEMM) with its intermediate
// buffers in a fixed, library-owned device array instead of caller memory.
//
// fp8q_linear_channelwise needs two scratch buffers between its two
// kernels: the E4M3 codes of x and the per-token scales.  Some callers have
// no way to provide them: their device memory is handed out entirely by a
// host framework's pool (plugins that receive no workspace, engines that
// budget every byte in advance), or they cannot afford the implicit device
// synchronisation of cudaMalloc / cudaFree inside a latency-bound decode
// loop.  This entry point takes the scratch from a file-scope __device__
// array instead, so it allocates nothing.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/fp8q.h"
#include "internal.h"

namespace fp8q {
namespace {

// Capacity of the array: codes for up to kNoAllocMaxCodes elements of x
// (M * K) followed by up to kNoAllocMaxRows per-token scales.  Every GPU
// that loads the library holds these 16 MiB + 64 KiB until the process
// exits.
constexpr int64_t kNoAllocMaxCodes = FP8Q_NOALLOC_MAX_CODES;
constexpr int64_t kNoAllocMaxRows = FP8Q_NOALLOC_MAX_ROWS;
static_assert(kNoAllocMaxCodes % 256 == 0, "the scales must start 256-byte aligned");
constexpr size_t kScaleOffset = static_cast<size_t>(kNoAllocMaxCodes);
constexpr size_t kScratchBytes = kScaleOffset + static_cast<size_t>(kNoAllocMaxRows) * sizeof(float);

}  // namespace
}  // namespace fp8q

// The scratch array itself (file scope).
static __device__ __align__(256) uint8_t g_noalloc_scratch[fp8q::kScratchBytes];

namespace fp8q {
namespace {

constexpr int kMaxDev = 64;
std::atomic<uint8_t *> g_scratch_addr[kMaxDev];

// Device address of g_noalloc_scratch on the current device, resolved once
// per device with that device current.  In host code the symbol itself is
// only a host-side stand-in and must never reach a kernel.
uint8_t *scratch_address()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
    uint8_t *p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr) return nullptr;
        p = static_cast<uint8_t *>(addr);
        g_scratch_addr[dev].store(p, std::memory_order_release);
    }
    return p;
}

}  // namespace
}  // namespace fp8q

extern "C" fp8q_status fp8q_linear_channelwise_noalloc(const void *x, const void *b, int64_t ldb,
                                                       const float *b_scale, const void *bias, void *out, int64_t M,
                                                       int64_t N, int64_t K, fp8q_out_dtype out_dtype, void *stream)
{
    using namespace fp8q;
    if (M < 0 || K <= 0) return FP8Q_ERR_INVALID_ARG;
    if (M == 0) return fp8q_linear_channelwise(x, b, ldb, b_scale, bias, out, M, N, K, nullptr, nullptr, out_dtype,
                                               nullptr, 0, stream);
    // Beyond the array's capacity: refused before any CUDA call.
    if (M > kNoAllocMaxRows || K > kNoAllocMaxCodes || M * K > kNoAllocMaxCodes) return FP8Q_ERR_UNSUPPORTED;
    uint8_t *scratch = scratch_address();
    if (scratch == nullptr) return FP8Q_ERR_CUDA;
    // Nothing in the array needs clearing: the quantizer writes every code
    // and scale the GEMM then reads, whatever an earlier call left there.
    return fp8q_linear_channelwise(x, b, ldb, b_scale, bias, out, M, N, K, scratch,
                                   reinterpret_cast<float *>(scratch + kScaleOffset), out_dtype, nullptr, 0, stream);
}
