// host_util.cu -- host utilities: tensor-map encoding through the driver
// entry point, the per-device status word and the SM count.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "internal.h"

namespace fp8q {

// Device status word: one per device that loads the library, written only
// by kernels that give up on a bounded wait.
__device__ unsigned g_status_word;

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

constexpr int kMaxDev = 64;
std::atomic<unsigned *> g_status_ptr[kMaxDev];
std::atomic<int> g_sms[kMaxDev];

}  // namespace

bool make_tmap_2d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, uint64_t cols, uint64_t rows,
                  uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows, bool swizzle128)
{
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

unsigned *device_status_ptr()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
    unsigned *p = g_status_ptr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess) return nullptr;
        p = static_cast<unsigned *>(addr);
        g_status_ptr[dev].store(p, std::memory_order_release);
    }
    return p;
}

int current_device_sms()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
    int n = g_sms[dev].load(std::memory_order_acquire);
    if (n <= 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        g_sms[dev].store(n, std::memory_order_release);
    }
    return n;
}

cudaError_t read_status_word(unsigned *value, bool reset, cudaStream_t st)
{
    unsigned *p = device_status_ptr();
    if (p == nullptr) return cudaErrorInvalidDevice;
    cudaError_t e = cudaMemcpyAsync(value, p, sizeof(unsigned), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e == cudaSuccess && reset) {
        e = cudaMemsetAsync(p, 0, sizeof(unsigned), st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    }
    return e;
}

}  // namespace fp8q
