// host_util.cu -- host utilities: tensor-map encoding through the driver
// entry point, the per-device status word and the SM count.
#include <cuda.h>
#include <cuda_runtime.h>

#include <stdlib.h>

#include <atomic>
#include <mutex>

#include "internal.h"

namespace fp8q {

// Device status word: one per device that loads the library, written only
// by kernels that give up on a bounded wait.
__device__ unsigned g_status_word;

#ifdef FP8Q_TRACE
// Trace builds: 16 timestamps for each of the first 4096 CTAs of each of
// the 4 most recent GEMM launches (launch i uses block i % 4), and 4 per
// ring stage (the first 128) of each launch's CTA 0.
__device__ unsigned long long g_trace_buf[4 * 4096 * 16];
__device__ unsigned long long g_trace_stages[4 * kTraceStages * 4];
std::atomic<unsigned> g_trace_launch{0};
#endif

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
                  uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swizzle)
{
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_tmap_3d_kblocks(CUtensorMap *map, const void *base, uint64_t K, uint64_t rows, uint64_t row_bytes,
                          uint32_t box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr || K % 128 != 0) return false;
    const cuuint64_t dims[3] = {128, rows, K / 128};
    const cuuint64_t strides[2] = {row_bytes, 128};
    const cuuint32_t box[3] = {128, box_rows, 2};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
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

unsigned long long *trace_buffer(unsigned long long **stages)
{
    *stages = nullptr;
#ifdef FP8Q_TRACE
    void *addr = nullptr, *saddr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_trace_buf) != cudaSuccess) return nullptr;
    if (cudaGetSymbolAddress(&saddr, g_trace_stages) != cudaSuccess) return nullptr;
    const unsigned i = g_trace_launch.fetch_add(1) % 4u;
    *stages = static_cast<unsigned long long *>(saddr) + static_cast<size_t>(i) * kTraceStages * 4;
    return static_cast<unsigned long long *>(addr) + static_cast<size_t>(i) * 4096 * 16;
#else
    return nullptr;
#endif
}

int prefetch_kblocks(bool swapped, bool blockwise, int grid)
{
    static const int v = [] {
        const char *s = getenv("FP8Q_PREFETCH_KB");
        return s != nullptr ? atoi(s) : -1;
    }();
    if (v >= 0) return v;
    if (!swapped) return 0;
    if (!blockwise) return 16;
    return 2 * static_cast<long long>(grid) <= 3 * static_cast<long long>(current_device_sms()) ? 16 : 0;
}

bool workspace_exchange_enabled()
{
    static const bool v = [] {
        const char *s = getenv("FP8Q_WORKSPACE_EXCHANGE");
        return s != nullptr && s[0] == '1';
    }();
    return v;
}

namespace {
// The device ranges the launches on a stream that may still be running when
// the next library kernel starts may write: the last launch's, plus, when
// that launch lets its successor start before its own dependency wait, the
// ranges recorded before it (up to kMaxRanges; more are recorded as
// "unknown", which every overlap test answers with yes).
constexpr int kMaxRanges = 6;
struct LaunchRecord {
    cudaStream_t stream;
    bool used, unknown;
    int n;
    uintptr_t lo[kMaxRanges], hi[kMaxRanges];
};
std::mutex g_launch_mu;
LaunchRecord g_launches[64];
int g_launch_next = 0;
}  // namespace

void note_launch_writes(cudaStream_t st, const void *base, size_t bytes, const void *base2, size_t bytes2,
                        const void *base3, size_t bytes3, bool keep_previous)
{
    std::lock_guard<std::mutex> g(g_launch_mu);
    LaunchRecord rec = {};
    rec.stream = st;
    rec.used = true;
    const void *bases[3] = {base, base2, base3};
    const size_t sizes[3] = {bytes, bytes2, bytes3};
    for (int i = 0; i < 3; ++i)
        if (bases[i] != nullptr && sizes[i] != 0) {
            rec.lo[rec.n] = reinterpret_cast<uintptr_t>(bases[i]);
            rec.hi[rec.n] = rec.lo[rec.n] + sizes[i];
            ++rec.n;
        }
    LaunchRecord *slot = nullptr;
    for (auto &r : g_launches)
        if (r.used && r.stream == st) {
            slot = &r;
            break;
        }
    if (keep_previous) {
        if (slot == nullptr) {
            rec.unknown = true;   // nothing known about what may still run
        } else {
            rec.unknown = slot->unknown;
            for (int i = 0; i < slot->n && !rec.unknown; ++i) {
                if (rec.n == kMaxRanges) {
                    rec.unknown = true;
                    break;
                }
                rec.lo[rec.n] = slot->lo[i];
                rec.hi[rec.n] = slot->hi[i];
                ++rec.n;
            }
        }
    }
    if (slot != nullptr) {
        *slot = rec;
        return;
    }
    g_launches[g_launch_next] = rec;
    g_launch_next = (g_launch_next + 1) % 64;
}

bool last_launch_writes_overlap(cudaStream_t st, const void *base, size_t bytes)
{
    std::lock_guard<std::mutex> g(g_launch_mu);
    const uintptr_t lo = reinterpret_cast<uintptr_t>(base), hi = lo + bytes;
    for (const auto &r : g_launches)
        if (r.used && r.stream == st) {
            if (r.unknown) return true;
            for (int i = 0; i < r.n; ++i)
                if (r.lo[i] < hi && lo < r.hi[i]) return true;
            return false;
        }
    // No record for this stream (evicted or never seen): assume the worst.
    return true;
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

#ifdef FP8Q_TRACE
// Diagnostics ABI of trace builds (include/fp8q_trace.h).
extern "C" __attribute__((visibility("default"))) int fp8q_trace_read(unsigned long long *host, int count)
{
    if (count > 4 * 4096 * 16) count = 4 * 4096 * 16;
    return cudaMemcpyFromSymbol(host, fp8q::g_trace_buf, sizeof(unsigned long long) * count) == cudaSuccess ? 0 : 3;
}
extern "C" __attribute__((visibility("default"))) int fp8q_trace_read_stages(unsigned long long *host, int count)
{
    if (count > 4 * fp8q::kTraceStages * 4) count = 4 * fp8q::kTraceStages * 4;
    return cudaMemcpyFromSymbol(host, fp8q::g_trace_stages, sizeof(unsigned long long) * count) == cudaSuccess ? 0
                                                                                                             : 3;
}
extern "C" __attribute__((visibility("default"))) int fp8q_trace_clear(void)
{
    void *addr = nullptr, *saddr = nullptr;
    if (cudaGetSymbolAddress(&addr, fp8q::g_trace_buf) != cudaSuccess) return 3;
    if (cudaGetSymbolAddress(&saddr, fp8q::g_trace_stages) != cudaSuccess) return 3;
    fp8q::g_trace_launch.store(0);
    if (cudaMemset(saddr, 0, sizeof(unsigned long long) * 4 * fp8q::kTraceStages * 4) != cudaSuccess) return 3;
    return cudaMemset(addr, 0, sizeof(unsigned long long) * 4 * 4096 * 16) == cudaSuccess ? 0 : 3;
}
#endif
