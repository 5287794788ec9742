"""The premise behind the GEMM's two MMA-issuing warps, measured: on this
GPU one issuing thread completes a chain of narrow tcgen05.mma (kind::f8f6f4,
cta_group::1, M = 128, K = 32) no faster than about one per 27 ns, the same
for N = 16 and N = 64, while wide MMAs (N >= 128) are bound by the tensor
pipe (N = 256 takes about 2.4x as long as N = 16); a second issuing warp
with its own accumulator overlaps the first for narrow N and gains nothing
where the pipe is the limit.

A small probe compiled here (operands zero in shared memory, no global
traffic) issues 256 MMAs per issuing warp into separate TMEM columns and
times them with %globaltimer; ``-s`` prints the table.  The bounds are
loose: they check the shape of the effect, not exact figures."""
import ctypes
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "fp8_w8a8_quantized_token_gb300", "csrc")

PROBE_SRC = r"""
#include <cuda_runtime.h>
#include "device_common.cuh"
using namespace fp8q;

constexpr int R = 256;

template <int N>
__global__ void __launch_bounds__(128) issue_probe(int nissue, unsigned *status, unsigned long long *ns)
{
    extern __shared__ __align__(1024) uint8_t raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t bars[4];
    __shared__ uint32_t holder;
    __shared__ int abort_flag;
    for (int i = threadIdx.x; i < 49152 / 16; i += blockDim.x) reinterpret_cast<uint4 *>(sm)[i] = make_uint4(0, 0, 0, 0);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (threadIdx.x == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(&bars[i], 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (threadIdx.x < 32) { tmem_alloc(&holder, 512); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = holder;
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0 && w < nissue) {
        const uint32_t a = smem_u32(sm), b = smem_u32(sm + 16384);
        const unsigned long long t0 = globaltimer_ns();
        for (int r = 0; r < R; ++r)
            umma_e4m3(tbase + static_cast<uint32_t>(w * N), umma_desc_sw128(a + (r & 3) * 32),
                      umma_desc_sw128(b + (r & 3) * 32), idesc_e4m3_f32<128, N>(), r > 0 ? 1u : 0u);
        umma_commit(&bars[w]);
        const bool ok = mbar_wait(&bars[w], 0, &abort_flag, status);
        ns[w] = ok ? globaltimer_ns() - t0 : 0ull;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x < 32) tmem_dealloc(tbase, 512);
}

template <int N>
static int run(int nissue, double *per_issuer_ns)
{
    unsigned *status; unsigned long long *ns;
    if (cudaMalloc(&status, 4) != cudaSuccess || cudaMalloc(&ns, 32) != cudaSuccess) return 1;
    cudaMemset(status, 0, 4);
    const int smem = 49152 + 1024;
    cudaFuncSetAttribute(issue_probe<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    double best = 1e30;
    for (int rep = 0; rep < 5; ++rep) {
        issue_probe<N><<<1, 128, smem>>>(nissue, status, ns);
        if (cudaDeviceSynchronize() != cudaSuccess) return 2;
        unsigned long long h[4] = {0, 0, 0, 0};
        cudaMemcpy(h, ns, 32, cudaMemcpyDeviceToHost);
        double worst = 0;
        for (int w = 0; w < nissue; ++w) {
            if (h[w] == 0) return 3;
            if (h[w] > worst) worst = static_cast<double>(h[w]);
        }
        if (worst < best) best = worst;
    }
    cudaFree(status); cudaFree(ns);
    *per_issuer_ns = best / R;
    return 0;
}

extern "C" int probe_mma_issue(int n, int nissue, double *per_issuer_ns)
{
    switch (n) {
        case 16: return run<16>(nissue, per_issuer_ns);
        case 64: return run<64>(nissue, per_issuer_ns);
        case 128: return run<128>(nissue, per_issuer_ns);
        case 256: return run<256>(nissue, per_issuer_ns);
        default: return 4;
    }
}
"""


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    d = tmp_path_factory.mktemp("mma_issue_probe")
    src, lib = d / "probe.cu", d / "libprobe.so"
    src.write_text(PROBE_SRC)
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-shared",
                    "-Xcompiler", "-fPIC", "-I", CSRC, "-o", str(lib), str(src)], check=True)
    L = ctypes.CDLL(str(lib))
    L.probe_mma_issue.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_double)]
    L.probe_mma_issue.restype = ctypes.c_int
    return L


def _ns(L, n, nissue):
    v = ctypes.c_double()
    assert L.probe_mma_issue(n, nissue, ctypes.byref(v)) == 0
    return v.value


def test_mma_issue_time_is_flat_in_n_and_two_issuers_overlap(probe):
    table = {}
    for n in (16, 64, 128, 256):
        for k in (1, 2):
            table[(n, k)] = _ns(probe, n, k)
    print()
    for (n, k), t in sorted(table.items()):
        print(f"M=128 N={n:3d} K=32 issuers={k}: {t:6.1f} ns per MMA per issuer, {t / k:6.1f} ns per MMA per CTA")
    # one issuer: narrow MMAs cost the same per instruction; wide ones are
    # bound by the tensor pipe
    assert table[(64, 1)] < 1.2 * table[(16, 1)]
    assert table[(256, 1)] > 1.8 * table[(16, 1)]
    # two issuers of narrow MMAs overlap: the CTA completes them faster
    assert table[(16, 2)] / 2 < 0.85 * table[(16, 1)]
    # wide MMAs already saturate the pipe: a second issuer does not help
    assert table[(256, 2)] / 2 > 0.8 * table[(256, 1)]
