"""Exhaustive pin of the E4M3 encoding: the oracle's encoder (written from the
float8_e4m3fn definition) against the GPU's cvt.rn.satfinite.e4m3x2.f32,
the conversion the library's quantizers use, over all 2^32 fp32 bit patterns.

The GPU side is a small probe compiled here with nvcc (not the library: it
checks the premise that the oracle's rounding is the hardware's).  NaN
inputs are outside the quantizers' contract; for them only a NaN code
(0x7F or 0xFF) is required."""
import ctypes
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

PROBE_SRC = r"""
#include <cuda_runtime.h>
#include <stdint.h>

__global__ void encode_range(uint32_t base, uint32_t pairs, uint8_t *out)
{
    const uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= pairs) return;
    const float lo = __uint_as_float(base + 2u * i), hi = __uint_as_float(base + 2u * i + 1u);
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    out[2u * i] = static_cast<uint8_t>(r & 0xFFu);
    out[2u * i + 1u] = static_cast<uint8_t>(r >> 8);
}

extern "C" int probe_encode_range(uint32_t base, uint32_t count, void *out, void *stream)
{
    const uint32_t pairs = count / 2u;
    encode_range<<<(pairs + 255u) / 256u, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        base, pairs, static_cast<uint8_t *>(out));
    return static_cast<int>(cudaGetLastError());
}
"""

CHUNK = 1 << 26


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    d = tmp_path_factory.mktemp("codec_probe")
    src, lib = d / "probe.cu", d / "libprobe.so"
    src.write_text(PROBE_SRC)
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-shared", "-Xcompiler", "-fPIC",
                    "-o", str(lib), str(src)], check=True)
    L = ctypes.CDLL(str(lib))
    L.probe_encode_range.argtypes = [ctypes.c_uint32, ctypes.c_uint32, ctypes.c_void_p, ctypes.c_void_p]
    L.probe_encode_range.restype = ctypes.c_int
    oracle.build()
    return L


def _bits(base: int) -> np.ndarray:
    return np.arange(CHUNK, dtype=np.uint32) + np.uint32(base)   # no overflow: base + CHUNK <= 2^32


def _oracle_chunk(base: int) -> np.ndarray:
    return oracle.e4m3_encode(_bits(base).view(np.float32))


def test_oracle_encoder_equals_hardware_on_every_fp32(probe):
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    out = torch.empty(CHUNK, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    nchunks = (1 << 32) // CHUNK
    checked = 0
    workers = max(1, min(8, os.cpu_count() or 1))
    with ThreadPoolExecutor(workers) as pool:
        futures = {c: pool.submit(_oracle_chunk, c * CHUNK) for c in range(min(nchunks, 2 * workers))}
        for c in range(nchunks):
            base = c * CHUNK
            assert probe.probe_encode_range(base, CHUNK, ctypes.c_void_p(out.data_ptr()),
                                            ctypes.c_void_p(stream.cuda_stream)) == 0
            got = out.cpu().numpy()
            ref = futures.pop(c).result()
            if c + 2 * workers < nchunks:
                futures[c + 2 * workers] = pool.submit(_oracle_chunk, (c + 2 * workers) * CHUNK)
            bits = _bits(base)
            nan = (bits & 0x7F800000) == 0x7F800000
            nan &= (bits & 0x007FFFFF) != 0
            bad = np.nonzero((got != ref) & ~nan)[0]
            assert bad.size == 0, [(hex(int(bits[i])), int(got[i]), int(ref[i])) for i in bad[:8]]
            assert np.all((got[nan] & 0x7F) == 0x7F)
            checked += int((~nan).sum())
    assert checked == (1 << 32) - 2 * ((1 << 23) - 1)
