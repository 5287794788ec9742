"""Build libfp8q.so in-tree with nvcc for sm_103a.

Each translation unit under ``csrc/`` compiles to an object in parallel,
then the objects link into ``libfp8q.so`` next to this file.  The CUDA
runtime is linked statically, so the library needs only the driver at run
time.  No fast-math: the quantizers rely on IEEE fp32 division.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
LIB = os.path.join(HERE, "libfp8q.so")
TRACE_LIB = os.path.join(HERE, "libfp8q_trace.so")
OBJ_DIR = os.path.join(HERE, "_build")

SOURCES = ["api.cu", "host_util.cu", "quant.cu", "gemm_channelwise.cu", "gemm_blockwise.cu", "plan.cpp",
           "noalloc.cu", "selftest.cu", "w8a16_gemv.cu", "linear_gemv.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required to build libfp8q")
    return cand


def _inputs_digest(extra: str = "") -> str:
    h = hashlib.sha256()
    names = sorted(os.listdir(CSRC)) + ["fp8q.h"]
    for n in names:
        path = os.path.join(CSRC, n) if n != "fp8q.h" else os.path.join(INCLUDE, n)
        if os.path.isfile(path):
            h.update(n.encode())
            with open(path, "rb") as f:
                h.update(f.read())
    h.update(" ".join(ARCH + NVCC_FLAGS).encode())
    h.update(extra.encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, trace: bool = False) -> str:
    """Compile the library if its sources changed; returns the .so path.

    trace=True builds libfp8q_trace.so instead: the same library with the
    GEMM's per-CTA phase timestamps compiled in (include/fp8q_trace.h)."""
    lib = TRACE_LIB if trace else LIB
    defines = ["-DFP8Q_TRACE"] if trace else []
    obj_dir = OBJ_DIR + ("_trace" if trace else "")
    digest = _inputs_digest(" ".join(defines))
    stamp = lib + ".digest"
    if not force and os.path.exists(lib) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                return lib
    os.makedirs(obj_dir, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src: str) -> str:
        obj = os.path.join(obj_dir, src + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *defines, "-I", INCLUDE, "-c", os.path.join(CSRC, src), "-o", obj]
        if src.endswith(".cpp"):
            cmd = [nvcc, "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
                   "-I", INCLUDE, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(stamp, "w") as f:
        f.write(digest)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, trace="--trace" in sys.argv))
