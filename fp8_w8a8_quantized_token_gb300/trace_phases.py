"""Per-CTA phase timeline of one GEMM launch, from the trace build.

    python -m fp8_w8a8_quantized_token_gb300.trace_phases MxNxK [MxNxK ...]

Builds ``libfp8q_trace.so`` (the library with the GEMM's per-CTA
%globaltimer stamps compiled in, ``include/fp8q_trace.h``), runs per-token
quantization + the channelwise GEMM three times as warm-up, then once more
after clearing the trace buffer, and prints for every phase the minimum,
median and maximum time (microseconds after the earliest CTA entry) over
the launch's CTAs.  Schedules that split K are traced twice: with the
split-K workspace and without it (partials exchanged in distributed shared
memory).  Inputs are the seeded synthetic tensors.  Needs a GPU.
"""
from __future__ import annotations

import ctypes
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import fp8_w8a8_quantized_token_gb300 as fq  # noqa: E402
import synthetic  # noqa: E402
from fp8_w8a8_quantized_token_gb300 import build as fbuild  # noqa: E402

# Slot order of the trace build (include/fp8q_trace.h).
PHASES = ["entry", "prologue done", "dependency wait passed", "first TMA issued", "first MMA issued",
          "last MMA committed", "epilogue saw accumulator (last tile)", "epilogue stored (last tile)",
          "split-K cluster barrier 1", "split-K reduction done", "split-K cluster barrier 2", "exit",
          "early weight loads issued", "TMEM allocated"]
SLOTS_PER_CTA = 16


def trace_launch(L, dev, M: int, N: int, K: int, workspace="auto"):
    x = synthetic.activations(M, K, outliers=True).to(dev)
    wq, ws = fq.fp8q_quant_per_token(synthetic.weights(N, K).to(dev))
    plan = fq.fp8q_gemm_plan(M, N, K)
    for _ in range(3):
        xq, xs = fq.fp8q_quant_per_token(x)
        fq.fp8q_scaled_mm_channelwise(xq, wq, xs, ws, workspace=workspace)
    torch.cuda.synchronize()
    if L.fp8q_trace_clear() != 0:
        raise RuntimeError("fp8q_trace_clear failed")
    xq, xs = fq.fp8q_quant_per_token(x)
    fq.fp8q_scaled_mm_channelwise(xq, wq, xs, ws, workspace=workspace)
    torch.cuda.synchronize()
    buf = (ctypes.c_ulonglong * (4096 * SLOTS_PER_CTA))()
    if L.fp8q_trace_read(ctypes.addressof(buf), 4096 * SLOTS_PER_CTA) != 0:
        raise RuntimeError("fp8q_trace_read failed")
    t = np.frombuffer(buf, dtype=np.uint64).reshape(4096, SLOTS_PER_CTA)[:plan["grid"]].astype(np.int64)
    return plan, t


def main(argv) -> int:
    if not argv:
        print(__doc__)
        return 2
    L = fq.load_library(fbuild.build(trace=True))
    L.fp8q_trace_read.argtypes = [ctypes.c_void_p, ctypes.c_int]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    for spec in argv:
        M, N, K = (int(v) for v in spec.split("x"))
        split = fq.fp8q_gemm_plan(M, N, K)["split_k"] > 1
        for workspace in (("auto", None) if split else ("auto",)):
            trace_one(L, dev, M, N, K, workspace)
    return 0


def trace_one(L, dev, M, N, K, workspace):
    plan, t = trace_launch(L, dev, M, N, K, workspace)
    t0 = t[:, 0].min()
    exchange = "" if plan["split_k"] == 1 else (" (split-K workspace)" if workspace else
                                                " (split-K exchange in distributed shared memory)")
    print(f"== M={M} N={N} K={K} plan={plan}{exchange}")
    for i, name in enumerate(PHASES):
        col = t[:, i]
        hit = col > 0
        if not hit.any():
            continue
        rel = (col[hit] - t0) / 1000.0
        print(f"  {name:>38}: min {rel.min():7.2f}  median {np.median(rel):7.2f}  max {rel.max():7.2f} us"
              f"  ({int(hit.sum())} CTAs)")


if __name__ == "__main__":
    sys.exit(main(sys.argv[1:]))
