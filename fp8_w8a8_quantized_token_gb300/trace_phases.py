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

    python -m fp8_w8a8_quantized_token_gb300.trace_phases --stages [--blockwise] MxNxK [MxNxK ...]

prints, for one launch (after the same warm-up), CTA 0's pipeline stages: when
each stage's loads were issued, when MMA issuer 0 saw it full and issued its
commit, and when the producer began waiting for a reused slot; then the
median interval between consecutive "full" events.

    python -m fp8_w8a8_quantized_token_gb300.trace_phases --back-to-back MxNxK

traces the steady state instead: four GEMM launches over four weight copies
(the inputs quantized beforehand) captured in one CUDA graph, replayed
three times as warm-up and once more after clearing the buffer; it prints
each launch's phase medians (microseconds after the graph's first CTA
entry) and, for launches 2-4, the gap from the previous launch's last CTA
exit to this launch's dependency release.
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


def trace_launch(L, dev, M: int, N: int, K: int, workspace="auto", blockwise: bool = False):
    x = synthetic.activations(M, K, outliers=True).to(dev)
    w = synthetic.weights(N, K).to(dev)
    wq, ws = fq.fp8q_quant_weight_block128(w) if blockwise else fq.fp8q_quant_per_token(w)
    plan = fq.fp8q_gemm_plan(M, N, K, blockwise)

    def run():
        if blockwise:
            xq, xsv = fq.fp8q_quant_per_token_group_row_padded(x, 128)
            fq.fp8q_scaled_mm_blockwise(xq, wq, xsv, ws, M=M, workspace=workspace)
        else:
            xq, xs = fq.fp8q_quant_per_token(x)
            fq.fp8q_scaled_mm_channelwise(xq, wq, xs, ws, workspace=workspace)

    for _ in range(3):
        run()
    torch.cuda.synchronize()
    if L.fp8q_trace_clear() != 0:
        raise RuntimeError("fp8q_trace_clear failed")
    run()
    torch.cuda.synchronize()
    buf = (ctypes.c_ulonglong * (4096 * SLOTS_PER_CTA))()
    if L.fp8q_trace_read(ctypes.addressof(buf), 4096 * SLOTS_PER_CTA) != 0:
        raise RuntimeError("fp8q_trace_read failed")
    t = np.frombuffer(buf, dtype=np.uint64).reshape(4096, SLOTS_PER_CTA)[:plan["grid"]].astype(np.int64)
    return plan, t


def stages(L, dev, M: int, N: int, K: int, blockwise: bool = False):
    plan, t = trace_launch(L, dev, M, N, K, blockwise=blockwise)
    n = 4 * 128 * 4
    buf = (ctypes.c_ulonglong * n)()
    if L.fp8q_trace_read_stages(ctypes.addressof(buf), n) != 0:
        raise RuntimeError("fp8q_trace_read_stages failed")
    s = np.frombuffer(buf, dtype=np.uint64).reshape(4, 128, 4)[0].astype(np.int64)
    t0 = t[0, 0]   # CTA 0 entry
    used = [k for k in range(128) if s[k, 1] > 0]
    print(f"== stages of CTA 0: M={M} N={N} K={K} {'blockwise' if blockwise else 'channelwise'} plan={plan}")
    print("  stage   wait-empty    issued    full-seen    committed   (ns after CTA 0 entry)")
    for k in used:
        cells = [s[k, 3], s[k, 0], s[k, 1], s[k, 2]]
        print(f"  {k:5d} " + "".join(f"{(c - t0) if c > 0 else -1:12d}" for c in cells))
    full = s[used, 1]
    if len(full) > 2:
        print(f"  median full-to-full interval: {np.median(np.diff(full)):.0f} ns over {len(full)} stages")


def back_to_back(L, dev, M: int, N: int, K: int):
    x = synthetic.activations(M, K, outliers=True).to(dev)
    xq, xs = fq.fp8q_quant_per_token(x)
    wq0, ws = fq.fp8q_quant_per_token(synthetic.weights(N, K).to(dev))
    copies = [wq0] + [wq0.clone() for _ in range(3)]
    outs = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(4)]
    plan = fq.fp8q_gemm_plan(M, N, K)
    # One zero-filled workspace for all launches where the schedule takes
    # one (stream-K); K-split schedules exchange in distributed shared memory.
    need = fq.fp8q_workspace_bytes(M, N, K) if plan.get("stream_k") else 0
    work = torch.zeros(need, dtype=torch.uint8, device=dev) if need else None
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        for i in range(4):
            fq.fp8q_scaled_mm_channelwise(xq, copies[i], xs, ws, out=outs[i], workspace=work)
    side.synchronize()
    if L.fp8q_trace_clear() != 0:   # capture writes launch i to block i
        raise RuntimeError("fp8q_trace_clear failed")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for i in range(4):
            fq.fp8q_scaled_mm_channelwise(xq, copies[i], xs, ws, out=outs[i], workspace=work)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    if L.fp8q_trace_clear() != 0:
        raise RuntimeError("fp8q_trace_clear failed")
    g.replay()
    torch.cuda.synchronize()
    n = 4 * 4096 * SLOTS_PER_CTA
    buf = (ctypes.c_ulonglong * n)()
    if L.fp8q_trace_read(ctypes.addressof(buf), n) != 0:
        raise RuntimeError("fp8q_trace_read failed")
    t = np.frombuffer(buf, dtype=np.uint64).reshape(4, 4096, SLOTS_PER_CTA)[:, :plan["grid"]].astype(np.int64)
    t0 = t[0, :, 0].min()
    print(f"== back to back: M={M} N={N} K={K} plan={plan}")
    cols = [("entry", 0), ("release", 2), ("first MMA", 4), ("last MMA", 5), ("stored", 7), ("exit", 11)]
    if plan.get("stream_k"):
        # (stream-K reuses the split-K slots: partial published, sources'
        # flags seen by the tile's owner, partials added)
        cols[4:4] = [("published", 8), ("flags seen", 9), ("added", 10)]
    print("  launch " + "".join(f"{c:>12}" for c, _ in cols) + "   gap(prev exit -> release)")
    for i in range(4):
        med = [np.median(t[i, :, j][t[i, :, j] > 0] - t0) / 1000.0 for _, j in cols]
        gap = ""
        if i > 0:
            prev_exit = t[i - 1, :, 11].max() - t0
            rel = t[i, :, 2][t[i, :, 2] > 0] - t0
            gap = f"   {(rel.min() - prev_exit) / 1000.0:6.2f} .. {(np.median(rel) - prev_exit) / 1000.0:6.2f} us"
        print(f"  {i + 1:6d} " + "".join(f"{v:12.2f}" for v in med) + gap)
    per_launch = (t[3, :, 11].max() - t[0, :, 11].max()) / 3000.0
    print(f"  launch period (last exit to last exit): {per_launch:.2f} us")


def main(argv) -> int:
    if not argv:
        print(__doc__)
        return 2
    if argv[0] == "--stages":
        L = fq.load_library(fbuild.build(trace=True))
        L.fp8q_trace_read.argtypes = [ctypes.c_void_p, ctypes.c_int]
        L.fp8q_trace_read_stages.argtypes = [ctypes.c_void_p, ctypes.c_int]
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        blockwise = "--blockwise" in argv
        for spec in argv[1:]:
            if spec != "--blockwise":
                stages(L, dev, *(int(v) for v in spec.split("x")), blockwise=blockwise)
        return 0
    if argv[0] == "--back-to-back":
        L = fq.load_library(fbuild.build(trace=True))
        L.fp8q_trace_read.argtypes = [ctypes.c_void_p, ctypes.c_int]
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        for spec in argv[1:]:
            back_to_back(L, dev, *(int(v) for v in spec.split("x")))
        return 0
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
