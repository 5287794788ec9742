"""Schedule sweep for the GEMM planner: writes ``csrc/tile_table.inc``.

For every linear shape of the benchmark workloads and a grid of M values,
each candidate schedule (operand orientation, MMA N extent, K-split or,
for swapped tiles, stream-K) is
timed on the GPU with the split-K workspace it uses -- 8 back-to-back
launches over rotating weight copies
(more than twice L2 in total) captured in a CUDA graph, replayed 10 times,
CUDA events on the launching stream -- and the fastest one becomes the
table row for that (N, K, scheme, M).  Run on a GB300:

    python fp8_w8a8_quantized_token_gb300/tune.py [--out path] [--shapes a,b]

then rebuild the library.  The planner looks rows up by (N, K, scheme) and
the nearest M (ties to the smaller M).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
sys.path.insert(0, ROOT)

SHAPES = {
    # label: (N, K, blockwise, M grid)
    "o_proj": (4096, 4096, 0, [1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024, 2048, 4096, 8192]),
    "qkv": (6144, 4096, 0, [1, 16, 32, 64, 128, 256, 512, 2048, 8192]),
    "down": (4096, 12288, 0, [1, 16, 32, 64, 128, 256, 512, 2048, 8192]),
    "gate_up": (24576, 4096, 0, [1, 16, 32, 64, 128, 256, 512, 2048, 8192]),
    "blk_4096x7168": (4096, 7168, 1, [1, 4, 16, 32, 64, 128, 256, 512, 2048, 8192]),
    "blk_24576x3072": (24576, 3072, 1, [1, 16, 64, 256, 1024, 8192]),
    "blk_3072x12288": (3072, 12288, 1, [1, 16, 64, 256, 1024, 8192]),
}
SPLITS = (1, 2, 4, 8)
SWAP_SPLITS = (0,) + SPLITS   # 0: stream-K (16- and 32-token tiles)


def candidates(M: int):
    c = []
    for mn in (16, 32, 64, 128):
        if mn < M / 8 or (mn > 16 and mn >= 2 * M):
            continue
        if M > 1024:
            continue
        c += [(1, mn, s) for s in (SWAP_SPLITS if mn <= 32 else SPLITS)]
    # Weights on the MMA's N side: half the MMA instructions of 128-row
    # weight tiles (a tcgen05.mma costs the same whatever its N).
    c += [(0, 256, s) for s in ((1, 2, 4) if M > 1024 else SPLITS)]
    # Narrow weight tiles (mid-size M: enough tiles for every SM without a
    # K split).
    if 64 <= M <= 2048:
        c += [(0, n, s) for n in (32, 64, 128) for s in (1, 2)]
    return c


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=os.path.join(HERE, "csrc", "tile_table.inc"))
    ap.add_argument("--shapes", default=",".join(SHAPES))
    args = ap.parse_args()

    import torch

    import fp8_w8a8_quantized_token_gb300 as fq
    from fp8_w8a8_quantized_token_gb300 import build as fbuild
    import synthetic

    fbuild.build()
    L = fq.load_library()
    P = ctypes.c_void_p
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    rows = []
    for label in args.shapes.split(","):
        N, K, bw, ms = SHAPES[label]
        w = synthetic.weights(N, K).to(dev)
        wq, ws = fq.fp8q_quant_weight_block128(w) if bw else fq.fp8q_quant_per_token(w)
        ncopy = max(2, min(12, (300 << 20) // (N * K)))
        copies = [wq] + [wq.clone() for _ in range(ncopy - 1)]
        del w
        for M in ms:
            x = synthetic.activations(M, K).to(dev)
            if bw:
                xq, xsv = fq.fp8q_quant_per_token_group_row_padded(x, 128)
                xs, m_pad = xsv.transpose(0, 1), xq.shape[0]
            else:
                (xq, xs), m_pad = fq.fp8q_quant_per_token(x), M
            out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)

            work = None

            def gemm(wqi, sp):
                wp, wn = (None, 0) if work is None else (P(work.data_ptr()), work.numel())
                if bw:
                    st = L.fp8q_scaled_mm_blockwise(P(xq.data_ptr()), P(wqi.data_ptr()), P(xs.data_ptr()),
                                                    P(ws.data_ptr()), None, P(out.data_ptr()), M, m_pad, N, K, 0,
                                                    wp, wn, sp)
                else:
                    st = L.fp8q_scaled_mm_channelwise(P(xq.data_ptr()), P(wqi.data_ptr()), K, P(xs.data_ptr()),
                                                      P(ws.data_ptr()), None, P(out.data_ptr()), M, N, K, 0, wp,
                                                      wn, sp)
                if st != 0:
                    raise RuntimeError(fq.status_str(st))

            timed = []
            for cand in candidates(M):
                fq.fp8q_set_plan_override(*cand)
                # Each candidate with the split-K workspace it uses (as the
                # library's callers pass it).
                need = fq.fp8q_workspace_bytes(M, N, K, bool(bw))
                work = torch.zeros(need, dtype=torch.uint8, device=dev) if need else None
                side = torch.cuda.Stream()
                with torch.cuda.stream(side):
                    for i in range(2):
                        gemm(copies[i % ncopy], P(side.cuda_stream))
                side.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=side):
                    for i in range(8):
                        gemm(copies[i % ncopy], P(side.cuda_stream))
                g.replay()
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                for _ in range(10):
                    g.replay()
                e1.record()
                torch.cuda.synchronize()
                timed.append((e0.elapsed_time(e1) * 1e3 / 80, cand))
            fq.fp8q_set_plan_override(-1)
            timed.sort()
            best_us, best = timed[0]
            rows.append((N, K, bw, M, *best))
            print(json.dumps({"shape": label, "M": M, "best_us": round(best_us, 2), "best": best,
                              "all": [(round(u, 2), c) for u, c in timed[1:]]}), flush=True)
    with open(args.out, "w") as f:
        f.write("// Generated by fp8_w8a8_quantized_token_gb300/tune.py on a GB300: the fastest measured\n")
        f.write("// schedule per shape and M.  Row: {N, K, blockwise, M, swap_ab, mma_n, split_k},\n")
        for r in rows:
            f.write("    {%d, %d, %d, %d, %d, %d, %d},\n" % r)
    print(f"wrote {len(rows)} rows to {args.out}")


if __name__ == "__main__":
    main()
