"""Small, fixed GPU cases for Nsight Compute captures.

    python -m fp8_w8a8_quantized_token_gb300.profile_cases <case> [<case> ...]

Each case prepares its inputs (weights quantized once), then launches its
target kernel WARMUP + 1 times on one stream; capture the last launch with
``ncu -k regex:<kernel> -s <WARMUP> -c 1`` (one case per command line) or
several cases in a row with ``-c <count>``.  Inputs are the seeded synthetic
tensors of the benchmark workloads.
"""
from __future__ import annotations

import sys

import torch

import fp8_w8a8_quantized_token_gb300 as fq
import synthetic

WARMUP = 2

# name: (kind, M, N, K)
CASES = {
    "prefill_oproj": ("channelwise", 8192, 4096, 4096),
    "prefill_gateup": ("channelwise", 8192, 24576, 4096),
    "mid_oproj": ("channelwise", 1024, 4096, 4096),
    "mid_oproj_512": ("channelwise", 512, 4096, 4096),
    "decode_oproj": ("channelwise", 16, 4096, 4096),
    "decode_down": ("channelwise", 1, 4096, 12288),
    "blockwise_prefill": ("blockwise", 8192, 24576, 3072),
    "blockwise_decode": ("blockwise", 16, 4096, 7168),
    "quant_token": ("quant_token", 8192, 0, 4096),
    "quant_group": ("quant_group", 8192, 0, 12288),
    "quant_silu_group": ("quant_silu_group", 4096, 0, 12288),   # input [4096, 2 x 12288]
    "quant_static": ("quant_static", 16384, 0, 4096),
    "w8a16_gateup": ("w8a16", 1, 24576, 4096),
}


def run(case: str, dev) -> None:
    kind, M, N, K = CASES[case]
    x = synthetic.activations(M, K, outliers=True).to(dev)
    if kind == "quant_token":
        for _ in range(WARMUP + 1):
            fq.fp8q_quant_per_token(x)
        return
    if kind == "quant_group":
        for _ in range(WARMUP + 1):
            fq.fp8q_quant_per_token_group_row_padded(x, 128)
        return
    if kind == "quant_silu_group":
        xm = synthetic.activations(M, 2 * K, outliers=True).to(dev)
        for _ in range(WARMUP + 1):
            fq.fp8q_quant_per_token_group_row_padded(xm, 128, scale_ue8m0=True, fuse_silu_and_mul=True)
        return
    if kind == "quant_static":
        s = torch.tensor([0.02], dtype=torch.float32, device=dev)
        for _ in range(WARMUP + 1):
            fq.fp8q_quant_static_per_tensor(x, s)
        return
    w = synthetic.weights(N, K).to(dev)
    if kind == "w8a16":
        wq, ws = fq.fp8q_quant_per_token(w)
        torch.cuda.synchronize()
        for _ in range(WARMUP + 1):
            fq.fp8q_scaled_mm_w8a16(x, wq, ws)
    elif kind == "channelwise":
        wq, ws = fq.fp8q_quant_per_token(w)
        xq, xs = fq.fp8q_quant_per_token(x)
        torch.cuda.synchronize()
        for _ in range(WARMUP + 1):
            fq.fp8q_scaled_mm_channelwise(xq, wq, xs, ws)
    else:
        wq, ws = fq.fp8q_quant_weight_block128(w)
        xq, xsv = fq.fp8q_quant_per_token_group_row_padded(x, 128)
        torch.cuda.synchronize()
        for _ in range(WARMUP + 1):
            fq.fp8q_scaled_mm_blockwise(xq, wq, xsv, ws, M=M)


def main(argv) -> int:
    if not argv or any(c not in CASES for c in argv):
        print("cases:", ", ".join(CASES))
        return 2
    fq.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    for c in argv:
        run(c, dev)
    torch.cuda.synchronize()
    print("ok", " ".join(argv))
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1:]))
