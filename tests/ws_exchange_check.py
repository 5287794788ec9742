"""Checks of the split-K workspace exchange, run by test_gpu_gemm.py in a
child process started with FP8Q_WORKSPACE_EXCHANGE=1 (the library reads the
flag once at start-up).  For every K-split schedule the GEMM tests force,
channelwise and blockwise, at M = 5 and 300: the output with the workspace
equals the output without it (distributed-shared-memory exchange) bit for
bit, a workspace one slot short is not used (identical again), schedules
with partial tiles under 128 x 128 floats ask for no workspace, and the
result is within the GEMM tolerance of the oracle."""
import os
import sys

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import fp8_w8a8_quantized_token_gb300 as fq  # noqa: E402
import oracle  # noqa: E402
import synthetic  # noqa: E402
from gpu_util import (THREADS, assert_gemm_close, out_values, quant_both_group, quant_both_per_token,  # noqa: E402
                      ref_values)
from test_gpu_gemm import SPLIT_SCHEDULES  # noqa: E402


def main():
    assert os.environ.get("FP8Q_WORKSPACE_EXCHANGE") == "1"
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    used = 0
    for swap, mma_n, split in SPLIT_SCHEDULES:
        fq.fp8q_set_plan_override(swap, mma_n, split)
        for blockwise in (False, True):
            for M in (5, 300):
                if blockwise:
                    N, K = 384, 1024
                    x = synthetic.activations(M, K, seed=M + 7, outliers=True)
                    w = synthetic.weights(N, K, seed=M + 7)
                    b = synthetic.bias(N, seed=M + 7)
                    xq, xs, rq, rs = quant_both_group(x, dev, 128)
                    wq, ws = fq.fp8q_quant_weight_block128(w.to(dev))
                    rwq, rws = oracle.quant_weight_blocks(w, 128, 128)

                    def run(workspace):
                        return fq.fp8q_scaled_mm_blockwise(xq, wq, xs.transpose(0, 1), ws, M=M, bias=b.to(dev),
                                                           workspace=workspace)
                    ref = ref_values(oracle.gemm_blockwise(rq, rwq, rs, rws, M, bias=b, threads=THREADS))
                else:
                    N, K = 392, 1040
                    x = synthetic.activations(M, K, seed=M + 7, outliers=True)
                    w = synthetic.weights(N, K, seed=M + 7)
                    b = synthetic.bias(N, seed=M + 7)
                    xq, xs, rq, rs = quant_both_per_token(x, dev)
                    wq, ws, rwq, rws = quant_both_per_token(w, dev)

                    def run(workspace):
                        return fq.fp8q_scaled_mm_channelwise(xq, wq, xs, ws, bias=b.to(dev), workspace=workspace)
                    ref = ref_values(oracle.gemm_channelwise(rq, rwq, rs, rws, bias=b, threads=THREADS))
                need = fq.fp8q_workspace_bytes(M, N, K, blockwise)
                assert (need > 0) == (swap == 0 or mma_n >= 128), (swap, mma_n, split, need)
                used += need > 0
                out_ws, out_dsmem = run("auto"), run(None)
                short = torch.empty(max(need - 128 * mma_n * 4, 0), dtype=torch.uint8, device=dev)
                out_short = run(short) if need else out_dsmem
                torch.cuda.synchronize()
                what = f"{'blockwise' if blockwise else 'channelwise'} sched {swap},{mma_n},{split} M={M}"
                assert torch.equal(out_ws, out_dsmem), what
                assert torch.equal(out_short, out_dsmem), what
                assert_gemm_close(out_values(out_ws), ref, what)
    fq.fp8q_set_plan_override(-1)
    assert used > 0
    assert fq.fp8q_device_status() == fq.FP8Q_OK
    print("workspace exchange ok", used)


if __name__ == "__main__":
    main()
