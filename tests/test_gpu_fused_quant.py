"""Quantization fused into the blockwise GEMM (decode, 16- and 32-token tiles):
fp8q_linear_blockwise_fused quantizes the bf16 activation tiles inside the
GEMM.  Its codes and scales are the standalone quantizer's, so its output
must be bit-identical to the two-kernel path (group quantizer + blockwise
GEMM on the same schedule), and within the GEMM tolerance of the oracle."""
import ctypes

import numpy as np
import pytest
import torch

import fp8_w8a8_quantized_token_gb300 as fq
import oracle
import synthetic
from gpu_util import assert_gemm_close, out_values, ref_values

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    d = torch.device("cuda", 0)
    torch.cuda.set_device(d)
    fq.fp8q_set_plan_override(-1)
    return d


def _fused(x, wq, ws, bias, fp16, ldx=None):
    L = fq.load_library()
    P = ctypes.c_void_p
    M, K = x.shape
    N = wq.shape[0]
    out = torch.empty((M, N), dtype=torch.float16 if fp16 else torch.bfloat16, device=x.device)
    st = L.fp8q_linear_blockwise_fused(P(x.data_ptr()), x.stride(0) if ldx is None else ldx, P(wq.data_ptr()),
                                       P(ws.data_ptr()), None if bias is None else P(bias.data_ptr()),
                                       P(out.data_ptr()), M, N, K, 1 if fp16 else 0,
                                       P(torch.cuda.current_stream().cuda_stream))
    assert st == fq.FP8Q_OK, fq.status_str(st)
    return out


def _two_kernel(x, wq, ws, bias, fp16):
    # No workspace, as the fused kernel takes none: where the plan is
    # stream-K both then run the same K-split schedule of the same tiles.
    xq, xsv = fq.fp8q_quant_per_token_group_row_padded(x, 128)
    return fq.fp8q_scaled_mm_blockwise(xq, wq, xsv, ws, bias=bias, M=x.shape[0],
                                       out_dtype=torch.float16 if fp16 else torch.bfloat16, workspace=None)


@pytest.mark.parametrize("M,N,K,bias,fp16", [
    (1, 4096, 7168, False, False),       # the blockwise decode layer
    (16, 4096, 7168, True, False),
    (7, 4096, 7168, False, True),
    (3, 3072, 12288, True, False),       # long K: K split, 12 blocks per CTA
    (13, 24576, 3072, False, False),     # wide N
    (5, 256, 512, True, True),           # tiny: one K block per CTA
    (16, 512, 128, False, False),        # K = one block
    # 32-token tiles (four rows per quantizing thread)
    (32, 4096, 7168, False, False),
    (31, 4096, 7168, True, True),        # ragged token tile
    (19, 256, 512, True, False),         # 13 zero-filled token rows
    (32, 512, 128, False, True),
    (29, 512, 1024, True, False),
    (25, 1024, 1024, False, False),
    (24, 4096, 7168, True, False),       # the M = 32 row's tile (the M = 16 row's cannot hold 24 tokens)
])
def test_fused_equals_two_kernel_path_and_oracle(dev, M, N, K, bias, fp16):
    plan = fq.fp8q_gemm_plan(M, N, K, True)
    assert plan["swap_ab"] == 1 and plan["mma_n"] in (16, 32), plan
    x = synthetic.activations(M, K, outliers=True, seed=M * 3 + K).to(dev)
    w = synthetic.weights(N, K, seed=N + K).to(dev)
    wq, ws = fq.fp8q_quant_weight_block128(w)
    b = synthetic.bias(N, seed=N).to(dev) if bias else None
    out = _fused(x, wq, ws, b, fp16)
    ref2 = _two_kernel(x, wq, ws, b, fp16)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref2.view(torch.int16))
    # against the oracle (group quantizer + exact blockwise GEMM)
    rq, rs = oracle.quant_group_row_padded(x.cpu(), 128, threads=8)
    rwq, rws = oracle.quant_weight_blocks(w.cpu(), 128, 128)
    ref = oracle.gemm_blockwise(rq, rwq, rs, rws, M, bias=None if b is None else b.cpu(), out_fp16=fp16,
                                threads=8)
    assert_gemm_close(out_values(out), ref_values(ref, out_fp16=fp16), "fused blockwise linear")


def test_fused_special_rows(dev):
    """Zero rows (eps floor), huge and tiny rows, a ragged last token tile."""
    M, N, K = 11, 512, 1024
    x = synthetic.activations(M, K, outliers=True, seed=77).float()
    x[2] = 0.0
    x[4] *= 1e-30
    x[6, :128] = 0.0
    x[9] *= 1e4
    x = x.to(torch.bfloat16).to(dev)
    w = synthetic.weights(N, K, seed=78).to(dev)
    wq, ws = fq.fp8q_quant_weight_block128(w)
    out = fq.fp8q_linear_blockwise_fused(x, wq, ws)
    ref2 = _two_kernel(x, wq, ws, None, False)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref2.view(torch.int16))


def test_fused_strided_input_and_unsupported_schedule(dev):
    M, N, K, ldx = 6, 512, 1024, 1536
    big = synthetic.activations(M, ldx, outliers=True, seed=81).to(dev)
    x = big[:, :K]
    w = synthetic.weights(N, K, seed=82).to(dev)
    wq, ws = fq.fp8q_quant_weight_block128(w)
    out = _fused(x, wq, ws, None, False, ldx=ldx)
    ref2 = _two_kernel(x.contiguous(), wq, ws, None, False)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref2.view(torch.int16))
    # a prefill size has no 16- or 32-token schedule: refused, nothing enqueued
    xp = synthetic.activations(512, K, seed=83).to(dev)
    with pytest.raises(RuntimeError, match="UNSUPPORTED"):
        fq.fp8q_linear_blockwise_fused(xp, wq, ws)


def test_fused_back_to_back_layers_reuse_activations(dev):
    """Ten fused launches on one stream, each layer's output the next
    layer's input (the dependency wait must order the activation loads)."""
    M, D = 4, 1024
    x = synthetic.activations(M, D, seed=79).to(dev)
    ws_ = []
    for i in range(10):
        w = synthetic.weights(D, D, seed=80 + i).to(dev)
        ws_.append(fq.fp8q_quant_weight_block128(w))
    h = x
    outs = []
    for wq, ws in ws_:
        h = fq.fp8q_linear_blockwise_fused(h, wq, ws)
        outs.append(h)
    h2 = x
    for (wq, ws), o in zip(ws_, outs):
        h2 = _two_kernel(h2, wq, ws, None, False)
        torch.cuda.synchronize()
        assert torch.equal(o.view(torch.int16), h2.view(torch.int16))
