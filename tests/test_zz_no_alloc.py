"""fp8q_linear_channelwise_noalloc: the channelwise linear layer for callers
that cannot allocate device memory (their memory belongs to another
allocator, or cudaMalloc's synchronisation is not acceptable to them).  Its
quantized activations live in one fixed array inside the library instead of
caller buffers.

The GPU test calls it through the C ABI twice in a row, on different shapes
(the second smaller, so the array still holds the first call's larger
contents; the second on a stream other than the current one), and compares
each result with fp8q_linear_channelwise run on caller-allocated buffers
without a workspace.  Both run the same kernels on the same schedule with
the same split-K exchange, so the outputs must be identical bit for bit;
the oracle's GEMM tolerance is checked as well.  This file is named to be
collected last."""
import ctypes

import pytest
import torch

import fp8_w8a8_quantized_token_gb300 as fq
import synthetic
from gpu_util import assert_gemm_close, out_values


def test_sizes_beyond_the_scratch_array_are_refused_before_any_cuda_call():
    from fp8_w8a8_quantized_token_gb300 import build as fbuild
    fbuild.build()
    lib = fq.load_library()
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: the size check comes first
    too_many_codes = fq.NOALLOC_MAX_CODES // 4096 + 1
    assert lib.fp8q_linear_channelwise_noalloc(fake, fake, 4096, fake, None, fake, too_many_codes, 256, 4096,
                                               fq.FP8Q_OUT_BF16, None) == fq.FP8Q_ERR_UNSUPPORTED
    assert lib.fp8q_linear_channelwise_noalloc(fake, fake, 16, fake, None, fake, fq.NOALLOC_MAX_ROWS + 1, 256, 16,
                                               fq.FP8Q_OUT_BF16, None) == fq.FP8Q_ERR_UNSUPPORTED
    assert lib.fp8q_linear_channelwise_noalloc(None, None, 64, None, None, None, 0, 64, 64, fq.FP8Q_OUT_BF16,
                                               None) == fq.FP8Q_OK


def _layer(dev, M, N, K, seed, bias):
    x = synthetic.activations(M, K, seed=seed, outliers=True).to(dev)
    wq, ws = fq.fp8q_quant_per_token(synthetic.weights(N, K, seed=seed).to(dev))
    b = synthetic.bias(N, seed=seed).to(dev) if bias else None
    return x, wq, ws, b


@pytest.mark.gpu
def test_noalloc_linear_matches_the_allocating_entry_point_on_two_calls():
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fq.fp8q_set_plan_override(-1)
    lib = fq.load_library()
    side = torch.cuda.Stream(dev)
    for call, (M, N, K, bias) in enumerate([(300, 512, 4096, True), (7, 384, 1024, False)]):
        x, wq, ws, b = _layer(dev, M, N, K, seed=60 + call, bias=bias)
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
        # the second call on a stream that is not the current one
        s = torch.cuda.current_stream(dev) if call == 0 else side
        s.wait_stream(torch.cuda.current_stream(dev))
        st = lib.fp8q_linear_channelwise_noalloc(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(wq.data_ptr()),
                                                 K, ctypes.c_void_p(ws.data_ptr()),
                                                 None if b is None else ctypes.c_void_p(b.data_ptr()),
                                                 ctypes.c_void_p(out.data_ptr()), M, N, K, fq.FP8Q_OUT_BF16,
                                                 ctypes.c_void_p(s.cuda_stream))
        assert st == fq.FP8Q_OK, fq.status_str(st)
        s.synchronize()
        ref = fq.fp8q_linear_channelwise(x, wq, ws, bias=b, workspace=None)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"no-alloc call {call + 1} ({M}x{N}x{K}) differs from the allocating call"
        assert_gemm_close(out_values(out), oracle_linear(x, wq, ws, b), f"no-alloc call {call + 1} ({M}x{N}x{K})")
    assert fq.fp8q_device_status() == fq.FP8Q_OK


def oracle_linear(x, wq, ws, b):
    import oracle
    from gpu_util import THREADS, ref_values, u8
    rq, rs = oracle.quant_per_token(x.cpu(), threads=THREADS)
    return ref_values(oracle.gemm_channelwise(rq, u8(wq), rs, ws.cpu().numpy(), bias=None if b is None else b.cpu(),
                                              threads=THREADS))
