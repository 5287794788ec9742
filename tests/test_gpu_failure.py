"""Failure detection on the GPU without a GPU fault: a pipeline wait that can
never complete gives up after its time limit, the device status word reports
FP8Q_ERR_TIMEOUT, reading it resets it, and the context keeps working."""
import ctypes
import time

import pytest
import torch

import fp8_w8a8_quantized_token_gb300 as fq
import oracle
import synthetic
from gpu_util import assert_gemm_close, out_values, quant_both_per_token, ref_values

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    d = torch.device("cuda", 0)
    torch.cuda.set_device(d)
    fq.fp8q_set_plan_override(-1)
    return d


def test_stalled_wait_reports_timeout_and_the_context_survives(dev):
    assert fq.fp8q_device_status(reset=True) == fq.FP8Q_OK
    t0 = time.monotonic()
    fq.fp8q_selftest_wait_timeout()
    L = fq.load_library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    status = L.fp8q_last_device_status(stream)        # synchronizes the stream, keeps the word
    waited = time.monotonic() - t0
    assert status == fq.FP8Q_ERR_TIMEOUT
    assert 1.5 < waited < 60, waited                   # the 2 s limit, not a hang
    assert L.fp8q_last_device_status(stream) == fq.FP8Q_ERR_TIMEOUT
    assert fq.fp8q_device_status(reset=True) == fq.FP8Q_ERR_TIMEOUT
    assert fq.fp8q_device_status(reset=True) == fq.FP8Q_OK

    # the same context still computes correctly
    x = synthetic.activations(16, 512, seed=8)
    w = synthetic.weights(256, 512, seed=8)
    xq, xs, rq, rs = quant_both_per_token(x, dev)
    wq, ws, rwq, rws = quant_both_per_token(w, dev)
    out = fq.fp8q_scaled_mm_channelwise(xq, wq, xs, ws)
    torch.cuda.synchronize()
    assert_gemm_close(out_values(out), ref_values(oracle.gemm_channelwise(rq, rwq, rs, rws)), "after timeout")
    assert fq.fp8q_device_status(reset=True) == fq.FP8Q_OK
