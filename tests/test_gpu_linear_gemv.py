"""GPU parity of the linear layers at decode sizes.  One token with K <=
12288 (channelwise: on layers of at most 4096 x 4096 weights) runs as ONE
launch with the per-token (channelwise) or group-128 (blockwise)
quantization fused into a matrix-vector product on the CUDA cores; two to
four tokens, longer rows and larger channelwise layers take the quantizer
and the tensor-core GEMM.  Either way the codes and scales
left in the caller's buffers are bit-exact against the oracle's per-token
quantizer, the output is within the GEMM bar of the oracle's GEMM on those
codes, and the fused launch leaves the same codes and scales as the
two-kernel composition (forced by a schedule override)."""
import ctypes

import numpy as np
import pytest
import torch

import fp8_w8a8_quantized_token_gb300 as fq
import oracle
import synthetic
from gpu_util import THREADS, assert_gemm_close, f32, out_values, ref_values, u8

pytestmark = pytest.mark.gpu

P = ctypes.c_void_p


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    d = torch.device("cuda", 0)
    torch.cuda.set_device(d)
    fq.fp8q_set_plan_override(-1)
    return d


@pytest.fixture
def schedule():
    yield
    fq.fp8q_set_plan_override(-1)


def linear(dev, x, wq, ws, bias=None, out_dtype=torch.bfloat16):
    """fp8q_linear_channelwise through the C ABI with caller-owned scratch
    (filled with canaries first); returns out, xq, xs."""
    L = fq.load_library()
    M, K = x.shape
    N = wq.shape[0]
    xd = x.to(dev)
    xq = torch.full((M, K), 0x5A, dtype=torch.uint8, device=dev)
    xs = torch.full((M,), -3.0, dtype=torch.float32, device=dev)
    out = torch.empty((M, N), dtype=out_dtype, device=dev)
    bd = None if bias is None else bias.to(dev)
    st = P(torch.cuda.current_stream(dev).cuda_stream)
    rc = L.fp8q_linear_channelwise(P(xd.data_ptr()), P(wq.data_ptr()), wq.stride(0), P(ws.data_ptr()),
                                   None if bd is None else P(bd.data_ptr()), P(out.data_ptr()), M, N, K,
                                   P(xq.data_ptr()), P(xs.data_ptr()),
                                   fq.FP8Q_OUT_FP16 if out_dtype == torch.float16 else fq.FP8Q_OUT_BF16,
                                   None, 0, st)
    assert rc == fq.FP8Q_OK
    torch.cuda.synchronize()
    return out, xq, xs


def weights(dev, N, K, seed):
    w = synthetic.weights(N, K, seed=seed)
    wq, ws = fq.fp8q_quant_per_token(w.to(dev))
    torch.cuda.synchronize()
    return wq, ws


def check(dev, x, wq, ws, bias=None, out_dtype=torch.bfloat16, what=""):
    out, xq, xs = linear(dev, x, wq, ws, bias, out_dtype)
    rq, rs = oracle.quant_per_token(x, threads=THREADS)
    assert np.array_equal(u8(xq), rq), f"{what}: codes differ from the oracle's"
    assert np.array_equal(f32(xs), rs), f"{what}: scales differ from the oracle's"
    fp16 = out_dtype == torch.float16
    ref = ref_values(oracle.gemm_channelwise(rq, u8(wq), rs, f32(ws), bias=bias, out_fp16=fp16, threads=THREADS),
                     fp16)
    assert_gemm_close(out_values(out), ref, what)
    return out, xq, xs


@pytest.mark.parametrize("M", [1, 2, 3, 4])
@pytest.mark.parametrize("N,K", [(392, 1040), (8, 16), (4096, 4096), (264, 12288), (136, 4112)])
def test_few_token_linear_parity(dev, M, N, K):
    """K not a multiple of the 512-byte chunk, a single 16-element piece, N
    not a multiple of the CTA's rows, one to three chunks per warp; M > 1 on
    the two-kernel path."""
    wq, ws = weights(dev, N, K, seed=N + K)
    x = synthetic.activations(M, K, outliers=True, seed=M + K)
    check(dev, x, wq, ws, what=f"{M}x{N}x{K}")


@pytest.mark.parametrize("M", [1, 3])
def test_few_token_linear_bias_and_fp16(dev, M):
    wq, ws = weights(dev, 1024, 2048, seed=7)
    x = synthetic.activations(M, 2048, outliers=True, seed=8)
    b = synthetic.bias(1024, seed=9)
    check(dev, x, wq, ws, bias=b, what="bias bf16")
    check(dev, x, wq, ws, bias=b, out_dtype=torch.float16, what="bias fp16")


def test_few_token_linear_special_rows(dev):
    """A zero row (the scale is eps / 448), a row of one huge outlier among
    tiny values, and a row with values on E4M3 rounding midpoints."""
    K, N = 1024, 256
    wq, ws = weights(dev, N, K, seed=11)
    x = torch.zeros((4, K), dtype=torch.float32)
    x[1] = 1e-3
    x[1, 517] = 3.0e4
    g = torch.Generator().manual_seed(12)
    # Row 2: amax 448 makes s = 1, so x / s = x; values halfway between
    # neighbouring E4M3 codes in [1, 2) (spacing 1/8) round to even.
    x[2] = (torch.randint(8, 16, (K,), generator=g).float() + 0.5) / 8.0
    x[2, 0] = 448.0
    x[3] = torch.randn(K, generator=g) * 2.0
    check(dev, x.to(torch.bfloat16), wq, ws, what="special rows")


def test_few_token_linear_same_codes_as_two_kernels(dev, schedule):
    """The override forces the quantizer + tensor-core GEMM: both paths leave
    the same codes and scales, and their outputs agree within the bar."""
    M, N, K = 1, 4096, 4096
    wq, ws = weights(dev, N, K, seed=21)
    x = synthetic.activations(M, K, outliers=True, seed=22)
    out1, xq1, xs1 = check(dev, x, wq, ws, what="fused")
    fq.fp8q_set_plan_override(1, 16, 4)
    out2, xq2, xs2 = linear(dev, x, wq, ws)
    fq.fp8q_set_plan_override(-1)
    assert torch.equal(xq1, xq2) and torch.equal(xs1, xs2)
    assert_gemm_close(out_values(out1), out_values(out2), "fused vs two kernels")


def test_few_token_linear_full_size_decode_layers(dev):
    """The decode layers at their own sizes: qkv 6144x4096, down 4096x12288,
    gate_up 24576x4096 at M = 1 and 4 (two kernels: larger than the fused
    channelwise form takes), every output against the oracle."""
    for (N, K) in [(6144, 4096), (4096, 12288), (24576, 4096)]:
        wq, ws = weights(dev, N, K, seed=N)
        for M in (1, 4):
            x = synthetic.activations(M, K, outliers=True, seed=M)
            check(dev, x, wq, ws, what=f"{M}x{N}x{K}")


def test_few_token_linear_weights_rewritten_right_before(dev):
    """The kernel streams its first weights before waiting for the previous
    launch; weights written by that launch must still be read fresh."""
    M, N, K = 1, 512, 2048
    x = synthetic.activations(M, K, seed=31)
    wq = torch.empty((N, K), dtype=fq.E4M3, device=dev)
    ws = torch.empty((N,), dtype=torch.float32, device=dev)
    xd = x.to(dev)
    outs, ws_cpu = [], []
    for i in range(4):
        w = synthetic.weights(N, K, seed=200 + i).to(dev)
        torch.cuda.synchronize()
        fq.fp8q_quant_per_token(w, xq=wq, x_scale=ws)
        outs.append(fq.fp8q_linear_channelwise(xd, wq, ws))
        ws_cpu.append(w.cpu())
    torch.cuda.synchronize()
    rq, rs = oracle.quant_per_token(x)
    for i in range(4):
        rwq, rws = oracle.quant_weight_per_channel(ws_cpu[i])
        ref = ref_values(oracle.gemm_channelwise(rq, rwq, rs, rws, threads=THREADS))
        assert_gemm_close(out_values(outs[i]), ref, f"iteration {i}")


@pytest.mark.parametrize("M,K", [(1, 4112), (1, 8208), (1, 12288), (1, 12304), (1, 49152), (2, 32768)])
def test_few_token_linear_wide_rows(dev, M, K):
    """Rows of two and three chunks per warp (the last chunk present for one
    warp only: 4112, 8208), the longest row the fused channelwise launch
    takes (12288, four channels per CTA) and longer ones, which take the
    quantizer and the GEMM."""
    assert fq.fp8q_linear_channelwise_launches(M, 136, K) == (1 if M == 1 and K <= 12288 else 2)
    wq, ws = weights(dev, 136, K, seed=K)
    x = synthetic.activations(M, K, outliers=True, seed=K + M)
    check(dev, x, wq, ws, what=f"{M}x136x{K}")


# ---------------------------------------------------------------------------
# The blockwise linear for one token (group-128 quantization fused, K <= 8192)
# ---------------------------------------------------------------------------

def linear_blockwise(dev, x, wq, ws, bias=None, out_dtype=torch.bfloat16):
    """fp8q_linear_blockwise through the C ABI with caller-owned, canary-filled
    row-padded scratch; returns out, xq [m_pad, K], xs [K/128, m_pad]."""
    L = fq.load_library()
    M, K = x.shape
    N = wq.shape[0]
    m_pad = fq.ceil_align(M, 4)
    xd = x.to(dev)
    xq = torch.full((m_pad, K), 0x5A, dtype=torch.uint8, device=dev)
    xs = torch.full((K // 128, m_pad), -3.0, dtype=torch.float32, device=dev)
    out = torch.empty((M, N), dtype=out_dtype, device=dev)
    bd = None if bias is None else bias.to(dev)
    st = P(torch.cuda.current_stream(dev).cuda_stream)
    rc = L.fp8q_linear_blockwise(P(xd.data_ptr()), P(wq.data_ptr()), P(ws.data_ptr()),
                                 None if bd is None else P(bd.data_ptr()), P(out.data_ptr()), M, N, K,
                                 P(xq.data_ptr()), P(xs.data_ptr()), m_pad,
                                 fq.FP8Q_OUT_FP16 if out_dtype == torch.float16 else fq.FP8Q_OUT_BF16, None, 0, st)
    assert rc == fq.FP8Q_OK
    torch.cuda.synchronize()
    return out, xq, xs


def check_blockwise(dev, x, wq, ws, bias=None, out_dtype=torch.bfloat16, what=""):
    M = x.shape[0]
    out, xq, xs = linear_blockwise(dev, x, wq, ws, bias, out_dtype)
    rq, rs = oracle.quant_group_row_padded(x, 128, threads=THREADS)
    gq, gs = u8(xq), xs.cpu().numpy()
    assert np.array_equal(gq[:M], rq[:M]), f"{what}: group codes differ from the oracle's"
    assert np.array_equal(gs[:, :M], rs[:, :M]), f"{what}: group scales differ from the oracle's"
    assert (gq[M:] == 0x5A).all() and (gs[:, M:] == -3.0).all(), f"{what}: padding rows written"
    fp16 = out_dtype == torch.float16
    ref = ref_values(oracle.gemm_blockwise(rq, u8(wq), rs, ws.cpu().numpy(), M, bias=bias, out_fp16=fp16), fp16)
    assert_gemm_close(out_values(out), ref, what)
    return out, xq, xs


@pytest.mark.parametrize("N,K", [(4096, 7168), (256, 128), (384, 1152), (24576, 3072), (128, 4224), (3072, 12288),
                                 (256, 12416)])
def test_one_token_blockwise_linear_parity(dev, N, K):
    """The blockwise decode layer (two chunks per warp), one K block, a K
    that leaves a warp's 512-value span partly past the row (1152 = 2 x 512
    + 128), a wide N, a second chunk for one warp only (4224), the longest
    row the fused launch takes (three chunks per warp) and one past it (two
    kernels)."""
    assert fq.fp8q_linear_blockwise_launches(1, K) == (1 if K <= 12288 else 2)
    w = synthetic.weights(N, K, seed=N + K)
    wq, ws = fq.fp8q_quant_weight_block128(w.to(dev))
    x = synthetic.activations(1, K, outliers=True, seed=K)
    check_blockwise(dev, x, wq, ws, what=f"blockwise 1x{N}x{K}")


def test_one_token_blockwise_linear_bias_fp16_and_special_groups(dev):
    """Bias, fp16 output, and groups of zeros (scale eps / 448), of one huge
    outlier and of E4M3 rounding midpoints."""
    N, K = 512, 1024
    w = synthetic.weights(N, K, seed=41)
    wq, ws = fq.fp8q_quant_weight_block128(w.to(dev))
    b = synthetic.bias(N, seed=42)
    x = synthetic.activations(1, K, outliers=True, seed=43).float()
    x[0, 128:256] = 0.0
    x[0, 256:384] = 1e-3
    x[0, 300] = 2.0e4
    g = torch.Generator().manual_seed(44)
    x[0, 384:512] = (torch.randint(8, 16, (128,), generator=g).float() + 0.5) / 8.0
    x[0, 384] = 448.0
    x = x.to(torch.bfloat16)
    check_blockwise(dev, x, wq, ws, bias=b, what="blockwise bias bf16")
    check_blockwise(dev, x, wq, ws, bias=b, out_dtype=torch.float16, what="blockwise bias fp16")


def test_one_token_blockwise_same_codes_as_two_kernels(dev, schedule):
    N, K = 4096, 7168
    w = synthetic.weights(N, K, seed=51)
    wq, ws = fq.fp8q_quant_weight_block128(w.to(dev))
    x = synthetic.activations(1, K, outliers=True, seed=52)
    out1, xq1, xs1 = check_blockwise(dev, x, wq, ws, what="fused")
    plan = fq.fp8q_gemm_plan(1, N, K, True)
    fq.fp8q_set_plan_override(plan["swap_ab"], plan["mma_n"], 0 if plan["stream_k"] else plan["split_k"])
    assert fq.fp8q_linear_blockwise_launches(1, K) == 2
    out2, xq2, xs2 = linear_blockwise(dev, x, wq, ws)
    fq.fp8q_set_plan_override(-1)
    assert torch.equal(xq1, xq2) and torch.equal(xs1, xs2)
    assert_gemm_close(out_values(out1), out_values(out2), "blockwise fused vs two kernels")
