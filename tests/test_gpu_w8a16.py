"""GPU parity of the weight-only FP8 linear (W8A16: bf16 activations, E4M3
weights converted exactly to bf16 in shared memory, kind::f16 MMAs) through
the C ABI, against the oracle (exact products, double sums), within the GEMM
tolerance; edge shapes, bias, fp16 output, strided input, the sampled
full-size decode layer."""
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
    return d


def _case(dev, M, N, K, bias=False, fp16=False, seed=0):
    x = synthetic.activations(M, K, outliers=True, seed=seed + M + K)
    w = synthetic.weights(N, K, seed=seed + N)
    wq, ws = fq.fp8q_quant_per_token(w.to(dev))          # per-channel E4M3 weights
    b = synthetic.bias(N, seed=seed) if bias else None
    out = fq.fp8q_scaled_mm_w8a16(x.to(dev), wq, ws, bias=None if b is None else b.to(dev),
                                  out_dtype=torch.float16 if fp16 else torch.bfloat16)
    torch.cuda.synchronize()
    ref = oracle.gemm_w8a16(x, wq.cpu(), ws.cpu(), bias=b, out_fp16=fp16, threads=8)
    assert_gemm_close(out_values(out), ref_values(ref, fp16), f"w8a16 {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [
    (1, 4096, 4096), (7, 4096, 4096), (16, 512, 1024),   # 16-token tiles
    (24, 384, 1040),                                     # 32-token tile, ragged K (not a multiple of 128)
    (33, 1024, 2048),                                    # two 32-token tiles, ragged
    (5, 256, 128),                                       # one K block
])
def test_w8a16_parity(dev, M, N, K):
    _case(dev, M, N, K)


def test_w8a16_bias_fp16_and_long_k(dev):
    _case(dev, 16, 4096, 12288, bias=True, fp16=True, seed=3)
    _case(dev, 3, 1024, 7168, bias=True, seed=4)


@pytest.mark.parametrize("M", [1, 2, 3, 4])
@pytest.mark.parametrize("N,K", [(392, 1040), (8, 16), (4096, 4096), (264, 12288)])
def test_w8a16_few_tokens_on_cuda_cores(dev, M, N, K):
    """One or two tokens: matrix-vector products on the CUDA cores (K not a
    multiple of the 512-byte chunk, one 16-element piece, N not a multiple of
    a CTA's rows); three and four: the 16-token tensor-core tiles; bias and
    fp16 output on every other case."""
    _case(dev, M, N, K, bias=(M % 2 == 1), fp16=(M == 2), seed=M)


def test_w8a16_few_tokens_strided_operands(dev):
    """Row strides above K for both the activations and the weights (two
    tokens: the CUDA-core path)."""
    M, N, K, ldx, ldw = 2, 520, 2064, 2080, 2112
    big = synthetic.activations(M, ldx, outliers=True, seed=21)
    w = synthetic.weights(N, K, seed=22).to(dev)
    wq, ws = fq.fp8q_quant_per_token(w)
    wstore = torch.zeros((N, ldw), dtype=fq.E4M3, device=dev)
    wstore[:, :K] = wq
    wstore[:, K:].view(torch.uint8).fill_(0x7E)     # 448 past K: must never be read
    out = fq.fp8q_scaled_mm_w8a16(big.to(dev)[:, :K], wstore[:, :K], ws)
    torch.cuda.synchronize()
    ref = oracle.gemm_w8a16(big[:, :K].contiguous(), wq.cpu(), ws.cpu())
    assert_gemm_close(out_values(out), ref_values(ref), "w8a16 few tokens strided")


@pytest.mark.parametrize("M", [2, 16, 32])
def test_w8a16_every_e4m3_code_converts_exactly(dev, M):
    """One-hot activation rows pick single weights: with unit weight scales,
    out[m, n] = w[n, m] exactly (an E4M3 value is a bf16 value), so every
    finite code, subnormals and both zeros included, must come out as the
    oracle's decode of it -- an exhaustive check of the on-chip E4M3
    conversion of the CUDA-core path (M = 2) and the 16- and 32-token
    tiles."""
    N, K = 128, 256
    rng = np.random.default_rng(11)
    codes = rng.integers(0, 256, (N, K)).astype(np.uint8)
    codes[:, :M] = ((np.arange(N)[:, None] * M + np.arange(M)[None, :]) & 0xFF).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x00                # the two NaN codes are outside the contract
    assert np.unique(codes[:, :M]).size == 254
    x = torch.zeros((M, K), dtype=torch.bfloat16)
    x[torch.arange(M), torch.arange(M)] = 1.0
    wq = torch.from_numpy(codes).to(dev).view(fq.E4M3)
    ws = torch.ones(N, dtype=torch.float32, device=dev)
    out = fq.fp8q_scaled_mm_w8a16(x.to(dev), wq, ws)
    torch.cuda.synchronize()
    want = oracle.e4m3_decode(codes[:, :M]).reshape(N, M).T
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.array_equal(got, want)


def test_w8a16_strided_input_and_m0(dev):
    M, N, K, ldx = 9, 512, 1024, 1536
    big = synthetic.activations(M, ldx, outliers=True, seed=5)
    x = big.to(dev)[:, :K]
    w = synthetic.weights(N, K, seed=6).to(dev)
    wq, ws = fq.fp8q_quant_per_token(w)
    out = fq.fp8q_scaled_mm_w8a16(x, wq, ws)
    torch.cuda.synchronize()
    ref = oracle.gemm_w8a16(big[:, :K].contiguous(), wq.cpu(), ws.cpu())
    assert_gemm_close(out_values(out), ref_values(ref), "w8a16 strided")
    out0 = fq.fp8q_scaled_mm_w8a16(x[:0], wq, ws)
    assert out0.shape == (0, N)


def test_w8a16_e4m3_exact_activations_equal_channelwise(dev):
    """Activations that are E4M3 codes times power-of-two row scales: W8A16
    and the W8A8 channelwise GEMM compute the same products; both within
    tolerance of the same oracle value."""
    M, N, K = 12, 1024, 2048
    rng = np.random.default_rng(7)
    codes = rng.integers(0, 256, (M, K)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x10
    sa = np.exp2(rng.integers(-4, 5, M)).astype(np.float32)
    x = torch.from_numpy((oracle.e4m3_decode(codes).reshape(M, K) * sa[:, None]).astype(np.float32))
    x = x.to(torch.bfloat16)
    wq, ws = fq.fp8q_quant_per_token(synthetic.weights(N, K, seed=8).to(dev))
    out = fq.fp8q_scaled_mm_w8a16(x.to(dev), wq, ws)
    torch.cuda.synchronize()
    ref = oracle.gemm_channelwise(codes, wq.cpu(), sa, ws.cpu())
    assert_gemm_close(out_values(out), ref_values(ref), "w8a16 = channelwise")


def test_w8a16_full_size_decode_layer_sampled(dev):
    """The gate_up shape at a decode size: all outputs of 6 sampled rows."""
    M, N, K = 16, 24576, 4096
    x = synthetic.activations(M, K, outliers=True, seed=9)
    wq, ws = fq.fp8q_quant_per_token(synthetic.weights(N, K, seed=10).to(dev))
    out = fq.fp8q_scaled_mm_w8a16(x.to(dev), wq, ws)
    torch.cuda.synchronize()
    rows = [0, 3, 7, 8, 14, 15]
    ref = oracle.gemm_w8a16(x[rows], wq.cpu(), ws.cpu(), threads=8)
    assert_gemm_close(out_values(out)[rows], ref_values(ref), "w8a16 full size")


def test_w8a16_rejects_bad_arguments(dev):
    L = fq.load_library()
    P = ctypes.c_void_p
    x = torch.zeros((4, 256), dtype=torch.bfloat16, device=dev)
    w = torch.zeros((128, 256), dtype=fq.E4M3, device=dev)
    ws = torch.ones(128, dtype=torch.float32, device=dev)
    out = torch.empty((4, 128), dtype=torch.bfloat16, device=dev)
    st = P(torch.cuda.current_stream().cuda_stream)
    call = lambda M, N, K, ldx, ldw: L.fp8q_scaled_mm_w8a16(P(x.data_ptr()), ldx, P(w.data_ptr()), ldw,
                                                             P(ws.data_ptr()), None, P(out.data_ptr()), M, N, K,
                                                             0, st)
    assert call(4, 128, 250, 256, 256) == fq.FP8Q_ERR_INVALID_ARG      # K % 16
    assert call(4, 128, 256, 200, 256) == fq.FP8Q_ERR_INVALID_ARG      # ldx < K
    assert call(4, 100, 256, 256, 256) == fq.FP8Q_ERR_INVALID_ARG      # N % 8
    assert call(4, 128, 256, 256, 256) == fq.FP8Q_OK
    torch.cuda.synchronize()
