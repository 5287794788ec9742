"""Pins of the oracle's weight-only FP8 linear (W8A16: bf16 activations,
E4M3 weights with per-output-channel scales, the Marlin linear of the A100
page): against float64 matmul of the decoded operands, integer brute force,
and the already pinned channelwise W8A8 GEMM on activations that are exact
E4M3 multiples."""
import numpy as np
import pytest
import torch

import oracle
import synthetic


def _bf16(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).float().numpy().astype(np.float64)


def _round_bf16(y: np.ndarray) -> np.ndarray:
    return torch.from_numpy(y.astype(np.float32)).to(torch.bfloat16).float().numpy()


def test_small_integer_lattice_is_exact():
    rng = np.random.default_rng(11)
    M, N, K = 4, 8, 128
    xv = rng.integers(-8, 9, (M, K)).astype(np.float32)
    wv = rng.integers(-8, 9, (N, K)).astype(np.float32)
    w = oracle.e4m3_encode(wv).reshape(N, K)            # integers |v| <= 8 are exact E4M3 values
    out = oracle.gemm_w8a16(torch.from_numpy(xv).to(torch.bfloat16), w, np.ones(N, np.float32))
    ref = xv.astype(np.int64) @ wv.astype(np.int64).T    # exact integers; the output rounds them to bf16
    got = oracle.bf16_bits_to_float(out)
    assert np.array_equal(got, _round_bf16(ref.astype(np.float64)))


def test_one_hot_rows_read_every_finite_code():
    """One-hot activation rows pick single weights: with unit scales,
    out[m, n] is the weight code w[n, m] decoded, for all 254 finite codes
    (subnormals and both zeros included), against torch's own float8_e4m3fn
    conversion (independent of the oracle's codec)."""
    M, N, K = 16, 128, 256
    rng = np.random.default_rng(12)
    codes = rng.integers(0, 256, (N, K)).astype(np.uint8)
    codes[:, :M] = ((np.arange(N)[:, None] * M + np.arange(M)[None, :]) & 0xFF).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x00
    assert np.unique(codes[:, :M]).size == 254
    x = torch.zeros((M, K), dtype=torch.bfloat16)
    x[torch.arange(M), torch.arange(M)] = 1.0
    out = oracle.gemm_w8a16(x, codes, np.ones(N, np.float32))
    want = torch.from_numpy(codes[:, :M].copy()).view(torch.float8_e4m3fn).float().numpy().T
    assert np.array_equal(oracle.bf16_bits_to_float(out), want)


def test_against_float64_matmul_of_decoded_operands():
    M, N, K = 7, 48, 384
    x = synthetic.activations(M, K, outliers=True, seed=12)
    wq, ws = oracle.quant_weight_per_channel(synthetic.weights(N, K, seed=13))
    bias = synthetic.bias(N, seed=14)
    out, yd = oracle.gemm_w8a16(x, wq, ws, bias=bias, return_double=True)
    wdec = oracle.e4m3_decode(wq).reshape(N, K).astype(np.float64)
    ref = (_bf16(x) @ wdec.T) * ws.astype(np.float64)[None, :] + _bf16(bias)[None, :]
    assert np.allclose(yd, ref, rtol=1e-12, atol=1e-12)
    assert np.array_equal(oracle.bf16_bits_to_float(out), _round_bf16(ref))


def test_equals_channelwise_on_exact_e4m3_activations():
    """x = dec(xq) * 2^e per row is exactly representable in bf16, so W8A16
    on x must equal the channelwise GEMM on (xq, 2^e)."""
    M, N, K = 5, 32, 256
    rng = np.random.default_rng(15)
    codes = rng.integers(0, 256, (M, K)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x10                 # no NaN codes
    sa = np.exp2(rng.integers(-6, 7, M)).astype(np.float32)
    x = torch.from_numpy((oracle.e4m3_decode(codes).reshape(M, K) * sa[:, None]).astype(np.float32))
    assert torch.equal(x.to(torch.bfloat16).float(), x)  # exact in bf16
    wq, ws = oracle.quant_weight_per_channel(synthetic.weights(N, K, seed=16))
    for fp16 in (False, True):
        a = oracle.gemm_w8a16(x.to(torch.bfloat16), wq, ws, out_fp16=fp16)
        b = oracle.gemm_channelwise(codes, wq, sa, ws, out_fp16=fp16)
        assert np.array_equal(a, b)


def test_weight_scale_and_bias_enter_linearly():
    M, N, K = 3, 16, 128
    x = synthetic.activations(M, K, seed=17)
    wq, ws = oracle.quant_weight_per_channel(synthetic.weights(N, K, seed=18))
    _, y1 = oracle.gemm_w8a16(x, wq, ws, return_double=True)
    _, y2 = oracle.gemm_w8a16(x, wq, 2.0 * ws, return_double=True)
    assert np.array_equal(y2, 2.0 * y1)
    bias = synthetic.bias(N, seed=19)
    _, y3 = oracle.gemm_w8a16(x, wq, ws, bias=bias, return_double=True)
    assert np.allclose(y3 - y1, _bf16(bias)[None, :], rtol=0, atol=1e-12)


@pytest.mark.parametrize("threads", [1, 4])
def test_threaded_rows_match(threads):
    x = synthetic.activations(9, 256, seed=20)
    wq, ws = oracle.quant_weight_per_channel(synthetic.weights(24, 256, seed=21))
    assert np.array_equal(oracle.gemm_w8a16(x, wq, ws, threads=threads), oracle.gemm_w8a16(x, wq, ws))
