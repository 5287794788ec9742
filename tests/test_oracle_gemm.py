"""Pins for the oracle's channelwise and blockwise scaled GEMMs.

Expected values come from integer matrix products (numpy int64), from numpy
float64 matmul of exactly decoded operands (sums of E4M3 products are exact
in double, so any summation order gives the same bits), from the fully
dequantized product (scales applied before the sum), and from invariants
that tie the two GEMMs together (K = 128, unit scales, power-of-two scaling,
padded rows).
"""
import numpy as np
import pytest
import torch

import oracle

FINITE = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


def dec(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def random_codes(shape, seed):
    return np.random.default_rng(seed).choice(FINITE, size=shape).astype(np.uint8)


def bf16_value(bits):
    return oracle.bf16_bits_to_float(bits)


def test_brute_force_integer_lattice_4x8x128():
    rng = np.random.default_rng(20)
    ai = rng.integers(-8, 9, size=(4, 128))
    bi = rng.integers(-8, 9, size=(8, 128))
    a = torch.from_numpy(ai.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    b = torch.from_numpy(bi.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    exact = ai.astype(np.int64) @ bi.astype(np.int64).T          # [4, 8]
    ones4, ones8 = np.ones(4, np.float32), np.ones(8, np.float32)
    out, y = oracle.gemm_channelwise(a, b, ones4, ones8, return_double=True)
    assert np.array_equal(y, exact.astype(np.float64))
    ref_bits = torch.from_numpy(exact.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(out, ref_bits)
    # power-of-two scales act exactly
    sa = np.array([0.5, 2.0, 4.0, 0.125], np.float32)
    sb = (2.0 ** np.arange(-3, 5)).astype(np.float32)
    _, y2 = oracle.gemm_channelwise(a, b, sa, sb, return_double=True)
    assert np.array_equal(y2, exact * sa[:, None].astype(np.float64) * sb[None, :].astype(np.float64))


def test_channelwise_matches_float64_matmul():
    M, N, K = 13, 40, 384
    a, b = random_codes((M, K), 21), random_codes((N, K), 22)
    rng = np.random.default_rng(23)
    sa = rng.uniform(0.001, 0.01, M).astype(np.float32)
    sb = rng.uniform(0.0001, 0.001, N).astype(np.float32)
    _, y = oracle.gemm_channelwise(a, b, sa, sb, return_double=True)
    acc = dec(a) @ dec(b).T
    ref = acc * sa[:, None].astype(np.float64) * sb[None, :].astype(np.float64)
    assert np.array_equal(y, ref)


def test_channelwise_bias_and_output_rounding():
    M, N, K = 5, 24, 256
    a, b = random_codes((M, K), 24), random_codes((N, K), 25)
    sa = np.full(M, 1e-3, np.float32)
    sb = np.full(N, 2e-3, np.float32)
    bias = torch.linspace(-1, 1, N).to(torch.bfloat16)
    out0, y0 = oracle.gemm_channelwise(a, b, sa, sb, return_double=True)
    out1, y1 = oracle.gemm_channelwise(a, b, sa, sb, bias=bias, return_double=True)
    assert np.allclose(y1 - y0, bias.double().numpy()[None, :], rtol=0, atol=1e-12)
    for yv, o in zip(y1.reshape(-1), out1.reshape(-1)):
        assert o == oracle.f64_to_bf16_bits(yv)
    out16 = oracle.gemm_channelwise(a, b, sa, sb, bias=bias, out_fp16=True)
    with np.errstate(over="ignore"):
        ref16 = y1.astype(np.float16).view(np.uint16)
    assert np.array_equal(out16, ref16)


def _blockwise_inputs(M, N, K, seed, m_pad=None):
    m_pad = m_pad or M
    a = random_codes((m_pad, K), seed)
    w = random_codes((N, K), seed + 1)
    rng = np.random.default_rng(seed + 2)
    sa = rng.uniform(1e-3, 1e-2, size=(K // 128, m_pad)).astype(np.float32)
    sw = rng.uniform(1e-4, 1e-3, size=(N // 128, K // 128)).astype(np.float32)
    return a, w, sa, sw


def test_blockwise_equals_fully_dequantized_product():
    M, N, K = 6, 256, 512
    a, w, sa, sw = _blockwise_inputs(M, N, K, 30)
    _, y = oracle.gemm_blockwise(a, w, sa, sw, M, return_double=True)
    a_deq = dec(a[:M]) * np.repeat(sa.T[:M].astype(np.float64), 128, axis=1)
    w_deq = dec(w) * np.repeat(np.repeat(sw.astype(np.float64), 128, axis=0), 128, axis=1)
    ref = a_deq @ w_deq.T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-300)


def test_blockwise_is_sum_of_per_block_products():
    M, N, K = 3, 128, 384
    a, w, sa, sw = _blockwise_inputs(M, N, K, 31)
    _, y = oracle.gemm_blockwise(a, w, sa, sw, M, return_double=True)
    for m in range(M):
        for n in range(0, N, 17):
            total = 0.0
            for kb in range(K // 128):
                sl = slice(kb * 128, (kb + 1) * 128)
                p = float(np.dot(dec(a[m, sl]), dec(w[n, sl])))
                total += p * float(sa[kb, m]) * float(sw[n // 128, kb])
            assert y[m, n] == total


def test_blockwise_k128_reduces_to_channelwise():
    M, N, K = 8, 384, 128
    a, w, sa, sw = _blockwise_inputs(M, N, K, 32)
    out_b, y_b = oracle.gemm_blockwise(a, w, sa, sw, M, return_double=True)
    sb = np.repeat(sw[:, 0], 128)
    out_c, y_c = oracle.gemm_channelwise(a, w, sa[0], sb, return_double=True)
    assert np.array_equal(y_b, y_c) and np.array_equal(out_b, out_c)


def test_blockwise_unit_scales_equal_channelwise_unit_scales():
    M, N, K = 4, 128, 1024
    a, w, _, _ = _blockwise_inputs(M, N, K, 33)
    sa = np.ones((K // 128, M), np.float32)
    sw = np.ones((N // 128, K // 128), np.float32)
    _, y_b = oracle.gemm_blockwise(a, w, sa, sw, M, return_double=True)
    _, y_c = oracle.gemm_channelwise(a, w, np.ones(M, np.float32), np.ones(N, np.float32), return_double=True)
    assert np.array_equal(y_b, y_c)
    assert np.array_equal(y_c, dec(a) @ dec(w).T)


def test_blockwise_power_of_two_activation_scaling():
    M, N, K = 4, 128, 256
    a, w, sa, sw = _blockwise_inputs(M, N, K, 34)
    _, y = oracle.gemm_blockwise(a, w, sa, sw, M, return_double=True)
    _, y8 = oracle.gemm_blockwise(a, w, sa * np.float32(8.0), sw, M, return_double=True)
    assert np.array_equal(y8, 8.0 * y)


def test_blockwise_padding_rows_never_reach_the_output():
    M, m_pad, N, K = 5, 8, 256, 256
    a, w, sa, sw = _blockwise_inputs(M, N, K, 35, m_pad=m_pad)
    a_zero, sa_zero = a.copy(), sa.copy()
    a_zero[M:] = 0
    sa_zero[:, M:] = 0.0
    a_junk, sa_junk = a.copy(), sa.copy()
    a_junk[M:] = 0x7F                 # NaN codes
    sa_junk[:, M:] = np.nan
    o1 = oracle.gemm_blockwise(a_zero, w, sa_zero, sw, M)
    o2 = oracle.gemm_blockwise(a_junk, w, sa_junk, sw, M)
    assert o1.shape == (M, N) and np.array_equal(o1, o2)


def test_sampled_positions_match_full_products():
    M, N, K = 7, 256, 384
    a, w, sa, sw = _blockwise_inputs(M, N, K, 36, m_pad=8)
    full = oracle.gemm_blockwise(a, w, sa, sw, M)
    rng = np.random.default_rng(37)
    ms, ns = rng.integers(0, M, 50), rng.integers(0, N, 50)
    assert np.array_equal(oracle.gemm_blockwise_at(a, w, sa, sw, ms, ns), full[ms, ns])
    sa_c = np.random.default_rng(38).uniform(0.01, 0.1, M).astype(np.float32)
    sb_c = np.random.default_rng(39).uniform(0.01, 0.1, N).astype(np.float32)
    bias = torch.randn(N, generator=torch.Generator().manual_seed(0)).to(torch.bfloat16)
    fullc = oracle.gemm_channelwise(a[:M], w, sa_c, sb_c, bias=bias)
    assert np.array_equal(oracle.gemm_channelwise_at(a[:M], w, sa_c, sb_c, ms, ns, bias=bias), fullc[ms, ns])


@pytest.mark.parametrize("threads", [2, 5])
def test_threaded_gemm_matches_single_thread(threads):
    M, N, K = 11, 128, 256
    a, w, sa, sw = _blockwise_inputs(M, N, K, 40, m_pad=12)
    assert np.array_equal(oracle.gemm_blockwise(a, w, sa, sw, M, threads=1),
                          oracle.gemm_blockwise(a, w, sa, sw, M, threads=threads))
