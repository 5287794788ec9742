"""Pins for the oracle's dynamic activation quantizers and weight quantizers.

What fixes the expected values here is not the oracle: rows built from
E4M3-representable values whose scale is a known power of two (so the
expected codes are the codes the row was built from), the zero-row and
eps-floor cases, the rounding error bound of RNE, the layout and constants
printed on the row-padding page (``tests/golden/row_padding_cases.txt``), and
library routines (numpy float32 division, numpy block reductions, torch's
float8_e4m3fn cast).
"""
import os

import numpy as np
import pytest
import torch

import oracle
import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "row_padding_cases.txt")


def load_row_padding_golden():
    consts, cases = {}, []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if parts[0] == "case":
                cases.append((int(parts[1]), int(parts[2])))
            else:
                consts[parts[0]] = float(parts[1])
    return consts, cases


def bf16_from_float(v: np.ndarray) -> torch.Tensor:
    t = torch.from_numpy(np.asarray(v, dtype=np.float32)).to(torch.bfloat16)
    assert np.array_equal(t.float().numpy(), np.asarray(v, dtype=np.float32)), "value not bf16-exact"
    return t


def representable_rows(M, K, exps, seed):
    """Rows made of E4M3 values times 2^exps[r], with one +-448 * 2^exps[r]
    entry per row: the row's scale is exactly 2^exps[r] and the expected code
    of every entry is the code it was built from."""
    rng = np.random.default_rng(seed)
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    codes = rng.choice(finite, size=(M, K)).astype(np.uint8)
    pos = rng.integers(0, K, size=M)
    codes[np.arange(M), pos] = np.where(rng.random(M) < 0.5, 0x7E, 0xFE)
    dec = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    vals = dec * (2.0 ** np.asarray(exps, dtype=np.float64))[:, None]
    return codes, bf16_from_float(vals)


def test_exact_roundtrip_per_token():
    M, K = 24, 256
    exps = np.arange(-12, 12)
    codes, x = representable_rows(M, K, exps, seed=5)
    xq, xs = oracle.quant_per_token(x)
    assert np.array_equal(xs, (2.0 ** exps).astype(np.float32))
    assert np.array_equal(xq, codes)


def test_exact_roundtrip_group_quant():
    M, K, g = 7, 512, 128
    rng = np.random.default_rng(6)
    exps = rng.integers(-10, 10, size=(M, K // g))
    codes = np.zeros((M, K), dtype=np.uint8)
    x = torch.zeros((M, K), dtype=torch.bfloat16)
    for j in range(K // g):
        c, xj = representable_rows(M, g, exps[:, j], seed=10 + j)
        codes[:, j * g:(j + 1) * g] = c
        x[:, j * g:(j + 1) * g] = xj
    xq, xs = oracle.quant_group_row_padded(x, g)
    m_pad = 8
    assert xq.shape == (m_pad, K) and xs.shape == (K // g, m_pad)
    assert np.array_equal(xq[:M], codes)
    # scale of (row r, group j) sits at flat index j * m_pad + r
    flat = xs.reshape(-1)
    for r in range(M):
        for j in range(K // g):
            assert flat[j * m_pad + r] == np.float32(2.0 ** exps[r, j])


def test_zero_row_and_eps_floor():
    K = 128
    eps = np.float32(1e-10)
    x = np.zeros((3, K), dtype=np.float32)
    x[1, 5] = 1e-12          # amax below eps: the floor applies to amax
    x[2, 7] = -3.0
    xq, xs = oracle.quant_per_token(torch.from_numpy(x).to(torch.bfloat16))
    floor_scale = np.float32(eps) / np.float32(448.0)
    assert xs[0] == floor_scale and xs[1] == floor_scale
    assert xs[2] == np.float32(3.0) / np.float32(448.0)
    assert np.all(xq[0] == 0)
    # 1e-12 / (1e-10 / 448) = 4.48 -> nearest E4M3 values 4.5 (code 0x49)
    assert xq[1, 5] == 0x49
    assert xq[2, 7] == 0xFE


def test_scale_is_fp32_division_of_amax():
    x = synthetic.activations(64, 1024, seed=3, outliers=True)
    xq, xs = oracle.quant_per_token(x)
    amax = x.float().abs().amax(dim=1).numpy().astype(np.float32)
    ref = np.maximum(amax, np.float32(1e-10)) / np.float32(448.0)
    assert np.array_equal(xs, ref.astype(np.float32))


def _e4m3_half_ulp(v: np.ndarray) -> np.ndarray:
    a = np.abs(v)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    return 0.5 * 2.0 ** (e - 3)


def test_rounding_error_bound_and_max_element():
    x = synthetic.activations(32, 2048, seed=4, outliers=True)
    xq, xs = oracle.quant_per_token(x)
    xf = x.float().numpy().astype(np.float64)
    dec = torch.from_numpy(xq).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    v = xf / xs[:, None].astype(np.float64)
    # x / s is one fp32 rounding away from the exact quotient: allow one fp32 ulp
    bound = (_e4m3_half_ulp(v) + np.abs(v) * 2.0 ** -23) * xs[:, None]
    err = np.abs(dec * xs[:, None] - xf)
    assert np.all(err <= bound)
    # the entry of largest magnitude maps to +-448
    idx = np.argmax(np.abs(xf), axis=1)
    top = xq[np.arange(32), idx]
    assert np.all((top == 0x7E) | (top == 0xFE))


def test_matches_torch_cast_cross_check():
    """Cross-check against torch-CPU ops: amax, float32 divide, clamp and the
    library's own float8_e4m3fn cast."""
    x = synthetic.activations(48, 4096, seed=7, outliers=True)
    xq, xs = oracle.quant_per_token(x)
    xf = x.float()
    s = torch.clamp(xf.abs().amax(dim=1, keepdim=True), min=1e-10) / 448.0
    q = (xf / s).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(xs, s.reshape(-1).numpy())
    assert np.array_equal(xq, q)


def test_row_independence():
    x = synthetic.activations(16, 512, seed=8)
    xq0, xs0 = oracle.quant_per_token(x)
    x2 = x.clone()
    x2[5] *= 3.7
    x2[5, 3] = 100.0
    xq1, xs1 = oracle.quant_per_token(x2)
    keep = np.arange(16) != 5
    assert np.array_equal(xq0[keep], xq1[keep]) and np.array_equal(xs0[keep], xs1[keep])
    assert not np.array_equal(xq0[5], xq1[5])


def test_group_quant_equals_per_token_quant_of_each_group_slice():
    M, K, g = 9, 768, 128
    x = synthetic.activations(M, K, seed=9, outliers=True)
    xq, xs = oracle.quant_group_row_padded(x, g)
    m_pad = 12
    for j in range(K // g):
        q, s = oracle.quant_per_token(x[:, j * g:(j + 1) * g].contiguous())
        assert np.array_equal(xq[:M, j * g:(j + 1) * g], q)
        assert np.array_equal(xs[j, :M], s)
    assert xs.shape == (K // g, m_pad)


def test_row_padded_layout_and_golden_cases():
    consts, cases = load_row_padding_golden()
    g, align = int(consts["group_size"]), int(consts["row_alignment"])
    assert consts["eps"] == 1e-10
    K = 384
    for M, m_pad in cases:
        x = synthetic.activations(M, K, seed=M)
        xq, xs = oracle.quant_group_row_padded(x, g, row_alignment=align, xq_init=0xA5, xs_init=-7.0)
        assert xq.shape == (m_pad, K)
        assert xs.shape == (K // g, m_pad)
        # torch view of the storage as the pages build it: (K/g, m_pad).T
        view = torch.from_numpy(xs).transpose(0, 1)
        assert view.shape == (m_pad, K // g) and view.stride() == (1, m_pad)
        # padding rows are never written
        assert np.all(xq[M:] == 0xA5) and np.all(xs[:, M:] == -7.0)
        # first M rows equal the unpadded quantization (alignment 1): the
        # row-padded path is bit-identical to the legacy one
        xq1, xs1 = oracle.quant_group_row_padded(x, g, row_alignment=1)
        assert np.array_equal(xq[:M], xq1) and np.array_equal(xs[:, :M], xs1)


def test_weight_per_channel_equals_per_token_on_rows():
    w = synthetic.weights(96, 512, seed=11)
    wq, ws = oracle.quant_weight_per_channel(w)
    q, s = oracle.quant_per_token(w)
    assert np.array_equal(wq, q) and np.array_equal(ws, s)


def test_weight_block_quant_scales_and_codes():
    N, K = 256, 384
    w = synthetic.weights(N, K, seed=12)
    wq, ws = oracle.quant_weight_blocks(w, 128, 128)
    wf = w.float().numpy()
    amax = np.abs(wf).reshape(N // 128, 128, K // 128, 128).max(axis=(1, 3)).astype(np.float32)
    ref_s = np.maximum(amax, np.float32(1e-10)) / np.float32(448.0)
    assert np.array_equal(ws, ref_s)
    s_full = np.repeat(np.repeat(ref_s, 128, axis=0), 128, axis=1)
    q = torch.from_numpy((wf / s_full).astype(np.float32)).clamp(-448, 448).to(torch.float8_e4m3fn)
    assert np.array_equal(wq, q.view(torch.uint8).numpy())


@pytest.mark.parametrize("threads", [1, 3])
def test_threaded_rows_match_single_thread(threads):
    x = synthetic.activations(37, 256, seed=13)
    a = oracle.quant_group_row_padded(x, 128, threads=1)
    b = oracle.quant_group_row_padded(x, 128, threads=threads)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
