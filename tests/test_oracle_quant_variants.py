"""Pins of the oracle's quantizer variants: static per-tensor quantization,
power-of-two (UE8M0) group scales and the fused silu_and_mul input.

Each check ties the oracle to something other than itself: float64
mathematics with an error bound (exp, silu), the definition of a power of
two, the already pinned group quantizer and E4M3 codec (the variants reduce
to them), and brute-force nearest-value search over the 256 E4M3 codes."""
import numpy as np
import pytest
import torch

import oracle
import synthetic

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _ulp32(x: np.ndarray) -> np.ndarray:
    """Spacing of fp32 numbers at |x| (float64 result)."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(x, np.finfo(np.float32).tiny)))
    return np.exp2(np.maximum(e, -126.0) - 23.0)


def _enc(v: np.ndarray) -> np.ndarray:
    """E4M3 codes of fp32 values, shaped like the values."""
    return oracle.e4m3_encode(v).reshape(np.shape(v))


def _bf16_values(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# exp and silu: against float64 mathematics
# ---------------------------------------------------------------------------

def test_exp_f32_within_two_ulp_of_exp():
    rng = np.random.default_rng(1)
    t = np.concatenate([
        np.linspace(-32.0, 88.0, 400001, dtype=np.float32),
        rng.uniform(-32.0, 88.0, 400000).astype(np.float32),
        rng.uniform(-1.0, 1.0, 200000).astype(np.float32),
        # around the reduction boundaries n*ln2 +- ln2/2
        (np.arange(-46, 127) * np.float32(np.log(2)) + np.float32(np.log(2) / 2)).astype(np.float32),
    ])
    got = oracle.exp_f32(t).astype(np.float64)
    exact = np.exp(t.astype(np.float64))
    err = np.abs(got - exact) / _ulp32(exact)
    assert err.max() <= 2.0, (err.max(), t[np.argmax(err)])
    assert np.median(err) <= 0.5


def test_exp_f32_special_values_and_range_ends():
    t = np.array([0.0, -0.0, 88.0, 88.0001, 1e30, np.inf, -32.0, -32.0001, -1e30, -np.inf], dtype=np.float32)
    got = oracle.exp_f32(t)
    assert got[0] == 1.0 and got[1] == 1.0
    assert np.isfinite(got[2]) and got[2] > 1e38
    assert np.all(np.isposinf(got[3:6]))
    assert 0.0 < got[6] < 2.0 ** -46
    assert np.all(got[7:] == 0.0)


def test_silu_mul_against_float64_definition():
    rng = np.random.default_rng(2)
    a = np.concatenate([np.linspace(-40, 40, 200001), rng.normal(0, 3, 200000)]).astype(np.float32)
    b = rng.normal(0, 2, a.size).astype(np.float32)
    got = oracle.silu_mul(a, b).astype(np.float64)
    a64, b64 = a.astype(np.float64), b.astype(np.float64)
    exact = a64 / (1.0 + np.exp(-a64)) * b64
    # exp (2 ulp) + add + divide + multiply: a few ulp of the result
    err = np.abs(got - exact) / _ulp32(exact)
    assert err.max() <= 4.0, (err.max(), a[np.argmax(err)])


def test_silu_mul_special_cases():
    a = np.array([0.0, 18.0, 25.0, 1000.0, -89.0, -1000.0, 1.0], dtype=np.float32)
    one = np.ones_like(a)
    got = oracle.silu_mul(a, one)
    assert got[0] == 0.0
    # exp(-a) < 2^-25 -> 1 + exp(-a) == 1 in fp32 -> silu(a) == a exactly
    assert np.array_equal(got[1:4], a[1:4])
    # exp(-a) = +inf -> a / inf = -0
    assert np.all(got[4:6] == 0.0) and np.all(np.signbit(got[4:6]))
    # linear in the second factor, up to one rounding
    b = np.float32(3.0)
    assert oracle.silu_mul(a[6:], np.array([b]))[0] == np.float32(got[6] * b)


# ---------------------------------------------------------------------------
# power-of-two scales
# ---------------------------------------------------------------------------

def test_pow2_ceil_is_the_smallest_power_of_two_not_below():
    rng = np.random.default_rng(3)
    s = np.exp2(rng.uniform(-120, 120, 100000)).astype(np.float32)
    p = oracle.pow2_ceil(s)
    bits = p.view(np.uint32)
    assert np.all(bits & 0x7FFFFF == 0)                  # powers of two
    assert np.all(p >= s) and np.all(p.astype(np.float64) / 2 < s)
    pw = np.exp2(np.arange(-126, 128)).astype(np.float32)
    assert np.array_equal(oracle.pow2_ceil(pw), pw)      # fixed points
    tiny = np.array([0.0, 1e-45, 1e-40, np.finfo(np.float32).tiny], dtype=np.float32)
    assert np.all(oracle.pow2_ceil(tiny) == np.finfo(np.float32).tiny)
    assert np.isposinf(oracle.pow2_ceil(np.array([np.inf], dtype=np.float32)))[0]


# ---------------------------------------------------------------------------
# the group quantizer's options
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("g", [16, 32, 64, 128])
def test_no_options_reduces_to_the_group_quantizer(g):
    x = synthetic.activations(13, 512, outliers=True, seed=30 + g)
    q0, s0 = oracle.quant_group_row_padded(x, g)
    q1, s1 = oracle.quant_group_row_padded_ex(x, g)
    assert np.array_equal(q0, q1) and np.array_equal(s0.view(np.uint32), s1.view(np.uint32))


@pytest.mark.parametrize("g", [16, 32, 64, 128])
def test_ue8m0_scales_and_codes(g):
    M, K = 11, 512
    x = synthetic.activations(M, K, outliers=True, seed=40 + g)
    _, s_raw = oracle.quant_group_row_padded(x, g)
    q, s = oracle.quant_group_row_padded_ex(x, g, scale_ue8m0=True)
    # scales: the plain scales rounded up to powers of two
    assert np.array_equal(s[:, :M], oracle.pow2_ceil(s_raw[:, :M]))
    assert np.all(s[:, :M].view(np.uint32) & 0x7FFFFF == 0)
    # codes: x / s is exact (s a power of two); no value needs saturation
    xv = _bf16_values(oracle._bits16(x)).astype(np.float64)
    sv = np.repeat(s[:, :M].T, g, axis=1).astype(np.float64)
    ratio = xv / sv
    assert np.abs(ratio).max() <= 448.0
    assert np.array_equal(q[:M], _enc(ratio.astype(np.float32)))


def _silu_inputs(M, K, seed):
    gate = synthetic.activations(M, K, outliers=True, seed=seed)
    up = synthetic.activations(M, K, seed=seed + 1)
    return torch.cat([gate, up], dim=1)


@pytest.mark.parametrize("g", [16, 64, 128])
@pytest.mark.parametrize("ue8m0", [False, True])
def test_silu_and_mul_group_quant(g, ue8m0):
    M, K = 9, 256
    x = _silu_inputs(M, K, 50 + g)
    q, s = oracle.quant_group_row_padded_ex(x, g, row_alignment=4, scale_ue8m0=ue8m0, fuse_silu_and_mul=True)
    xv = _bf16_values(oracle._bits16(x))
    y = oracle.silu_mul(xv[:, :K], xv[:, K:]).reshape(M, K)
    # the group quantization of y, stated directly in numpy fp32
    yg = y.reshape(M, K // g, g)
    amax = np.abs(yg).max(axis=2)
    s_ref = (np.maximum(amax, np.float32(1e-10)) / np.float32(448.0)).astype(np.float32)
    if ue8m0:
        s_ref = oracle.pow2_ceil(s_ref)
    assert np.array_equal(s[:, :M].T.view(np.uint32), s_ref.view(np.uint32))
    v = np.clip(yg / s_ref[:, :, None], np.float32(-448.0), np.float32(448.0)).astype(np.float32)
    assert np.array_equal(q[:M], _enc(v.reshape(M, K)))
    # and against float64 mathematics: each code is within half an E4M3
    # step (plus the fp32 error of y) of silu(gate) * up / s
    x64 = xv.astype(np.float64)
    y64 = x64[:, :K] / (1.0 + np.exp(-x64[:, :K])) * x64[:, K:]
    deq = oracle.e4m3_decode(q[:M]).reshape(M, K // g, g)
    t = (y64.reshape(M, K // g, g) / s_ref[:, :, None].astype(np.float64))
    step = np.where(np.abs(t) < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(t), 1e-30))) - 3))
    assert np.all(np.abs(deq - t) <= 0.5 * step + 1e-5 * np.abs(t) + 1e-12)


def test_silu_and_mul_rows_beyond_m_untouched():
    x = _silu_inputs(5, 128, 60)
    q, s = oracle.quant_group_row_padded_ex(x, 64, row_alignment=4, fuse_silu_and_mul=True, xq_init=0xAB,
                                            xs_init=-7.0)
    assert q.shape == (8, 128) and np.all(q[5:] == 0xAB) and np.all(s[:, 5:] == -7.0)


# ---------------------------------------------------------------------------
# static per-tensor quantization
# ---------------------------------------------------------------------------

def _nearest_e4m3(v: float) -> int:
    """Brute force over the 256 codes: nearest finite value, ties to the
    even code (last mantissa bit 0), +-448 beyond the range."""
    vals = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    best, bd = None, None
    for c in range(256):
        if np.isnan(vals[c]):
            continue
        d = abs(vals[c] - v)
        if bd is None or d < bd or (d == bd and (c & 1) == 0 and (best & 1) == 1):
            best, bd = c, d
    if v == 0.0:
        best = 0x80 if np.signbit(v) else 0
    return best


def test_static_quant_unit_scale_is_nearest_e4m3_value():
    rng = np.random.default_rng(4)
    vals = np.concatenate([rng.normal(0, 60, 300), [0.0, 448.0, 464.0, 500.0, 1e4, -1e4, 2.0 ** -10, 0.0068359375]])
    x = torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).reshape(1, -1)
    pad = (-x.shape[1]) % 16
    x = torch.nn.functional.pad(x, (0, pad))
    q = oracle.quant_static(x, 1.0)
    xv = x.float().numpy().reshape(-1).astype(np.float64)
    ref = np.array([_nearest_e4m3(min(max(v, -448.0), 448.0)) for v in xv], dtype=np.uint8)
    assert np.array_equal(q.reshape(-1), ref)


def test_static_quant_with_the_row_scale_equals_per_token_quant():
    x = synthetic.activations(6, 384, outliers=True, seed=70)
    q_tok, s_tok = oracle.quant_per_token(x)
    for m in range(6):
        q = oracle.quant_static(x[m:m + 1], float(s_tok[m]))
        assert np.array_equal(q[0], q_tok[m])


def test_static_quant_saturates_and_divides_in_fp32():
    x = synthetic.activations(4, 256, outliers=True, seed=71)
    s = np.float32(0.013)
    q = oracle.quant_static(x, float(s))
    xv = _bf16_values(oracle._bits16(x))
    v = np.clip(xv / s, np.float32(-448.0), np.float32(448.0)).astype(np.float32)
    assert np.array_equal(q, _enc(v))
    assert np.any(np.abs(xv / s) > 448.0)           # the case exercises saturation
    assert np.all((q[np.abs(xv / s) > 448.0] & 0x7F) == 0x7E)
