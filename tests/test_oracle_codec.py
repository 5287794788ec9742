"""Pins for the oracle's E4M3 codec and its bf16 / fp16 output rounding.

The oracle's codec is written from the E4M3 (float8_e4m3fn) format
definition.  Here it is checked against things that are not the oracle:
torch's own float8_e4m3fn conversions (a library routine), a brute-force
nearest-value search, numpy's float64 -> float16 conversion and exact
rational arithmetic.
"""
from fractions import Fraction

import numpy as np
import torch

import oracle

ALL_CODES = np.arange(256, dtype=np.uint8)
FINITE_CODES = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


def torch_decode(codes: np.ndarray) -> np.ndarray:
    return torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def torch_encode(values: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.asarray(values, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def test_decode_matches_torch_for_all_256_codes():
    ours = oracle.e4m3_decode(ALL_CODES)
    ref = torch_decode(ALL_CODES)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zero survives decoding
    assert np.signbit(ours[0x80]) and not np.signbit(ours[0x00])


def test_decode_extremes():
    d = oracle.e4m3_decode(np.array([0x7E, 0xFE, 0x01, 0x08, 0x38], dtype=np.uint8))
    assert d.tolist() == [448.0, -448.0, 2.0 ** -9, 2.0 ** -6, 1.0]


def test_encode_decode_roundtrip_is_identity_on_finite_codes():
    vals = oracle.e4m3_decode(FINITE_CODES).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), FINITE_CODES)


def _pattern_floats():
    """fp32 values spanning every sign, every exponent and the top 11
    mantissa bits, each with low-bit patterns that decide rounding
    (exact ties, one ulp either side of a tie, sticky bits)."""
    signs = np.array([0, 1], dtype=np.uint32) << np.uint32(31)
    exps = np.arange(0, 255, dtype=np.uint32) << np.uint32(23)
    hi = np.arange(0, 2048, dtype=np.uint32) << np.uint32(12)
    lo = np.array([0, 1, 0x7FF, 0x800, 0x801, 0xFFF, 0x400, 0x123], dtype=np.uint32)
    bits = (signs[:, None, None, None] | exps[None, :, None, None] | hi[None, None, :, None]
            | lo[None, None, None, :]).reshape(-1)
    return bits.view(np.float32)


def test_encode_matches_torch_cast_after_clamp():
    v = _pattern_floats()
    v = v[np.isfinite(v)]
    clamped = np.clip(v, -448.0, 448.0).astype(np.float32)
    ours = oracle.e4m3_encode(v)            # the oracle saturates by itself
    ref = torch_encode(clamped)
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, [(float(v[i]), int(ours[i]), int(ref[i])) for i in bad[:10]]


def _brute_force_encode(v: float) -> int:
    """Nearest finite E4M3 value of the same sign; ties to the even code."""
    if v != v:
        return 0x7F
    sign = 0x80 if np.signbit(v) else 0x00
    a = abs(float(v))
    best, best_d = None, None
    for c in range(0, 0x7F):  # positive finite codes 0x00..0x7E
        d = abs(a - oracle.e4m3_decode(np.array([c], dtype=np.uint8))[0])
        if best is None or d < best_d or (d == best_d and c % 2 == 0):
            best, best_d = c, d
    return sign | best


def test_encode_matches_brute_force_nearest():
    rng = np.random.default_rng(1)
    pos = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    mids = (pos[:-1] + pos[1:]) / 2                     # exact ties
    samples = np.concatenate([
        mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
        np.nextafter(mids.astype(np.float32), np.float32(1e9)),
        rng.uniform(0, 460, 400), 2.0 ** rng.uniform(-14, 9, 400), [0.0, 1e-30, 447.99, 448.0, 500.0],
    ]).astype(np.float32)
    samples = np.concatenate([samples, -samples])
    ours = oracle.e4m3_encode(samples)
    for v, c in zip(samples, ours):
        assert c == _brute_force_encode(float(v)), (float(v), int(c))


def test_encode_saturation_nan_and_signed_zero():
    cases = [  # a list, not a dict: 0.0 and -0.0 compare equal as keys
        (1e30, 0x7E), (-1e30, 0xFE), (np.inf, 0x7E), (-np.inf, 0xFE), (449.0, 0x7E), (-464.0, 0xFE),
        (0.0, 0x00), (-0.0, 0x80), (-1e-10, 0x80),
        (-(2.0 ** -10), 0x80),              # tie between 0 and 2^-9 -> even (zero), sign kept
        (-(2.0 ** -10) * 1.0001, 0x81),
        (2.0 ** -10 * 3, 0x02),             # tie between 2^-9 and 2^-8 -> even code 2
    ]
    v = np.array([c[0] for c in cases], dtype=np.float32)
    assert oracle.e4m3_encode(v).tolist() == [c[1] for c in cases]
    assert oracle.e4m3_encode(np.array([np.nan], dtype=np.float32))[0] == 0x7F


def _exact_round(y: float, mbits: int, emin: int) -> Fraction:
    """Round-to-nearest-even of y onto a binary grid (normal/subnormal), exactly."""
    f = Fraction(y)
    a = abs(f)
    if a == 0:
        return f
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, emin)
    step = Fraction(2) ** (e - mbits)
    q = a / step
    fl = q.numerator // q.denominator
    rem = q - fl
    r = fl + 1 if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1) else fl
    out = r * step
    return -out if f < 0 else out


def test_bf16_rounding_single_rne_from_double():
    rng = np.random.default_rng(2)
    ys = list(rng.normal(0, 3, 300)) + list(2.0 ** rng.uniform(-130, 120, 100))
    # a tie in fp32 reached only through double rounding: single rounding
    # must give the upper neighbour 0x3F81, float32-then-bf16 would give 0x3F80
    ys += [1.00390625 + 2.0 ** -40, 1.00390625, 1.01171875]
    for y in ys:
        bits = oracle.f64_to_bf16_bits(y)
        got = Fraction(float(oracle.bf16_bits_to_float(np.array([bits]))[0]))
        assert got == _exact_round(y, 7, -126), (y, hex(bits))
    assert oracle.f64_to_bf16_bits(1.00390625 + 2.0 ** -40) == 0x3F81
    assert oracle.f64_to_bf16_bits(1.00390625) == 0x3F80
    assert oracle.f64_to_bf16_bits(-0.0) == 0x8000


def test_bf16_rounding_matches_torch_on_float32_values():
    v = _pattern_floats()
    v = v[np.isfinite(v)][::97]
    ref = torch.from_numpy(v.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ours = np.array([oracle.f64_to_bf16_bits(float(x)) for x in v], dtype=np.uint16)
    assert np.array_equal(ours, ref)


def test_f16_rounding_matches_numpy_double_to_half():
    rng = np.random.default_rng(3)
    ys = np.concatenate([rng.normal(0, 100, 500), 2.0 ** rng.uniform(-26, 16, 300),
                         [65504.0, 65519.99, 65520.0, 1e6, 2.0 ** -25, 2.0 ** -24 * 1.5]])
    ys = np.concatenate([ys, -ys])
    with np.errstate(over="ignore"):
        ref = ys.astype(np.float16).view(np.uint16)
    for y, r in zip(ys, ref):
        assert oracle.f64_to_f16_bits(y) == int(r), y
