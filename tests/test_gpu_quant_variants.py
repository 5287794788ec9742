"""GPU parity of the quantizer variants through the C ABI -- static
per-tensor quantization, power-of-two (UE8M0) group scales and the
silu_and_mul-fused group input: codes and fp32 scales bit-exact against the
oracle on the same seeded inputs; rows beyond M never written."""
import ctypes

import numpy as np
import pytest
import torch

import fp8_w8a8_quantized_token_gb300 as fq
import oracle
import synthetic
from gpu_util import u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    d = torch.device("cuda", 0)
    torch.cuda.set_device(d)
    return d


def _silu_input(M, K, seed):
    gate = synthetic.activations(M, K, outliers=True, seed=seed)
    up = synthetic.activations(M, K, seed=seed + 1)
    return torch.cat([gate, up], dim=1).contiguous()


def _group_both(x_cpu, dev, g, ue8m0, silu, row_alignment=4):
    M, W = x_cpu.shape
    K = W // 2 if silu else W
    m_pad = (M + row_alignment - 1) // row_alignment * row_alignment
    xq = torch.empty((m_pad, K), dtype=fq.E4M3, device=dev)
    xq.view(torch.uint8).fill_(0x5A)
    xs = torch.full((K // g, m_pad), -1.0, dtype=torch.float32, device=dev)
    q, s = fq.fp8q_quant_per_token_group_row_padded(x_cpu.to(dev), g, row_alignment=row_alignment, xq=xq,
                                                    x_scale_storage=xs, scale_ue8m0=ue8m0,
                                                    fuse_silu_and_mul=silu)
    torch.cuda.synchronize()
    rq, rs = oracle.quant_group_row_padded_ex(x_cpu, g, row_alignment=row_alignment, scale_ue8m0=ue8m0,
                                              fuse_silu_and_mul=silu, threads=8)
    gq, gs = u8(xq), xs.cpu().numpy()
    assert np.array_equal(gq[:M], rq[:M]), np.argwhere(gq[:M] != rq[:M])[:5]
    assert np.array_equal(gs[:, :M].view(np.uint32), rs[:, :M].view(np.uint32))
    assert np.all(gq[M:] == 0x5A) and np.all(gs[:, M:] == -1.0)
    assert s.stride(0) == 1 and tuple(s.shape) == (m_pad, K // g)
    return gq, gs


@pytest.mark.parametrize("g", [16, 32, 64, 128])
@pytest.mark.parametrize("ue8m0,silu", [(True, False), (False, True), (True, True)])
@pytest.mark.parametrize("M,K", [(1, 256), (7, 4096), (300, 1024), (33, 3072)])
def test_group_variants_bit_exact(dev, g, ue8m0, silu, M, K):
    seed = M * 31 + K + g
    x = _silu_input(M, K, seed) if silu else synthetic.activations(M, K, outliers=True, seed=seed)
    _group_both(x, dev, g, ue8m0, silu)


@pytest.mark.parametrize("g", [16, 32, 64, 128])
@pytest.mark.parametrize("ue8m0", [False, True])
def test_group_many_rows_bit_exact(dev, g, ue8m0):
    """Every group size and scale format at many rows (K = 3200, not a
    multiple of the 256-thread grid stride), padding rows (row_alignment 8)
    left untouched."""
    M, K = 1100, 3200
    x = synthetic.activations(M, K, outliers=True, seed=g * 3 + ue8m0)
    _group_both(x, dev, g, ue8m0, False, row_alignment=8)


def test_group_many_rows_short_rows(dev):
    """K = 48 with g = 16: six units per row, three groups, 26 idle lanes."""
    x = synthetic.activations(1030, 48, outliers=True, seed=5)
    _group_both(x, dev, 16, False, False)


def test_silu_every_bf16_gate_value(dev):
    """All 63488 finite bf16 gate values (up = 1): with groups of 16 the
    scales expose max|silu(gate)| of every group bit-exactly, the codes the
    rest -- GPU silu (with its fixed exp) against the oracle's."""
    bits = np.arange(1 << 16, dtype=np.uint32)
    finite = (bits & 0x7F80) != 0x7F80
    gate_bits = bits[finite].astype(np.uint16)
    n = gate_bits.size
    K = 4096
    rows = (n + K - 1) // K
    gate = np.zeros(rows * K, dtype=np.uint16)
    gate[:n] = gate_bits
    up = np.full(rows * K, 0x3F80, dtype=np.uint16)          # bf16 1.0
    x = np.concatenate([gate.reshape(rows, K), up.reshape(rows, K)], axis=1)
    x = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16)
    for ue8m0 in (False, True):
        _group_both(x, dev, 16, ue8m0, True, row_alignment=1)


def _random_bf16_bits(rng, shape, exp_lo, exp_hi):
    """bf16 values with uniform random sign and 7-bit significand and a
    uniform exponent in [exp_lo, exp_hi] (biased)."""
    sign = rng.integers(0, 2, shape, dtype=np.uint32) << 15
    expo = rng.integers(exp_lo, exp_hi + 1, shape, dtype=np.uint32) << 7
    frac = rng.integers(0, 128, shape, dtype=np.uint32)
    return (sign | expo | frac).astype(np.uint16)


@pytest.mark.parametrize("g", [16, 128])
def test_silu_random_significands_bit_exact(dev, g):
    """Gate and up values with random significands over 2^-20 .. 2^12, so
    the fp32 products silu(gate) * up and their quotients by the group scale
    take general 24-bit significands (the quantizer divides them with a
    Markstein correction): codes and scales bit-exact against the oracle."""
    rng = np.random.default_rng(g)
    M, K = 512, 4096
    gate = _random_bf16_bits(rng, (M, K), 127 - 20, 127 + 12)
    up = _random_bf16_bits(rng, (M, K), 127 - 20, 127 + 12)
    x = torch.from_numpy(np.concatenate([gate, up], axis=1).view(np.int16)).view(torch.bfloat16)
    _group_both(x, dev, g, False, True)


def test_silu_tiny_scales_take_the_division(dev):
    """Groups whose scale is below 2^-90 (tiny values, eps 1e-38) quantize
    with the IEEE division: bit-exact against the oracle as well."""
    rng = np.random.default_rng(3)
    M, K = 8, 256
    gate = _random_bf16_bits(rng, (M, K), 1, 20)          # 2^-126 .. 2^-107
    up = _random_bf16_bits(rng, (M, K), 127 - 4, 127 + 4)
    gate[1] = _random_bf16_bits(rng, (K,), 127 - 60, 127 - 50)
    x = torch.from_numpy(np.concatenate([gate, up], axis=1).view(np.int16)).view(torch.bfloat16)
    m_pad = M
    for g in (16, 128):
        xq = torch.empty((m_pad, K), dtype=fq.E4M3, device=dev)
        xs = torch.empty((K // g, m_pad), dtype=torch.float32, device=dev)
        fq.fp8q_quant_per_token_group_row_padded(x.to(dev), g, eps=1e-38, row_alignment=1, xq=xq,
                                                 x_scale_storage=xs, fuse_silu_and_mul=True)
        torch.cuda.synchronize()
        rq, rs = oracle.quant_group_row_padded_ex(x, g, eps=1e-38, row_alignment=1, fuse_silu_and_mul=True)
        assert np.array_equal(u8(xq), rq)
        assert np.array_equal(xs.cpu().numpy().view(np.uint32), rs.view(np.uint32))
        assert (xs.cpu().numpy()[:, 0] < 2.0 ** -90).all()


def _device_silu(a, b, dev):
    L = fq.load_library()
    at = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)
    bt = torch.from_numpy(np.ascontiguousarray(b, dtype=np.float32)).to(dev)
    out = torch.full_like(at, float("nan"))
    st = L.fp8q_selftest_silu_mul(ctypes.c_void_p(at.data_ptr()), ctypes.c_void_p(bt.data_ptr()),
                                  ctypes.c_void_p(out.data_ptr()), at.numel(),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == fq.FP8Q_OK, fq.status_str(st)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def test_silu_device_function_bit_exact(dev):
    """The fused quantizer's silu(a) * b in fp32, bit for bit against the
    oracle: every finite bf16 gate with b = 1 (the quotient a / (1 +
    exp(-a)) depends on the gate alone, so this covers every quotient the
    kernel can form), an odd count (the last thread's single element), and
    two million random bf16 (gate, up) pairs."""
    bits = np.arange(1 << 16, dtype=np.uint32)
    finite = (bits & 0x7F80) != 0x7F80
    a = oracle.bf16_bits_to_float(bits[finite].astype(np.uint16)).astype(np.float32)
    b = np.ones_like(a)
    got = _device_silu(a, b, dev)
    ref = oracle.silu_mul(a, b)
    diff = np.flatnonzero(got.view(np.uint32) != ref.view(np.uint32))
    assert diff.size == 0, (a[diff[:5]], got[diff[:5]], ref[diff[:5]])
    got = _device_silu(a[:1001], b[:1001], dev)
    assert np.array_equal(got.view(np.uint32), ref[:1001].view(np.uint32))
    rng = np.random.default_rng(17)
    n = 2_000_000
    ga = oracle.bf16_bits_to_float(_random_bf16_bits(rng, (n,), 1, 254)).astype(np.float32)
    ub = oracle.bf16_bits_to_float(_random_bf16_bits(rng, (n,), 127 - 30, 127 + 30)).astype(np.float32)
    got = _device_silu(ga, ub, dev)
    ref = oracle.silu_mul(ga, ub)
    same = (got.view(np.uint32) == ref.view(np.uint32)) | (np.isnan(got) & np.isnan(ref))
    assert same.all(), np.flatnonzero(~same)[:5]


def test_silu_exp_range_ends(dev):
    K = 256
    vals = [0.0, -0.0, 1.0, -1.0, 17.0, 18.0, 25.0, 100.0, 1e30, 3e38, -3e38, -1e30, -100.0, -88.5, -88.0,
            -87.9, -32.0, -31.9, 32.0, 32.1, 88.0, 88.5, 1e-30, -1e-30, 2.0 ** -126, 0.5]
    gate = torch.zeros((2, K))
    gate[0, :len(vals)] = torch.tensor(vals)
    gate[1] = torch.linspace(-120, 120, K)
    up = torch.ones((2, K))
    up[1] = torch.linspace(-3, 3, K)
    x = torch.cat([gate, up], dim=1).to(torch.bfloat16)
    for g in (16, 128):
        for ue8m0 in (False, True):
            _group_both(x, dev, g, ue8m0, True)


def test_silu_prefill_rows_sampled(dev):
    """The MLP shape of the benchmark workload (gate/up of 12288 each) at a
    prefill size; 48 rows checked against the oracle row by row."""
    M, K = 2048, 12288
    x = _silu_input(M, K, 91).to(dev)
    q, s = fq.fp8q_quant_per_token_group_row_padded(x, 128, scale_ue8m0=True, fuse_silu_and_mul=True)
    torch.cuda.synchronize()
    gq, gs = u8(q), s.cpu().numpy()
    rows = np.random.default_rng(5).choice(M, 48, replace=False)
    xr = x[torch.from_numpy(rows).to(dev)].cpu()
    rq, rs = oracle.quant_group_row_padded_ex(xr, 128, row_alignment=1, scale_ue8m0=True, fuse_silu_and_mul=True,
                                              threads=8)
    assert np.array_equal(gq[rows], rq)
    assert np.array_equal(gs[rows].view(np.uint32), rs.T.view(np.uint32))


def test_ue8m0_scales_are_powers_of_two_and_no_code_saturates(dev):
    x = synthetic.activations(64, 2048, outliers=True, seed=92)
    gq, gs = _group_both(x, dev, 128, True, False)
    assert np.all(gs[:, :64].view(np.uint32) & 0x7FFFFF == 0)
    assert not np.any((gq[:64] & 0x7F) == 0x7F)          # no NaN codes


def test_flags_zero_through_ex_equals_plain(dev):
    L = fq.load_library()
    M, K, g = 37, 1024, 64
    x = synthetic.activations(M, K, outliers=True, seed=93).to(dev)
    qa, sa = fq.fp8q_quant_per_token_group_row_padded(x, g, row_alignment=4)
    qb = torch.empty_like(qa)
    sb = torch.empty((K // g, qa.shape[0]), dtype=torch.float32, device=dev)
    st = L.fp8q_quant_per_token_group_row_padded_ex(ctypes.c_void_p(x.data_ptr()), M, K, K, g, 1e-10, 4, 0,
                                                    ctypes.c_void_p(qb.data_ptr()), ctypes.c_void_p(sb.data_ptr()),
                                                    qa.shape[0], ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert st == fq.FP8Q_OK
    assert np.array_equal(u8(qa)[:M], u8(qb)[:M])
    assert np.array_equal(sa.transpose(0, 1).cpu().numpy()[:, :M], sb.cpu().numpy()[:, :M])


def test_ex_rejects_bad_flags_and_short_rows(dev):
    L = fq.load_library()
    M, K = 4, 256
    x = torch.zeros((M, 2 * K), dtype=torch.bfloat16, device=dev)
    q = torch.empty((M, K), dtype=fq.E4M3, device=dev)
    s = torch.empty((K // 128, M), dtype=torch.float32, device=dev)
    P = ctypes.c_void_p
    args = lambda ldx, flags: (P(x.data_ptr()), M, K, ldx, 128, 1e-10, 4, flags, P(q.data_ptr()),
                               P(s.data_ptr()), M, P(torch.cuda.current_stream().cuda_stream))
    assert L.fp8q_quant_per_token_group_row_padded_ex(*args(2 * K, 4)) == fq.FP8Q_ERR_INVALID_ARG
    assert L.fp8q_quant_per_token_group_row_padded_ex(*args(K, fq.FP8Q_QUANT_SILU_AND_MUL)) == \
        fq.FP8Q_ERR_INVALID_ARG
    assert L.fp8q_quant_per_token_group_row_padded_ex(*args(2 * K, fq.FP8Q_QUANT_SILU_AND_MUL)) == fq.FP8Q_OK
    torch.cuda.synchronize()


# ---------------------------------------------------------------------------
# static per-tensor quantization
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M,K", [(1, 16), (5, 256), (64, 4096), (300, 12288), (2, 65552)])
@pytest.mark.parametrize("scale", [1.0, 0.013, 2.0 ** -10, 3.5])
def test_static_bit_exact(dev, M, K, scale):
    x = synthetic.activations(M, K, outliers=True, seed=M + K)
    s = torch.tensor([scale], dtype=torch.float32, device=dev)
    q, rep = fq.fp8q_quant_static_per_tensor(x.to(dev), s, repeat_scale=True)
    torch.cuda.synchronize()
    ref = oracle.quant_static(x, scale, threads=8)
    assert np.array_equal(u8(q), ref)
    assert np.all(rep.cpu().numpy() == np.float32(scale))


def test_static_strided_input_no_rep_and_m0(dev):
    M, K, ldx = 9, 1024, 1536
    big = synthetic.activations(M, ldx, outliers=True, seed=94)
    x = big.to(dev)[:, :K]
    s = torch.tensor([0.02], dtype=torch.float32, device=dev)
    xq = torch.empty((M + 1, K), dtype=fq.E4M3, device=dev)
    xq.view(torch.uint8).fill_(0x5A)
    q, rep = fq.fp8q_quant_static_per_tensor(x, s, xq=xq[:M])
    torch.cuda.synchronize()
    assert rep is None
    assert np.array_equal(u8(xq)[:M], oracle.quant_static(big[:, :K].contiguous(), 0.02))
    assert np.all(u8(xq)[M] == 0x5A)
    q0, _ = fq.fp8q_quant_static_per_tensor(x[:0], s)
    assert q0.shape == (0, K)


def test_static_scale_from_a_device_tensor_feeds_the_channelwise_gemm(dev):
    """The repeated scale is the per-token vector the channelwise GEMM takes:
    static-quantized activations through the GEMM equal the oracle GEMM on
    the oracle's static codes."""
    from gpu_util import assert_gemm_close, out_values, ref_values
    M, N, K = 24, 512, 1024
    x = synthetic.activations(M, K, seed=95)
    w = synthetic.weights(N, K, seed=95)
    s = torch.tensor([float(x.float().abs().max()) / 448.0], dtype=torch.float32, device=dev)
    xq, rep = fq.fp8q_quant_static_per_tensor(x.to(dev), s, repeat_scale=True)
    wq, ws = fq.fp8q_quant_per_token(w.to(dev))
    out = fq.fp8q_scaled_mm_channelwise(xq, wq, rep, ws)
    torch.cuda.synchronize()
    rq = oracle.quant_static(x, float(s.item()))
    rwq, rws = oracle.quant_per_token(w)
    ref = oracle.gemm_channelwise(rq, rwq, np.full(M, np.float32(s.item())), rws)
    assert_gemm_close(out_values(out), ref_values(ref), "static quant -> channelwise gemm")
