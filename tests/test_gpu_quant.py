"""GPU parity of the quantizers through the C ABI: codes and fp32 scales
bit-exact against the oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import fp8_w8a8_quantized_token_gb300 as fq
import oracle
import synthetic
from gpu_util import THREADS, quant_both_group, quant_both_per_token, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    d = torch.device("cuda", 0)
    torch.cuda.set_device(d)
    return d


@pytest.mark.parametrize("M,K,outliers", [
    (16, 512, False),        # the tiny channelwise layer
    (1, 4096, True), (7, 4096, True), (300, 4096, True),
    (33, 12288, True), (5, 16, False), (64, 7168, False), (3, 3072, True),
    (2, 65552, False),       # longer than the register-cached path: two-pass kernel
    # many rows: the four-chunks-per-thread configuration, whole and ragged
    # last thread (K = 4112: 257 chunks over 96 threads)
    (1024, 4096, True), (1500, 4112, True), (1031, 12288, False), (1024, 48, False),
    # 4096 rows and more: one bulk copy of each row into shared memory; 64
    # threads of 8 units at K = 4096, ragged unit counts (K = 4112: 514 units
    # over 96 threads; K = 48: 6 units, one warp), 256 threads at the longest
    # bulk row (K = 16384), and the next longer row back on the
    # four-chunks-per-thread kernel (K = 16400)
    (4096, 4096, True), (4099, 4112, True), (4100, 48, False), (4096, 7168, True), (4096, 16384, False),
    (4096, 16400, False),
])
def test_per_token_bit_exact(dev, M, K, outliers):
    x = synthetic.activations(M, K, seed=M * 7 + K, outliers=outliers)
    quant_both_per_token(x, dev)


def test_per_token_strided_input_and_no_overrun(dev):
    M, K, ldx = 9, 1024, 1536
    big = synthetic.activations(M, ldx, seed=3, outliers=True)
    x_gpu = big.to(dev)[:, :K]
    xq = torch.empty((M + 1, K), dtype=fq.E4M3, device=dev)
    xq.view(torch.uint8).fill_(0x5A)
    xs = torch.full((M + 4,), -1.0, dtype=torch.float32, device=dev)
    fq.fp8q_quant_per_token(x_gpu, xq=xq[:M], x_scale=xs)
    torch.cuda.synchronize()
    rq, rs = oracle.quant_per_token(big[:, :K].contiguous())
    assert np.array_equal(u8(xq)[:M], rq)
    assert np.array_equal(xs.cpu().numpy()[:M], rs)
    assert np.all(u8(xq)[M] == 0x5A) and np.all(xs.cpu().numpy()[M:] == -1.0)


def test_many_rows_strided_input_and_no_overrun(dev):
    """Many-row quantization of a strided input (the per-token kernel's bulk
    row copies start at row * ldx); rows and scales beyond M are never
    written (per-token and group-128)."""
    M, K, ldx = 4100, 1024, 1536
    big = synthetic.activations(M, ldx, seed=13, outliers=True)
    x_gpu = big.to(dev)[:, :K]
    xq = torch.empty((M + 1, K), dtype=fq.E4M3, device=dev)
    xq.view(torch.uint8).fill_(0x5A)
    xs = torch.full((M + 4,), -1.0, dtype=torch.float32, device=dev)
    fq.fp8q_quant_per_token(x_gpu, xq=xq[:M], x_scale=xs)
    torch.cuda.synchronize()
    rq, rs = oracle.quant_per_token(big[:, :K].contiguous(), threads=THREADS)
    assert np.array_equal(u8(xq)[:M], rq)
    assert np.array_equal(xs.cpu().numpy()[:M], rs)
    assert np.all(u8(xq)[M] == 0x5A) and np.all(xs.cpu().numpy()[M:] == -1.0)
    gq, gsv = fq.fp8q_quant_per_token_group_row_padded(x_gpu, 128)
    torch.cuda.synchronize()
    rq, rs = oracle.quant_group_row_padded(big[:, :K].contiguous(), 128, threads=THREADS)
    assert np.array_equal(u8(gq)[:M], rq[:M])
    assert np.array_equal(gsv.transpose(0, 1).cpu().numpy()[:, :M], rs[:, :M])


def test_per_token_special_rows(dev):
    K = 256
    x = torch.zeros((6, K), dtype=torch.float32)
    x[1, 3] = 1e-12                 # below the eps floor
    x[2] = torch.linspace(-448, 448, K)
    x[3, :] = -0.0
    x[4, 0] = 3e38                  # huge amax: everything else underflows (signed zeros)
    x[4, 1:] = -torch.linspace(1, 2, K - 1)
    x[5] = torch.tensor([(-1) ** i * 2.0 ** (-(i % 20)) for i in range(K)])
    quant_both_per_token(x.to(torch.bfloat16), dev)


def _tie_rows(K):
    """Rows whose quotients x / s land exactly on midpoints between
    neighbouring E4M3 values (ties, resolved to the even code), or one bf16
    step beside them.  Each row's first element fixes amax = 448 * s, so
    s is exact; s has at most 3 significant bits and a midpoint 5, so every
    s * midpoint is a bf16 value,
    but 1 / s is not a power of two, so x * (1 / s) can miss the tie by an
    ulp -- where only the division gives the right code."""
    codes = np.arange(0x08, 0x7E, dtype=np.uint8)             # positive normal E4M3 values
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    mids = (vals[:-1] + vals[1:]) / 2
    rows = []
    for s in (1.5, 1.25, 1.75, 0.375, 3.0 * 2.0 ** -7, 1.25 * 2.0 ** 5, 1.75 * 2.0 ** -9):
        x = np.concatenate([[448.0 * s], s * mids, -s * mids])
        row = torch.zeros(K, dtype=torch.float64)
        row[:x.size] = torch.from_numpy(x)
        exact = row.to(torch.bfloat16)
        assert torch.equal(exact.double(), row), "a tie value is not a bf16 value"
        rows.append(exact)
        bump = exact.view(torch.int16).clone()
        bump[1:x.size] += 1                                     # one bf16 step off each tie
        rows.append(bump.view(torch.bfloat16))
    return torch.stack(rows)


def test_quotients_on_e4m3_rounding_midpoints(dev):
    x = _tie_rows(256)
    quant_both_per_token(x, dev)
    quant_both_group(x, dev, 128)


def test_special_tie_and_tiny_scale_rows_in_many_row_launches(dev):
    """The special rows, the midpoint rows and rows with zero or subnormal
    scales, repeated into launches of 4096 rows and more, so that the
    many-row (bulk copy) kernel quantizes them too."""
    special = torch.zeros((8, 256), dtype=torch.float32)
    special[1, 3] = 1e-12
    special[2] = torch.linspace(-448, 448, 256)
    special[3, :] = -0.0
    special[4, 0] = 3e38
    special[4, 1:] = -torch.linspace(1, 2, 255)
    special[5] = torch.tensor([(-1) ** i * 2.0 ** (-(i % 20)) for i in range(256)])
    special[6, 7] = 1e-40
    special[7, :3] = torch.tensor([3e-39, -2e-38, 5e-40])
    rows = torch.cat([special.to(torch.bfloat16), _tie_rows(256)])
    x = rows.repeat((4100 + rows.shape[0] - 1) // rows.shape[0], 1)[:4100].contiguous()
    quant_both_per_token(x, dev)
    for eps in (1e-44, 1e-41):
        q, sc = fq.fp8q_quant_per_token(x.to(dev), eps=eps)
        torch.cuda.synchronize()
        rq, rs = oracle.quant_per_token(x, eps=eps, threads=THREADS)
        assert np.array_equal(u8(q), rq)
        assert np.array_equal(sc.cpu().numpy().view(np.uint32), rs.view(np.uint32))


def test_every_bf16_significand_under_many_scales(dev):
    """Rows with scales over a wide exponent range; every row holds values
    of all 128 bf16 significands, both signs, at many exponents below its
    amax (and signed zeros), so each quotient pattern meets many scales."""
    rng = np.random.default_rng(77)
    M, K = 4096, 2048   # the many-row per-token kernel
    amax_exp = rng.integers(-30, 30, M)
    amax = (1.0 + rng.integers(0, 128, M) / 128.0) * 2.0 ** amax_exp
    sig = np.tile(np.arange(128), K // 128)[None, :] + np.zeros((M, 1), dtype=np.int64)
    exp = amax_exp[:, None] - rng.integers(1, 24, (M, K))
    vals = (1.0 + sig / 128.0) * 2.0 ** exp
    vals *= np.where(rng.random((M, K)) < 0.5, -1.0, 1.0)
    vals[:, 0] = amax
    vals[:, 1] = -0.0
    x = torch.from_numpy(vals).to(torch.bfloat16)
    assert torch.equal(x.double().abs().amax(dim=1), torch.from_numpy(amax))
    quant_both_per_token(x, dev)
    quant_both_group(x, dev, 128)


def test_per_token_m0_is_noop(dev):
    x = torch.empty((0, 64), dtype=torch.bfloat16, device=dev)
    xq, xs = fq.fp8q_quant_per_token(x)
    assert xq.shape == (0, 64) and xs.shape == (0,)


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 7, 13, 16, 31, 64, 256])
def test_group_row_padded_decode_sizes(dev, M):
    x = synthetic.activations(M, 7168, seed=M)
    xq, xs, _, _ = quant_both_group(x, dev, 128, xq_fill=0xA5, xs_fill=-7.0)
    m_pad = fq.ceil_align(M, 4)
    assert xq.shape == (m_pad, 7168) and xs.shape == (56, m_pad)
    # padding rows are never written
    assert np.all(u8(xq)[M:] == 0xA5)
    assert np.all(xs.cpu().numpy()[:, M:] == -7.0)


@pytest.mark.parametrize("M,K", [(8192, 3072), (1000, 12288), (37, 1024)])
def test_group_row_padded_prefill_sizes_with_outliers(dev, M, K):
    x = synthetic.activations(M, K, seed=K, outliers=True)
    quant_both_group(x, dev, 128)


@pytest.mark.parametrize("group", [16, 32, 64])
def test_group_sizes(dev, group):
    x = synthetic.activations(21, 1024, seed=group, outliers=True)
    quant_both_group(x, dev, group, xq_fill=0xA5, xs_fill=-7.0)


def test_group_quant_view_matches_the_pages_layout(dev):
    M, K = 5, 384
    x = synthetic.activations(M, K, seed=2).to(dev)
    xq, xsv = fq.fp8q_quant_per_token_group_row_padded(x, 128)
    assert tuple(xsv.shape) == (8, 3) and xsv.stride() == (1, 8)
    assert tuple(xq.shape) == (8, K)


def test_weight_block128_quant(dev):
    N, K = 384, 1024
    w = synthetic.weights(N, K, seed=5)
    wq, ws = fq.fp8q_quant_weight_block128(w.to(dev))
    torch.cuda.synchronize()
    rq, rs = oracle.quant_weight_blocks(w, 128, 128)
    assert np.array_equal(u8(wq), rq)
    assert np.array_equal(ws.cpu().numpy(), rs)


def test_weight_per_channel_quant_is_per_token_quant_of_rows(dev):
    w = synthetic.weights(512, 4096, seed=6)
    wq, ws = fq.fp8q_quant_per_token(w.to(dev))
    torch.cuda.synchronize()
    rq, rs = oracle.quant_weight_per_channel(w)
    assert np.array_equal(u8(wq), rq) and np.array_equal(ws.cpu().numpy(), rs)


def test_tiny_eps_zero_and_subnormal_scales(dev):
    """eps so small that max(amax, eps) / 448 is zero or subnormal in fp32:
    the kernels divide with the IEEE division there, as the oracle does."""
    x = torch.zeros((4, 256), dtype=torch.float32)
    x[1, 7] = 1e-40                    # subnormal scale
    x[2, :3] = torch.tensor([3e-39, -2e-38, 5e-40])
    x[3] = torch.linspace(-1, 1, 256)
    x = x.to(torch.bfloat16)
    for eps in (1e-44, 1e-41):
        q, s = fq.fp8q_quant_per_token(x.to(dev), eps=eps)
        torch.cuda.synchronize()
        rq, rs = oracle.quant_per_token(x, eps=eps)
        assert np.array_equal(u8(q), rq)
        assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))
