"""GPU parity of the scaled FP8 GEMMs through the C ABI against the oracle,
element by element, within |gpu - ref| <= 1e-2 * (|ref| + 1).

Both sides quantize the same seeded bf16 inputs independently (the codes
and scales are first checked bit-exact), then each side runs its own GEMM.
Every kernel instantiation and K-split is exercised by forcing the
schedule, on shapes with ragged M, N and K tails."""
import numpy as np
import pytest
import torch

import fp8_w8a8_quantized_token_gb300 as fq
import oracle
import synthetic
from gpu_util import (THREADS, assert_gemm_close, out_values, quant_both_group, quant_both_per_token, ref_values,
                      u8)

pytestmark = pytest.mark.gpu

# (swap_ab, mma_n, split_k); split_k 0 = stream-K (swapped tiles).  On the
# 392 x 1040 shapes below, M = 1 has 4 tiles x 9 K blocks = 36 pairs: 36
# stream-K CTAs of one K block each, so every tile is split 9 ways.
SCHEDULES = [(1, 16, 1), (1, 16, 3), (1, 16, 5), (1, 32, 2), (1, 32, 8), (1, 64, 1), (1, 64, 4), (1, 64, 7),
             (1, 128, 1), (1, 128, 2), (1, 128, 6), (0, 256, 1), (0, 256, 2), (0, 256, 5),
             (0, 128, 1), (0, 128, 3), (0, 64, 1), (0, 64, 2), (0, 32, 1), (0, 32, 4),
             (1, 16, 0), (1, 32, 0)]


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


def channelwise_case(dev, M, N, K, seed=0, bias=False, outliers=True, out_dtype=torch.bfloat16, workspace="auto"):
    x = synthetic.activations(M, K, seed=seed, outliers=outliers)
    w = synthetic.weights(N, K, seed=seed)
    b = synthetic.bias(N, seed=seed) if bias else None
    xq, xs, rq, rs = quant_both_per_token(x, dev)
    wq, ws, rwq, rws = quant_both_per_token(w, dev)
    out = fq.fp8q_scaled_mm_channelwise(xq, wq, xs, ws, bias=None if b is None else b.to(dev),
                                        out_dtype=out_dtype, workspace=workspace)
    torch.cuda.synchronize()
    fp16 = out_dtype == torch.float16
    ref = ref_values(oracle.gemm_channelwise(rq, rwq, rs, rws, bias=b, out_fp16=fp16, threads=THREADS), fp16)
    return out, ref


def test_tiny_layer_with_bias(dev):
    out, ref = channelwise_case(dev, 16, 256, 512, bias=True, outliers=False)
    assert_gemm_close(out_values(out), ref, "16x256x512+bias")


@pytest.mark.parametrize("swap,mma_n,split", SCHEDULES)
def test_channelwise_every_schedule(dev, schedule, swap, mma_n, split):
    fq.fp8q_set_plan_override(swap, mma_n, split)
    for M in (1, 70, 300):
        out, ref = channelwise_case(dev, M, 392, 1040, seed=M, bias=True)
        assert_gemm_close(out_values(out), ref, f"sched {swap},{mma_n},{split} M={M}")


SPLIT_SCHEDULES = [s for s in SCHEDULES if s[2] > 1]
STREAM_K_SCHEDULES = [s for s in SCHEDULES if s[2] == 0]


def _flags(work: torch.Tensor, grid: int) -> np.ndarray:
    return work[work.numel() - 4 * grid:].view(torch.int32).cpu().numpy()


@pytest.mark.parametrize("bw", [False, True])
def test_stream_k_workspace_flags_and_repeats(dev, schedule, bw):
    """Stream-K through a caller's zero-filled workspace: the plan asks for
    grid * (512 * mma_n + 4) bytes; two calls in a row on different inputs
    both match the oracle, repeating a call gives identical bits, and every
    flag is back at zero after each call."""
    fq.fp8q_set_plan_override(1, 16, 0)
    M, N, K = 13, 1024, 2176          # 8 tiles x 17 K blocks = 136 pairs
    plan = fq.fp8q_gemm_plan(M, N, K, blockwise=bw)
    assert plan["stream_k"] == 1 and plan["split_k"] == 1
    grid = plan["grid"]
    need = fq.fp8q_workspace_bytes(M, N, K, bw)
    assert need == grid * (512 * 16 + 4)
    work = torch.zeros(need, dtype=torch.uint8, device=dev)
    for seed in (1, 2):
        if bw:
            out, ctx = blockwise_case(dev, M, N, K, seed=seed, bias=True, workspace=work)
            ref = blockwise_ref(ctx, M)
        else:
            out, ref = channelwise_case(dev, M, N, K, seed=seed, bias=True, workspace=work)
        assert_gemm_close(out_values(out), ref, f"stream-K seed {seed}")
        assert not _flags(work, grid).any(), "flags left set"
        again = (blockwise_case(dev, M, N, K, seed=seed, bias=True, workspace=work)[0] if bw else
                 channelwise_case(dev, M, N, K, seed=seed, bias=True, workspace=work)[0])
        assert torch.equal(out, again), "stream-K result not deterministic"


def test_stream_k_without_workspace_falls_back(dev, schedule):
    """A stream-K plan called without a workspace, or with one 4 bytes short
    (one flag), runs the tiles split along K instead: the two give identical
    bits, and both meet the oracle bar."""
    fq.fp8q_set_plan_override(1, 32, 0)
    for M in (1, 20):
        out, ref = channelwise_case(dev, M, 768, 3072, seed=M, workspace=None)
        assert_gemm_close(out_values(out), ref, f"stream-K fallback M={M}")
        need = fq.fp8q_workspace_bytes(M, 768, 3072)
        short = torch.zeros(need - 4, dtype=torch.uint8, device=dev)
        out_short, _ = channelwise_case(dev, M, 768, 3072, seed=M, workspace=short)
        assert torch.equal(out_short, out), "a short workspace did not fall back to the K-split schedule"


def test_stream_k_graph_replays(dev, schedule):
    """CUDA-graph replays of a stream-K GEMM (same workspace every replay)
    on inputs rewritten between replays: each replay matches the oracle, so
    each launch leaves the flags ready for the next."""
    fq.fp8q_set_plan_override(1, 16, 0)
    M, N, K = 16, 2048, 4096
    w = synthetic.weights(N, K, seed=5)
    wq, ws, rwq, rws = quant_both_per_token(w, dev)
    need = fq.fp8q_workspace_bytes(M, N, K)
    work = torch.zeros(need, dtype=torch.uint8, device=dev)
    xq = torch.empty((M, K), dtype=fq.E4M3, device=dev)
    xs = torch.empty((M,), dtype=torch.float32, device=dev)
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fq.fp8q_scaled_mm_channelwise(xq, wq, xs, ws, out=out, workspace=work)
    side.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        fq.fp8q_scaled_mm_channelwise(xq, wq, xs, ws, out=out, workspace=work)
    for seed in (11, 12, 13):
        x = synthetic.activations(M, K, seed=seed, outliers=True)
        q, s, rq, rs = quant_both_per_token(x, dev)
        xq.copy_(q)
        xs.copy_(s)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        ref = ref_values(oracle.gemm_channelwise(rq, rwq, rs, rws, threads=THREADS))
        assert_gemm_close(out_values(out), ref, f"graph replay seed {seed}")
    assert not _flags(work, fq.fp8q_gemm_plan(M, N, K)["grid"]).any()
    assert fq.fp8q_device_status() == fq.FP8Q_OK


def test_split_k_requests_no_workspace_by_default(dev, schedule):
    """Without FP8Q_WORKSPACE_EXCHANGE=1 the K-split partials are exchanged in
    distributed shared memory: no schedule asks for a workspace."""
    for swap, mma_n, split in SPLIT_SCHEDULES:
        fq.fp8q_set_plan_override(swap, mma_n, split)
        for bw in (False, True):
            assert fq.fp8q_workspace_bytes(300, 384, 1024, bw) == 0


def test_split_k_workspace_exchange_equals_dsmem_exchange(dev):
    """With FP8Q_WORKSPACE_EXCHANGE=1 (read at start-up, so in a child
    process): for every K-split schedule, the partial sums exchanged through
    the caller's global workspace (partial tiles of 128 x 128 floats or
    more) and through distributed shared memory are added in the same
    order, so the outputs are identical; a workspace one slot short is not
    used; smaller partial tiles ask for none; and the result matches the
    oracle (tests/ws_exchange_check.py)."""
    import os
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    r = subprocess.run([sys.executable, os.path.join(here, "ws_exchange_check.py")], capture_output=True, text=True,
                       timeout=900, env=dict(os.environ, FP8Q_WORKSPACE_EXCHANGE="1"))
    assert r.returncode == 0 and "workspace exchange ok" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]


@pytest.mark.parametrize("M", [1, 2, 5, 16, 33, 64, 100, 128, 129, 256, 300, 512])
def test_channelwise_default_plan(dev, M):
    out, ref = channelwise_case(dev, M, 384, 1024, seed=M)
    assert_gemm_close(out_values(out), ref, f"M={M}")


@pytest.mark.parametrize("M,N,K", [
    (2048, 2560, 512),    # 80 tile pairs: more than one pair per two SMs (persistent pairs)
    (1000, 768, 1040),    # 8 token tiles, ragged M and K
    (300, 512, 256),      # 3 token tiles: the last pair's second tile is empty
])
def test_channelwise_paired_tiles(dev, schedule, M, N, K):
    """Non-swapped tiles computed by CTA pairs with 2-CTA MMAs (256 tokens x
    256 columns per pair, each CTA staging half of the weight slice),
    compared on sampled outputs."""
    fq.fp8q_set_plan_override(0, 256, 1)
    plan = fq.fp8q_gemm_plan(M, N, K)
    assert plan["pair"] == 1 and plan["two_sm"] == 1
    x = synthetic.activations(M, K, seed=M + 1, outliers=True)
    w = synthetic.weights(N, K, seed=M + 1)
    b = synthetic.bias(N, seed=M + 1)
    xq, xs, rq, rs = quant_both_per_token(x, dev)
    wq, ws, rwq, rws = quant_both_per_token(w, dev)
    out = fq.fp8q_scaled_mm_channelwise(xq, wq, xs, ws, bias=b.to(dev))
    torch.cuda.synchronize()
    rng = np.random.default_rng(M)
    ms, ns = rng.integers(0, M, 20000), rng.integers(0, N, 20000)
    ms[:N] = M - 1                     # the whole last row (the last pair's ragged tile)
    ns[:N] = np.arange(N)
    ref = ref_values(oracle.gemm_channelwise_at(rq, rwq, rs, rws, ms, ns, bias=b))
    assert_gemm_close(out_values(out)[ms, ns], ref, f"paired {M}x{N}x{K}")
    assert fq.fp8q_device_status() == fq.FP8Q_OK


def test_channelwise_fp16_output(dev):
    out, ref = channelwise_case(dev, 40, 256, 512, bias=True, out_dtype=torch.float16)
    assert out.dtype == torch.float16
    assert_gemm_close(out_values(out), ref, "fp16")


def test_channelwise_strided_weight_and_output_canary(dev):
    M, N, K, ldb = 24, 256, 512, 640
    x = synthetic.activations(M, K, seed=11)
    wbig = synthetic.weights(N, ldb, seed=11)
    xq, xs, rq, rs = quant_both_per_token(x, dev)
    wq_full, ws = fq.fp8q_quant_per_token(wbig.to(dev)[:, :K].contiguous())
    wstore = torch.zeros((N, ldb), dtype=fq.E4M3, device=dev)
    wstore[:, :K] = wq_full
    out_buf = torch.full((M + 2, N), 7.0, dtype=torch.bfloat16, device=dev)
    fq.fp8q_scaled_mm_channelwise(xq, wstore[:, :K], xs, ws, out=out_buf[:M])
    torch.cuda.synchronize()
    ref = ref_values(oracle.gemm_channelwise(rq, u8(wq_full), rs, ws.cpu().numpy()))
    assert_gemm_close(out_values(out_buf[:M]), ref, "strided b")
    assert torch.all(out_buf[M:] == 7.0)


@pytest.mark.parametrize("mma_n", [32, 64, 128])
@pytest.mark.parametrize("K", [384, 640, 1024])
def test_channelwise_double_k_block_stages(dev, schedule, mma_n, K):
    """Non-swapped channelwise tiles over whole 128-wide K blocks with K not
    split take stages of two K blocks (one 3-D TMA box per operand); an odd
    number of K blocks leaves the last stage's second block zero-filled."""
    fq.fp8q_set_plan_override(0, mma_n, 1)
    for M in (1, 70, 300):
        out, ref = channelwise_case(dev, M, 392, K, seed=M + K, bias=True)
        assert_gemm_close(out_values(out), ref, f"noswap{mma_n} K={K} M={M}")


@pytest.mark.parametrize("mma_n", [32, 64, 128])
def test_channelwise_double_k_block_strided_weight(dev, schedule, mma_n):
    """The same stages with the weights' row stride above K (ldb = K + 128)
    and an output canary row."""
    fq.fp8q_set_plan_override(0, mma_n, 1)
    M, N, K, ldb = 200, 264, 640, 768
    x = synthetic.activations(M, K, seed=13)
    w = synthetic.weights(N, K, seed=13)
    xq, xs, rq, rs = quant_both_per_token(x, dev)
    wq, ws = fq.fp8q_quant_per_token(w.to(dev))
    wstore = torch.zeros((N, ldb), dtype=fq.E4M3, device=dev)
    wstore[:, :K] = wq
    wstore[:, K:].view(torch.uint8).fill_(0x7E)     # 448 past K: must never be read
    out_buf = torch.full((M + 1, N), 7.0, dtype=torch.bfloat16, device=dev)
    fq.fp8q_scaled_mm_channelwise(xq, wstore[:, :K], xs, ws, out=out_buf[:M])
    torch.cuda.synchronize()
    ref = ref_values(oracle.gemm_channelwise(rq, u8(wq), rs, ws.cpu().numpy()))
    assert_gemm_close(out_values(out_buf[:M]), ref, f"noswap{mma_n} strided b")
    assert torch.all(out_buf[M:] == 7.0)


def blockwise_case(dev, M, N, K, seed=0, bias=False, outliers=True, garbage_padding=False, workspace="auto"):
    x = synthetic.activations(M, K, seed=seed, outliers=outliers)
    w = synthetic.weights(N, K, seed=seed)
    b = synthetic.bias(N, seed=seed) if bias else None
    fills = dict(xq_fill=0x7F, xs_fill=float("nan")) if garbage_padding else {}
    xq, xs, rq, rs = quant_both_group(x, dev, 128, **fills)
    wq, ws = fq.fp8q_quant_weight_block128(w.to(dev))
    torch.cuda.synchronize()
    rwq, rws = oracle.quant_weight_blocks(w, 128, 128)
    assert np.array_equal(u8(wq), rwq) and np.array_equal(ws.cpu().numpy(), rws)
    out = fq.fp8q_scaled_mm_blockwise(xq, wq, xs, ws, M=M, bias=None if b is None else b.to(dev),
                                      workspace=workspace)
    torch.cuda.synchronize()
    return out, (x, w, b, rq, rs, rwq, rws)


def blockwise_ref(ctx, M, threads=THREADS):
    x, w, b, rq, rs, rwq, rws = ctx
    return ref_values(oracle.gemm_blockwise(rq, rwq, rs, rws, M, bias=b, threads=threads))


@pytest.mark.parametrize("swap,mma_n,split", SCHEDULES)
def test_blockwise_every_schedule(dev, schedule, swap, mma_n, split):
    fq.fp8q_set_plan_override(swap, mma_n, split)
    for M in (3, 70, 260):
        out, ctx = blockwise_case(dev, M, 384, 1024, seed=M, bias=True)
        assert_gemm_close(out_values(out), blockwise_ref(ctx, M), f"sched {swap},{mma_n},{split} M={M}")


def test_blockwise_persistent_tiles(dev, schedule):
    """Non-swapped blockwise tiles are single CTAs (no pairs): each CTA runs
    its own MMAs and loads its whole 256-row weight slice.  9 x 24 tiles on
    a persistent grid of one CTA per SM: several tiles per CTA."""
    fq.fp8q_set_plan_override(0, 256, 1)
    M, N, K = 1100, 6144, 1024
    plan = fq.fp8q_gemm_plan(M, N, K, blockwise=True)
    assert plan["pair"] == 0 and plan["two_sm"] == 0 and plan["persistent"] == 1
    out, ctx = blockwise_case(dev, M, N, K, seed=21, bias=True)
    _, _, b, rq, rs, rwq, rws = ctx
    rng = np.random.default_rng(21)
    ms, ns = rng.integers(0, M, 20000), rng.integers(0, N, 20000)
    ref = ref_values(oracle.gemm_blockwise_at(rq, rwq, rs, rws, ms, ns, bias=b))
    assert_gemm_close(out_values(out)[ms, ns], ref, "blockwise persistent")


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 7, 13, 16, 31, 64, 256])
def test_blockwise_decode_layer_full_size(dev, M):
    """The row-padded decode layer: N = 4096, K = 7168, every M of the
    row-padding page's test, padding rows filled with NaN codes and NaN
    scales (they must not reach the output)."""
    out, ctx = blockwise_case(dev, M, 4096, 7168, seed=M, garbage_padding=True)
    got = out_values(out)
    assert got.shape == (M, 4096)
    if M <= 16:
        assert_gemm_close(got, blockwise_ref(ctx, M), f"M={M}")
    else:
        rng = np.random.default_rng(M)
        ms, ns = rng.integers(0, M, 4096), rng.integers(0, 4096, 4096)
        _, _, b, rq, rs, rwq, rws = ctx
        ref = ref_values(oracle.gemm_blockwise_at(rq, rwq, rs, rws, ms, ns, bias=b))
        assert_gemm_close(got[ms, ns], ref, f"M={M} sampled")


def test_blockwise_padding_rows_do_not_matter(dev):
    M = 13
    out1, _ = blockwise_case(dev, M, 512, 1024, seed=9, garbage_padding=True)
    out2, _ = blockwise_case(dev, M, 512, 1024, seed=9, garbage_padding=False)
    assert torch.equal(out1, out2)


def test_linear_compositions(dev):
    M, N, K = 37, 256, 1024
    x = synthetic.activations(M, K, seed=4, outliers=True)
    w = synthetic.weights(N, K, seed=4)
    b = synthetic.bias(N, seed=4)
    wq, ws = fq.fp8q_quant_per_token(w.to(dev))
    out = fq.fp8q_linear_channelwise(x.to(dev), wq, ws, bias=b.to(dev))
    torch.cuda.synchronize()
    rq, rs = oracle.quant_per_token(x)
    ref = ref_values(oracle.gemm_channelwise(rq, u8(wq), rs, ws.cpu().numpy(), bias=b))
    assert_gemm_close(out_values(out), ref, "linear channelwise")
    wq, ws = fq.fp8q_quant_weight_block128(w.to(dev))
    out = fq.fp8q_linear_blockwise(x.to(dev), wq, ws, bias=b.to(dev))
    torch.cuda.synchronize()
    assert out.shape == (M, N)
    rq, rs = oracle.quant_group_row_padded(x, 128)
    ref = ref_values(oracle.gemm_blockwise(rq, u8(wq), rs, ws.cpu().numpy(), M, bias=b))
    assert_gemm_close(out_values(out), ref, "linear blockwise")


def test_m0_and_status_word(dev):
    a = torch.empty((0, 256), dtype=fq.E4M3, device=dev)
    w = torch.zeros((128, 256), dtype=fq.E4M3, device=dev)
    s = torch.ones(128, dtype=torch.float32, device=dev)
    out = fq.fp8q_scaled_mm_channelwise(a, w, torch.empty(0, device=dev), s)
    assert out.shape == (0, 128)
    assert fq.fp8q_device_status() == fq.FP8Q_OK


@pytest.mark.parametrize("order", ["weights_then_gemm", "weights_act_gemm"])
def test_weights_rewritten_right_before_the_gemm(dev, order):
    """The GEMM streams weights before waiting for its predecessor; a weight
    buffer rewritten by the immediately preceding (or the one before that)
    launch on the stream must still be read fresh.  Each iteration writes
    new values into the SAME weight buffer with no synchronization."""
    M, N, K = 8, 512, 2048
    x = synthetic.activations(M, K, seed=50)
    xd = x.to(dev)
    wq = torch.empty((N, K), dtype=fq.E4M3, device=dev)
    ws = torch.empty((N,), dtype=torch.float32, device=dev)
    xq = torch.empty((M, K), dtype=fq.E4M3, device=dev)
    xs = torch.empty((M,), dtype=torch.float32, device=dev)
    ws_cpu, outs = [], []
    for i in range(4):
        w = synthetic.weights(N, K, seed=100 + i).to(dev)
        torch.cuda.synchronize()
        if order == "weights_then_gemm":
            fq.fp8q_quant_per_token(xd, xq=xq, x_scale=xs)
            fq.fp8q_quant_per_token(w, xq=wq, x_scale=ws)
        else:
            fq.fp8q_quant_per_token(w, xq=wq, x_scale=ws)
            fq.fp8q_quant_per_token(xd, xq=xq, x_scale=xs)
        outs.append(fq.fp8q_scaled_mm_channelwise(xq, wq, xs, ws))
        ws_cpu.append(w.cpu())
    torch.cuda.synchronize()
    rq, rs = oracle.quant_per_token(x)
    for i in range(4):
        rwq, rws = oracle.quant_weight_per_channel(ws_cpu[i])
        ref = ref_values(oracle.gemm_channelwise(rq, rwq, rs, rws, threads=THREADS))
        assert_gemm_close(out_values(outs[i]), ref, f"iteration {i}")
