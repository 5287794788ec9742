"""GPU parity at the full sizes of the benchmark workloads, on the planner's
own schedules (no override), through the C ABI.

Shapes (the Qwen3-8B-shaped linears of the "Tune FP8 GEMM Triton tiles on
L40S" page, Motivation; the blockwise prefill layers of the row-padding
page, Implementation breakdown):
  channelwise o_proj 4096x4096 at M in {512, 2048, 8192};
  channelwise qkv 6144x4096, down 4096x12288, gate_up 24576x4096 at
  M in {128, 512, 2048, 8192}, and gate_up at M in {1, 16} (the stream-K
  schedule, with the zero-filled workspace the binding allocates);
  blockwise 24576x3072 and 3072x12288 at M = 8192.

Per case:
  * the activation quantization is compared byte for byte with the oracle
    over the whole tensor (codes and scales bit-exact, as the row-padding
    page's Risks and impact section requires of the quantizer: max_abs_diff
    of 0), so per-token quantization is checked bit-exact at 8192 x 4096 and
    8192 x 12288, and group quantization at 8192 x 3072 and 8192 x 12288;
  * the GEMM output is compared with the oracle's exact result on 20,000
    seeded random positions plus one whole row and one whole column (the
    last ones, where tiles are ragged) under the spec bar
    |gpu - ref| <= 1e-2 * (|ref| + 1);
  * and under two tighter diagnostic checks:
      - every position: |gpu - ref| <= 2 bf16 ulp of max(|gpu|, |ref|)
        + K * 2^-24 * S, where S = sa * sw * sum_k |a_k w_k| (blockwise: the
        sum over K blocks of each block's scales times its sum of absolute
        products), evaluated exactly by the oracle on the codes with their
        sign bits cleared.  K * 2^-24 * S bounds the error of any fp32
        summation order of the K exact products; the 2 ulp cover the output
        rounding on both sides.  A dropped or doubled K block or a misplaced
        tile breaks it by many ulp on most positions;
      - at most 5 % of the positions differ at all from the exact result
        rounded once to bf16.  An fp32 accumulation moves only the outputs
        whose exact value lies within its small error of a rounding
        midpoint (well under 1 % here), while a scale wrong by a fraction
        of an ulp (0.3 %, which the 1e-2 bar cannot see) moves most of them.
    The observed maximum error (in bf16 ulp and as a fraction of the
    accumulation term) and the fraction of moved outputs are printed."""
import numpy as np
import pytest
import torch

import fp8_w8a8_quantized_token_gb300 as fq
import oracle
import synthetic
from gpu_util import THREADS, assert_gemm_close, ref_values, u8

pytestmark = pytest.mark.gpu

SAMPLES = 20000

CHANNELWISE = [
    ("o_proj", 4096, 4096, 512), ("o_proj", 4096, 4096, 2048), ("o_proj", 4096, 4096, 8192),
    ("qkv", 6144, 4096, 128), ("qkv", 6144, 4096, 512), ("qkv", 6144, 4096, 2048), ("qkv", 6144, 4096, 8192),
    ("down", 4096, 12288, 128), ("down", 4096, 12288, 512), ("down", 4096, 12288, 2048),
    ("down", 4096, 12288, 8192),
    ("gate_up", 24576, 4096, 1), ("gate_up", 24576, 4096, 16),     # stream-K rows of the table
    ("gate_up", 24576, 4096, 128), ("gate_up", 24576, 4096, 512), ("gate_up", 24576, 4096, 2048),
    ("gate_up", 24576, 4096, 8192),
]
BLOCKWISE = [("blk_24576x3072", 24576, 3072, 8192), ("blk_3072x12288", 3072, 12288, 8192)]


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    d = torch.device("cuda", 0)
    torch.cuda.set_device(d)
    fq.fp8q_set_plan_override(-1)
    return d


_cache = {}


def cached(key, make):
    if key not in _cache:
        _cache[key] = make()
    return _cache[key]


def activations(K):
    """The largest M's activations for this K (smaller M take the first rows:
    the generator is counter-based, so those are the same values)."""
    return cached(("x", K), lambda: synthetic.activations(8192, K, outliers=True))


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    _, e = np.frexp(np.abs(v))
    return np.where(v == 0, 2.0 ** -133, np.ldexp(1.0, np.maximum(e - 8, -133)))


def positions(M, N, seed):
    rng = np.random.default_rng(seed)
    ms = np.concatenate([rng.integers(0, M, SAMPLES), np.full(N, M - 1), np.arange(M)])
    ns = np.concatenate([rng.integers(0, N, SAMPLES), np.arange(N), np.full(M, N - 1)])
    return ms, ns


def check_tight(got, ref, S, K, what):
    err = np.abs(got - ref)
    ulp = bf16_ulp(np.maximum(np.abs(got), np.abs(ref)))
    acc = K * 2.0 ** -24 * S * (1 + 2.0 ** -7)   # S is itself bf16-rounded
    bound = 2 * ulp + acc
    ratio_ulp = float(np.max(err / ulp))
    ratio_acc = float(np.max(np.where(acc > 0, np.maximum(err - 2 * ulp, 0) / np.maximum(acc, 1e-300), 0)))
    print(f"{what}: max |err| {float(err.max()):.3e}, max err/ulp {ratio_ulp:.2f}, "
          f"outputs not equal to the exact result rounded: {float(np.mean(err > 0)):.4f}, "
          f"max (err - 2ulp)/accumulation term {ratio_acc:.3f}")
    moved = float(np.mean(err > 0))
    assert moved <= 0.05, f"{what}: {moved:.3f} of the outputs differ from the exact result rounded"
    bad = ~(err <= bound)
    if bad.any():
        i = int(np.argmax(bad))
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside the diagnostic bound, e.g. "
                             f"got {got[i]!r} ref {ref[i]!r} bound {bound[i]!r}")


def gathered(out: torch.Tensor, ms, ns) -> np.ndarray:
    idx_m = torch.as_tensor(ms, device=out.device)
    idx_n = torch.as_tensor(ns, device=out.device)
    return out[idx_m, idx_n].float().cpu().numpy().astype(np.float64)


def channelwise_weights(dev, N, K):
    def make():
        w = synthetic.weights(N, K)
        wq, ws = fq.fp8q_quant_per_token(w.to(dev))
        torch.cuda.synchronize()
        rwq, rws = oracle.quant_weight_per_channel(w)
        assert np.array_equal(u8(wq), rwq), "weight codes differ"
        assert np.array_equal(ws.cpu().numpy(), rws), "weight scales differ"
        return wq, ws, rwq, rws
    return cached(("wc", N, K), make)


@pytest.mark.parametrize("label,N,K,M", CHANNELWISE)
def test_channelwise_full_size_planner_schedule(dev, label, N, K, M):
    wq, ws, rwq, rws = channelwise_weights(dev, N, K)
    x = activations(K)[:M]
    xq, xs = fq.fp8q_quant_per_token(x.to(dev))
    plan = fq.fp8q_gemm_plan(M, N, K)
    out = fq.fp8q_scaled_mm_channelwise(xq, wq, xs, ws)
    torch.cuda.synchronize()
    assert fq.fp8q_device_status() == fq.FP8Q_OK
    rq, rs = oracle.quant_per_token(x, threads=THREADS)
    assert np.array_equal(u8(xq), rq), f"per-token codes differ at {M}x{K}"
    assert np.array_equal(xs.cpu().numpy(), rs), f"per-token scales differ at {M}x{K}"
    ms, ns = positions(M, N, seed=M + N)
    ref = ref_values(oracle.gemm_channelwise_at(rq, rwq, rs, rws, ms, ns))
    got = gathered(out, ms, ns)
    split = "streamK" if plan.get("stream_k") else plan["split_k"]
    sched = f"{'swap' if plan['swap_ab'] else 'noswap'}{plan['mma_n']}x{split}"
    what = f"{label} M={M} ({sched})"
    assert_gemm_close(got, ref, what)
    S = ref_values(oracle.gemm_channelwise_at(rq & 0x7F, rwq & 0x7F, rs, rws, ms, ns))
    check_tight(got, ref, S, K, what)


@pytest.mark.parametrize("label,N,K,M", BLOCKWISE)
def test_blockwise_full_size_planner_schedule(dev, label, N, K, M):
    w = synthetic.weights(N, K)
    wq, ws = fq.fp8q_quant_weight_block128(w.to(dev))
    torch.cuda.synchronize()
    rwq, rws = oracle.quant_weight_blocks(w, 128, 128)
    del w
    assert np.array_equal(u8(wq), rwq) and np.array_equal(ws.cpu().numpy(), rws)
    x = activations(K)[:M]
    xq, xsv = fq.fp8q_quant_per_token_group_row_padded(x.to(dev), 128)
    plan = fq.fp8q_gemm_plan(M, N, K, blockwise=True)
    out = fq.fp8q_scaled_mm_blockwise(xq, wq, xsv, ws, M=M)
    torch.cuda.synchronize()
    assert fq.fp8q_device_status() == fq.FP8Q_OK
    rq, rs = oracle.quant_group_row_padded(x, 128, threads=THREADS)
    assert np.array_equal(u8(xq)[:M], rq[:M]), f"group codes differ at {M}x{K}"
    assert np.array_equal(xsv.transpose(0, 1).cpu().numpy()[:, :M], rs[:, :M]), f"group scales differ at {M}x{K}"
    ms, ns = positions(M, N, seed=M + N + 1)
    ref = ref_values(oracle.gemm_blockwise_at(rq, rwq, rs, rws, ms, ns))
    got = gathered(out, ms, ns)
    sched = f"{'swap' if plan['swap_ab'] else 'noswap'}{plan['mma_n']}x{plan['split_k']}"
    what = f"{label} M={M} ({sched})"
    assert_gemm_close(got, ref, what)
    S = ref_values(oracle.gemm_blockwise_at(rq & 0x7F, rwq & 0x7F, rs, rws, ms, ns))
    check_tight(got, ref, S, K, what)
