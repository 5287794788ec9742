"""Helpers shared by the GPU parity tests: running both sides on the same
seeded inputs and comparing them."""
from __future__ import annotations

import os

import numpy as np
import torch

import fp8_w8a8_quantized_token_gb300 as fq
import oracle

THREADS = max(1, min(16, os.cpu_count() or 1))
RTOL = 1e-2  # the GEMM bar: |gpu - ref| <= 1e-2 * (|ref| + 1)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.uint8).cpu().numpy()


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def out_values(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def ref_values(bits: np.ndarray, out_fp16: bool = False) -> np.ndarray:
    return oracle.f16_bits_to_float(bits) if out_fp16 else oracle.bf16_bits_to_float(bits)


def assert_gemm_close(got: np.ndarray, ref: np.ndarray, what: str = "gemm"):
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = np.abs(got - ref)
    tol = RTOL * (np.abs(ref) + 1.0)
    bad = ~(err <= tol)  # NaN counts as bad
    if bad.any():
        idx = np.argwhere(bad)[:8]
        details = [(tuple(int(v) for v in i), float(got[tuple(i)]), float(ref[tuple(i)])) for i in idx]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance, e.g. {details}")


def quant_both_per_token(x_cpu: torch.Tensor, dev):
    """Quantize on the GPU and in the oracle; assert bit-exact; return both."""
    xq, xs = fq.fp8q_quant_per_token(x_cpu.to(dev))
    torch.cuda.synchronize()
    rq, rs = oracle.quant_per_token(x_cpu, threads=THREADS)
    gq, gs = u8(xq), f32(xs)
    if not np.array_equal(gq, rq):
        bad = np.argwhere(gq != rq)[:5]
        raise AssertionError(f"per-token codes differ at {bad.tolist()}: gpu {gq[tuple(bad[0])]} "
                             f"oracle {rq[tuple(bad[0])]}")
    assert np.array_equal(gs, rs), "per-token scales differ"
    return xq, xs, rq, rs


def quant_both_group(x_cpu: torch.Tensor, dev, group: int = 128, xq_fill: int | None = None,
                     xs_fill: float | None = None):
    M, K = x_cpu.shape
    m_pad = fq.ceil_align(M, 4)
    xq = torch.empty((m_pad, K), dtype=fq.E4M3, device=dev)
    xs = torch.empty((K // group, m_pad), dtype=torch.float32, device=dev)
    if xq_fill is not None:
        xq.view(torch.uint8).fill_(xq_fill)
    if xs_fill is not None:
        xs.fill_(xs_fill)
    xq, xsv = fq.fp8q_quant_per_token_group_row_padded(x_cpu.to(dev), group, xq=xq, x_scale_storage=xs)
    torch.cuda.synchronize()
    rq, rs = oracle.quant_group_row_padded(x_cpu, group, threads=THREADS)
    gq, gs = u8(xq), xs.cpu().numpy()
    assert np.array_equal(gq[:M], rq[:M]), "group codes differ"
    assert np.array_equal(gs[:, :M], rs[:, :M]), "group scales differ"
    return xq, xs, rq, rs
