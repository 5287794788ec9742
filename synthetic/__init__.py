"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This module draws random numbers and nothing else: it holds none of the
quantization or GEMM arithmetic.  Both the CPU oracle (``oracle/``) and the
CUDA library are fed from the tensors produced here, so that the two sides of
every parity test see bit-identical inputs.

Generator
---------
A counter-based generator built on the published splitmix64 finaliser
(Steele, Lea, Flood, "Fast splittable pseudorandom number generators",
OOPSLA 2014):

    z1 = (z  ^ (z  >> 30)) * 0xBF58476D1CE4E5B9
    z2 = (z1 ^ (z1 >> 27)) * 0x94D049BB133111EB
    mix64(z) = z2 ^ (z2 >> 31)              (all arithmetic mod 2^64)

The 64-bit word for counter ``c`` of stream ``(seed, tensor_id)`` is
``mix64(key + (c + 1) * 0x9E3779B97F4A7C15)`` with
``key = mix64(seed * 0x9E3779B97F4A7C15 ^ (tensor_id << 32))``.  A uniform in
(0, 1] takes the top 53 bits.  Element ``i`` of a normal tensor uses counters
``2i`` and ``2i+1`` through the Box–Muller transform
``sqrt(-2 ln u1) * cos(2 pi u2)``, computed in float64, scaled by ``std``,
then rounded to float32 and to bfloat16 (each round-to-nearest-even).

Workload recipe (values follow the FP8 W8A8 linear-layer pages: activations
~N(0,1), weights ~N(0,0.02), bias ~N(0,0.1); "outlier" activation channels are
``round(0.01*K)`` distinct columns picked by the generator and multiplied by
20 before rounding).
"""
from __future__ import annotations

import numpy as np
import torch

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_C1 = np.uint64(0xBF58476D1CE4E5B9)
_C2 = np.uint64(0x94D049BB133111EB)

# Fixed tensor ids so every consumer draws the same stream for the same role.
TID_ACT = 1
TID_WEIGHT = 2
TID_BIAS = 3
TID_OUTLIER = 4

_CHUNK = 1 << 22


def _mix64(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _C1
        z = (z ^ (z >> np.uint64(27))) * _C2
        return z ^ (z >> np.uint64(31))


def _key(seed: int, tensor_id: int) -> np.uint64:
    with np.errstate(over="ignore"):
        k = np.array([np.uint64(seed) * _GAMMA ^ (np.uint64(tensor_id) << np.uint64(32))],
                     dtype=np.uint64)
    return _mix64(k)[0]


def words(seed: int, tensor_id: int, start: int, count: int) -> np.ndarray:
    """Raw 64-bit words for counters [start, start+count) of one stream."""
    key = _key(seed, tensor_id)
    c = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(key + c * _GAMMA)


def uniform(seed: int, tensor_id: int, start: int, count: int) -> np.ndarray:
    """Uniforms in (0, 1] from the top 53 bits of each word (float64)."""
    w = words(seed, tensor_id, start, count)
    return ((w >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def normal(seed: int, tensor_id: int, count: int) -> np.ndarray:
    """``count`` standard normals (float64), element i from counters 2i, 2i+1."""
    out = np.empty(count, dtype=np.float64)
    for s in range(0, count, _CHUNK):
        n = min(_CHUNK, count - s)
        u = uniform(seed, tensor_id, 2 * s, 2 * n).reshape(n, 2)
        out[s:s + n] = np.sqrt(-2.0 * np.log(u[:, 0])) * np.cos(2.0 * np.pi * u[:, 1])
    return out


def outlier_columns(K: int, seed: int = 0, fraction: float = 0.01) -> np.ndarray:
    """``round(fraction*K)`` distinct column indices, sorted, drawn by the generator."""
    n = int(round(fraction * K))
    if n == 0:
        return np.zeros(0, dtype=np.int64)
    keys = words(seed, TID_OUTLIER, 0, K)
    return np.sort(np.argsort(keys, kind="stable")[:n]).astype(np.int64)


def bf16_normal(shape, std: float = 1.0, seed: int = 0, tensor_id: int = TID_ACT,
                outlier_cols: np.ndarray | None = None, outlier_scale: float = 20.0) -> torch.Tensor:
    """A CPU bfloat16 tensor of ``shape`` with N(0, std^2) entries (row-major)."""
    shape = tuple(int(s) for s in shape)
    count = int(np.prod(shape)) if shape else 1
    v = normal(seed, tensor_id, count) * std
    if outlier_cols is not None and len(outlier_cols) and count:
        v = v.reshape(-1, shape[-1])
        v[:, outlier_cols] *= outlier_scale
        v = v.reshape(-1)
    t = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16)
    return t.reshape(shape)


def activations(M: int, K: int, seed: int = 0, outliers: bool = False) -> torch.Tensor:
    """bf16 [M, K] activations ~N(0,1), optionally with 1% outlier columns x20."""
    cols = outlier_columns(K, seed) if outliers else None
    return bf16_normal((M, K), 1.0, seed, TID_ACT, cols)


def weights(N: int, K: int, seed: int = 0) -> torch.Tensor:
    """bf16 weights ~N(0, 0.02^2), stored [N, K] row-major (K contiguous)."""
    return bf16_normal((N, K), 0.02, seed, TID_WEIGHT)


def bias(N: int, seed: int = 0) -> torch.Tensor:
    """bf16 bias [N] ~N(0, 0.1^2)."""
    return bf16_normal((N,), 0.1, seed, TID_BIAS)
