"""CPU oracle for the FP8 W8A8 linear layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never touches it, and
it never touches the CUDA library: the two share no code.

The arithmetic lives in ``fp8q_oracle.c`` (plain single-threaded C, exact
double GEMM, fp32 quantization decisions).  This module builds it with gcc,
loads it with ctypes and wraps each function for numpy / torch-CPU arrays.
Every wrapper takes and returns host arrays; "bf16" data is passed as its
16-bit pattern.

Parity pins: the codec, both quantizers, both GEMMs and the bf16/fp16
output rounding are pinned by ``tests/test_oracle_*.py`` against closed forms,
library routines (torch's float8_e4m3fn cast, numpy float64 matmul, Python
Fractions), brute force and the values printed under ``tests/golden/``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8q_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``fp8q_oracle.c`` into ``liboracle.so`` next to it."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            P, I64, F32, INT = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int
            L.fp8q_oracle_e4m3_decode.restype = ctypes.c_double
            L.fp8q_oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.fp8q_oracle_e4m3_encode.restype = ctypes.c_uint8
            L.fp8q_oracle_e4m3_encode.argtypes = [F32]
            L.fp8q_oracle_e4m3_encode_array.argtypes = [P, P, I64]
            L.fp8q_oracle_e4m3_decode_array.argtypes = [P, P, I64]
            L.fp8q_oracle_f64_to_bf16.restype = ctypes.c_uint16
            L.fp8q_oracle_f64_to_bf16.argtypes = [ctypes.c_double]
            L.fp8q_oracle_f64_to_f16.restype = ctypes.c_uint16
            L.fp8q_oracle_f64_to_f16.argtypes = [ctypes.c_double]
            L.fp8q_oracle_quant_per_token.argtypes = [P, I64, I64, F32, P, P, I64, I64]
            L.fp8q_oracle_quant_group_row_padded.argtypes = [P, I64, I64, I64, F32, I64, P, P, I64, I64]
            L.fp8q_oracle_quant_weight_blocks.argtypes = [P, I64, I64, I64, I64, I64, F32, P, P]
            L.fp8q_oracle_quant_static.argtypes = [P, I64, I64, F32, P, I64, I64]
            L.fp8q_oracle_quant_group_row_padded_ex.argtypes = [P, I64, I64, I64, F32, INT, INT, I64, P, P, I64, I64]
            L.fp8q_oracle_exp_f32_array.argtypes = [P, P, I64]
            L.fp8q_oracle_silu_mul_array.argtypes = [P, P, P, I64]
            L.fp8q_oracle_pow2_ceil_array.argtypes = [P, P, I64]
            L.fp8q_oracle_gemm_channelwise.argtypes = [P, I64, P, I64, P, P, P, I64, I64, INT, P, I64, P, I64, I64]
            L.fp8q_oracle_gemm_blockwise.argtypes = [P, I64, P, I64, P, I64, P, P, I64, I64, INT, P, I64, P, I64, I64]
            L.fp8q_oracle_gemm_w8a16.argtypes = [P, I64, P, I64, P, P, I64, I64, INT, P, I64, P, I64, I64]
            L.fp8q_oracle_gemm_channelwise_at.argtypes = [P, I64, P, I64, P, P, P, I64, INT, P, P, I64, P]
            L.fp8q_oracle_gemm_blockwise_at.argtypes = [P, I64, P, I64, P, I64, P, P, I64, INT, P, P, I64, P]
            _lib = L
    return _lib


# --------------------------------------------------------------------------
# array helpers
# --------------------------------------------------------------------------

def _bits16(x) -> np.ndarray:
    """bf16 tensor / uint16 array -> C-contiguous uint16 numpy array."""
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().contiguous()
        if x.dtype in (torch.bfloat16, torch.float16):
            x = x.view(torch.int16)
        return x.numpy().view(np.uint16)
    return np.ascontiguousarray(x, dtype=np.uint16)


def _u8(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().contiguous()
        if x.dtype != torch.uint8:
            x = x.view(torch.uint8)
        return x.numpy()
    return np.ascontiguousarray(x, dtype=np.uint8)


def _f32(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        return x.detach().cpu().contiguous().numpy().astype(np.float32, copy=False)
    return np.ascontiguousarray(x, dtype=np.float32)


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _row_chunks(M: int, threads: int):
    threads = max(1, min(threads, M))
    step = (M + threads - 1) // threads
    return [(r, min(M, r + step)) for r in range(0, M, step)]


def _run_rows(fn, M: int, threads: int):
    """Run fn(r0, r1) over row ranges; ctypes releases the GIL per call, so
    threads > 1 splits rows across host cores (the per-row code is unchanged)."""
    chunks = _row_chunks(M, threads)
    if len(chunks) <= 1:
        for r0, r1 in chunks:
            fn(r0, r1)
        return
    with ThreadPoolExecutor(len(chunks)) as ex:
        list(ex.map(lambda c: fn(*c), chunks))


# --------------------------------------------------------------------------
# codec
# --------------------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    c = _u8(codes).reshape(-1)
    out = np.empty(c.size, dtype=np.float64)
    lib().fp8q_oracle_e4m3_decode_array(_ptr(c), _ptr(out), c.size)
    return out


def e4m3_encode(values) -> np.ndarray:
    v = np.ascontiguousarray(values, dtype=np.float32).reshape(-1)
    out = np.empty(v.size, dtype=np.uint8)
    lib().fp8q_oracle_e4m3_encode_array(_ptr(v), _ptr(out), v.size)
    return out


def f64_to_bf16_bits(y: float) -> int:
    return int(lib().fp8q_oracle_f64_to_bf16(float(y)))


def f64_to_f16_bits(y: float) -> int:
    return int(lib().fp8q_oracle_f64_to_f16(float(y)))


# --------------------------------------------------------------------------
# quantization
# --------------------------------------------------------------------------

def quant_per_token(x, eps: float = 1e-10, threads: int = 1):
    """bf16 [M, K] -> (uint8 codes [M, K], fp32 scales [M])."""
    xb = _bits16(x)
    M, K = xb.shape
    xq = np.zeros((M, K), dtype=np.uint8)
    xs = np.zeros(M, dtype=np.float32)
    L = lib()
    _run_rows(lambda r0, r1: L.fp8q_oracle_quant_per_token(_ptr(xb), K, K, eps, _ptr(xq), _ptr(xs), r0, r1),
              M, threads)
    return xq, xs


def quant_group_row_padded(x, group_size: int = 128, eps: float = 1e-10, row_alignment: int = 4,
                           xq_init: int = 0, xs_init: float = 0.0, threads: int = 1):
    """bf16 [M, K] -> (uint8 x_q [m_pad, K], fp32 x_s storage [K/g, m_pad]).

    Rows >= M of both buffers keep their initial fill (``xq_init``, ``xs_init``):
    the quantizer never writes them."""
    xb = _bits16(x)
    M, K = xb.shape
    assert K % group_size == 0
    m_pad = (M + row_alignment - 1) // row_alignment * row_alignment
    xq = np.full((m_pad, K), xq_init, dtype=np.uint8)
    xs = np.full((K // group_size, m_pad), xs_init, dtype=np.float32)
    L = lib()
    _run_rows(lambda r0, r1: L.fp8q_oracle_quant_group_row_padded(
        _ptr(xb), K, K, group_size, eps, m_pad, _ptr(xq), _ptr(xs), r0, r1), M, threads)
    return xq, xs


def quant_group_row_padded_ex(x, group_size: int = 128, eps: float = 1e-10, row_alignment: int = 4,
                              scale_ue8m0: bool = False, fuse_silu_and_mul: bool = False,
                              xq_init: int = 0, xs_init: float = 0.0, threads: int = 1):
    """The group quantizer with its options.  fuse_silu_and_mul: x is bf16
    [M, 2K] and the quantized [M, K] values are silu(x[:, :K]) * x[:, K:] in
    fp32; scale_ue8m0: scales rounded up to powers of two.  Returns (uint8
    x_q [m_pad, K], fp32 x_s storage [K/g, m_pad])."""
    xb = _bits16(x)
    M, W = xb.shape
    K = W // 2 if fuse_silu_and_mul else W
    assert K % group_size == 0 and (not fuse_silu_and_mul or W == 2 * K)
    m_pad = (M + row_alignment - 1) // row_alignment * row_alignment
    xq = np.full((m_pad, K), xq_init, dtype=np.uint8)
    xs = np.full((K // group_size, m_pad), xs_init, dtype=np.float32)
    L = lib()
    _run_rows(lambda r0, r1: L.fp8q_oracle_quant_group_row_padded_ex(
        _ptr(xb), K, W, group_size, eps, int(scale_ue8m0), int(fuse_silu_and_mul), m_pad, _ptr(xq), _ptr(xs),
        r0, r1), M, threads)
    return xq, xs


def quant_static(x, scale: float, threads: int = 1):
    """Static per-tensor quantization: bf16 [M, K] and one fp32 scale ->
    uint8 codes [M, K]."""
    xb = _bits16(x)
    M, K = xb.shape
    xq = np.zeros((M, K), dtype=np.uint8)
    L = lib()
    s = float(np.float32(scale))
    _run_rows(lambda r0, r1: L.fp8q_oracle_quant_static(_ptr(xb), K, K, s, _ptr(xq), r0, r1), M, threads)
    return xq


def exp_f32(t) -> np.ndarray:
    """The quantizer's fully specified fp32 exp (elementwise)."""
    t = np.ascontiguousarray(t, dtype=np.float32)
    out = np.empty_like(t)
    lib().fp8q_oracle_exp_f32_array(_ptr(t), _ptr(out), t.size)
    return out


def silu_mul(a, b) -> np.ndarray:
    """silu(a) * b in fp32, as the fused group quantizer computes it."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    b = np.ascontiguousarray(b, dtype=np.float32)
    out = np.empty_like(a)
    lib().fp8q_oracle_silu_mul_array(_ptr(a), _ptr(b), _ptr(out), a.size)
    return out


def pow2_ceil(s) -> np.ndarray:
    """fp32 scales rounded up to powers of two (UE8M0 scales)."""
    s = np.ascontiguousarray(s, dtype=np.float32)
    out = np.empty_like(s)
    lib().fp8q_oracle_pow2_ceil_array(_ptr(s), _ptr(out), s.size)
    return out


def quant_weight_blocks(w, block_n: int, block_k: int, eps: float = 1e-10):
    """bf16 w [N, K] -> (uint8 [N, K], fp32 scales [ceil(N/bn), ceil(K/bk)])."""
    wb = _bits16(w)
    N, K = wb.shape
    nb, kb = -(-N // block_n), -(-K // block_k)
    wq = np.zeros((N, K), dtype=np.uint8)
    ws = np.zeros((nb, kb), dtype=np.float32)
    lib().fp8q_oracle_quant_weight_blocks(_ptr(wb), N, K, K, block_n, block_k, eps, _ptr(wq), _ptr(ws))
    return wq, ws


def quant_weight_per_channel(w, eps: float = 1e-10):
    """Per-output-channel weights: bf16 w [N, K] -> (uint8 [N, K], fp32 [N])."""
    wq, ws = quant_weight_blocks(w, 1, _bits16(w).shape[1], eps)
    return wq, ws.reshape(-1)


# --------------------------------------------------------------------------
# GEMMs
# --------------------------------------------------------------------------

def gemm_channelwise(a, b, sa, sb, bias=None, out_fp16: bool = False, threads: int = 1,
                     return_double: bool = False):
    """a uint8 [M, K], b uint8 [N, K] (weight [K, N] stored K-contiguous),
    sa fp32 [M], sb fp32 [N], bias bf16 [N] or None -> out bits uint16 [M, N]."""
    a8, b8 = _u8(a), _u8(b)
    M, K = a8.shape
    N = b8.shape[0]
    sa_, sb_ = _f32(sa), _f32(sb)
    bb = None if bias is None else _bits16(bias)
    out = np.zeros((M, N), dtype=np.uint16)
    yd = np.zeros((M, N), dtype=np.float64) if return_double else None
    L = lib()
    _run_rows(lambda r0, r1: L.fp8q_oracle_gemm_channelwise(
        _ptr(a8), K, _ptr(b8), K, _ptr(sa_), _ptr(sb_), _ptr(bb), N, K, int(out_fp16),
        _ptr(out), N, _ptr(yd), r0, r1), M, threads)
    return (out, yd) if return_double else out


def gemm_w8a16(x, w, ws, bias=None, out_fp16: bool = False, threads: int = 1, return_double: bool = False):
    """Weight-only FP8: x bf16 [M, K], w uint8 E4M3 [N, K], ws fp32 [N],
    bias bf16 [N] or None -> out bits uint16 [M, N]."""
    xb, w8 = _bits16(x), _u8(w)
    M, K = xb.shape
    N = w8.shape[0]
    ws_ = _f32(ws)
    bb = None if bias is None else _bits16(bias)
    out = np.zeros((M, N), dtype=np.uint16)
    yd = np.zeros((M, N), dtype=np.float64) if return_double else None
    L = lib()
    _run_rows(lambda r0, r1: L.fp8q_oracle_gemm_w8a16(
        _ptr(xb), K, _ptr(w8), K, _ptr(ws_), _ptr(bb), N, K, int(out_fp16), _ptr(out), N, _ptr(yd), r0, r1),
        M, threads)
    return (out, yd) if return_double else out


def gemm_blockwise(a, w, sa_storage, sw, M: int, bias=None, out_fp16: bool = False,
                   threads: int = 1, return_double: bool = False):
    """a uint8 [m_pad, K] (rows >= M ignored), w uint8 [N, K],
    sa_storage fp32 [K/128, m_pad] (column-major activation scales),
    sw fp32 [N/128, K/128] -> out bits uint16 [M, N]."""
    a8, w8 = _u8(a), _u8(w)
    m_pad, K = a8.shape
    N = w8.shape[0]
    sa_, sw_ = _f32(sa_storage), _f32(sw)
    assert sa_.shape == (K // 128, m_pad) and sw_.shape == (N // 128, K // 128)
    bb = None if bias is None else _bits16(bias)
    out = np.zeros((M, N), dtype=np.uint16)
    yd = np.zeros((M, N), dtype=np.float64) if return_double else None
    L = lib()
    _run_rows(lambda r0, r1: L.fp8q_oracle_gemm_blockwise(
        _ptr(a8), K, _ptr(w8), K, _ptr(sa_), m_pad, _ptr(sw_), _ptr(bb), N, K, int(out_fp16),
        _ptr(out), N, _ptr(yd), r0, r1), M, threads)
    return (out, yd) if return_double else out


def gemm_channelwise_at(a, b, sa, sb, ms, ns, bias=None, out_fp16: bool = False):
    a8, b8 = _u8(a), _u8(b)
    K = a8.shape[1]
    ms_ = np.ascontiguousarray(ms, dtype=np.int64)
    ns_ = np.ascontiguousarray(ns, dtype=np.int64)
    sa_, sb_ = _f32(sa), _f32(sb)
    bb = None if bias is None else _bits16(bias)
    out = np.zeros(ms_.size, dtype=np.uint16)
    lib().fp8q_oracle_gemm_channelwise_at(_ptr(a8), K, _ptr(b8), K, _ptr(sa_), _ptr(sb_), _ptr(bb), K,
                                          int(out_fp16), _ptr(ms_), _ptr(ns_), ms_.size, _ptr(out))
    return out


def gemm_blockwise_at(a, w, sa_storage, sw, ms, ns, bias=None, out_fp16: bool = False):
    a8, w8 = _u8(a), _u8(w)
    m_pad, K = a8.shape
    ms_ = np.ascontiguousarray(ms, dtype=np.int64)
    ns_ = np.ascontiguousarray(ns, dtype=np.int64)
    sa_, sw_ = _f32(sa_storage), _f32(sw)
    bb = None if bias is None else _bits16(bias)
    out = np.zeros(ms_.size, dtype=np.uint16)
    lib().fp8q_oracle_gemm_blockwise_at(_ptr(a8), K, _ptr(w8), K, _ptr(sa_), m_pad, _ptr(sw_), _ptr(bb), K,
                                        int(out_fp16), _ptr(ms_), _ptr(ns_), ms_.size, _ptr(out))
    return out


def bf16_bits_to_float(bits) -> np.ndarray:
    """uint16 bf16 bit patterns -> float64 values (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def f16_bits_to_float(bits) -> np.ndarray:
    return np.ascontiguousarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)
