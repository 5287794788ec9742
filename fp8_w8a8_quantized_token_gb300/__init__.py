"""fp8_w8a8_quantized_token_gb300 -- FP8 W8A8 linear layer for GB300 (sm_103a).

A thin Python binding over the C ABI of ``libfp8q.so`` (``include/fp8q.h``).
The functions here carry the C entry points' names and only marshal
arguments: they check dtypes, devices and shapes, allocate outputs with
PyTorch, and pass raw device pointers plus the current CUDA stream.  Every
step of the computation runs in the library's CUDA kernels; there is no
fallback of any kind.  If the library is missing, importing works but every
call raises ``RuntimeError``.

Tensors:
  activations  torch.bfloat16, [M, K], contiguous rows (stride(1) == 1)
  quantized    torch.float8_e4m3fn
  scales       torch.float32
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfp8q.so")

FP8Q_OK, FP8Q_ERR_INVALID_ARG, FP8Q_ERR_UNSUPPORTED, FP8Q_ERR_CUDA, FP8Q_ERR_TIMEOUT = range(5)
FP8Q_OUT_BF16, FP8Q_OUT_FP16 = 0, 1
E4M3 = torch.float8_e4m3fn
# Capacity of the library's own scratch array (fp8q_linear_channelwise_noalloc).
NOALLOC_MAX_CODES, NOALLOC_MAX_ROWS = 16 * 1024 * 1024, 16384

# Every symbol include/fp8q.h declares (checked by the ABI test).
EXPORTED = (
    "fp8q_quant_per_token",
    "fp8q_quant_per_token_group_row_padded",
    "fp8q_quant_per_token_group_row_padded_ex",
    "fp8q_quant_static_per_tensor",
    "fp8q_quant_weight_block128",
    "fp8q_scaled_mm_channelwise",
    "fp8q_scaled_mm_blockwise",
    "fp8q_linear_channelwise",
    "fp8q_linear_blockwise",
    "fp8q_linear_channelwise_noalloc",
    "fp8q_linear_blockwise_fused",
    "fp8q_scaled_mm_w8a16",
    "fp8q_gemm_plan",
    "fp8q_workspace_bytes",
    "fp8q_linear_channelwise_launches",
    "fp8q_linear_blockwise_launches",
    "fp8q_set_plan_override",
    "fp8q_device_status",
    "fp8q_last_device_status",
    "fp8q_selftest_wait_timeout",
    "fp8q_selftest_silu_mul",
    "fp8q_status_str",
    "fp8q_version",
)


class Fp8qError(RuntimeError):
    def __init__(self, func: str, status: int):
        self.status = status
        super().__init__(f"{func} failed: {status_str(status)}")


class Plan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("swap_ab", "mma_n", "tile_m", "tile_n", "split_k", "stages", "grid", "persistent", "from_table",
                 "pair", "two_sm", "stream_k", "kb_per_stage")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


_lib = None


def load_library(path: str | None = None):
    """Load libfp8q.so (built in-tree by ``build.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"libfp8q.so not found at {path}: run __graft_entry__.build() "
                           "(or python fp8_w8a8_quantized_token_gb300/build.py) first")
    L = ctypes.CDLL(path)
    P, I64, I32, F32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    sig = {
        "fp8q_quant_per_token": [P, I64, I64, I64, P, P, F32, P],
        "fp8q_quant_per_token_group_row_padded": [P, I64, I64, I64, I32, F32, I32, P, P, I64, P],
        "fp8q_quant_per_token_group_row_padded_ex": [P, I64, I64, I64, I32, F32, I32, I32, P, P, I64, P],
        "fp8q_quant_static_per_tensor": [P, I64, I64, I64, P, P, P, P],
        "fp8q_quant_weight_block128": [P, I64, I64, P, P, F32, P],
        "fp8q_scaled_mm_channelwise": [P, P, I64, P, P, P, P, I64, I64, I64, ctypes.c_int, P, SZ, P],
        "fp8q_scaled_mm_blockwise": [P, P, P, P, P, P, I64, I64, I64, I64, ctypes.c_int, P, SZ, P],
        "fp8q_linear_channelwise": [P, P, I64, P, P, P, I64, I64, I64, P, P, ctypes.c_int, P, SZ, P],
        "fp8q_linear_blockwise": [P, P, P, P, P, I64, I64, I64, P, P, I64, ctypes.c_int, P, SZ, P],
        "fp8q_linear_channelwise_noalloc": [P, P, I64, P, P, P, I64, I64, I64, ctypes.c_int, P],
        "fp8q_linear_blockwise_fused": [P, I64, P, P, P, P, I64, I64, I64, ctypes.c_int, P],
        "fp8q_scaled_mm_w8a16": [P, I64, P, I64, P, P, P, I64, I64, I64, ctypes.c_int, P],
        "fp8q_gemm_plan": [I64, I64, I64, I32, I32, ctypes.POINTER(Plan)],
        "fp8q_device_status": [P, I32],
        "fp8q_last_device_status": [P],
        "fp8q_selftest_wait_timeout": [P],
        "fp8q_selftest_silu_mul": [P, P, P, I64, P],
        "fp8q_set_plan_override": [I32, I32, I32],
    }
    for name, args in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    L.fp8q_status_str.argtypes = [ctypes.c_int]
    L.fp8q_status_str.restype = ctypes.c_char_p
    L.fp8q_version.argtypes = []
    L.fp8q_version.restype = ctypes.c_int32
    L.fp8q_workspace_bytes.argtypes = [I64, I64, I64, I32]
    L.fp8q_workspace_bytes.restype = SZ
    L.fp8q_linear_channelwise_launches.argtypes = [I64, I64, I64]
    L.fp8q_linear_channelwise_launches.restype = ctypes.c_int32
    L.fp8q_linear_blockwise_launches.argtypes = [I64, I64]
    L.fp8q_linear_blockwise_launches.restype = ctypes.c_int32
    _lib = L
    return L


def status_str(status: int) -> str:
    return load_library().fp8q_status_str(int(status)).decode()


def _check(func: str, status: int):
    if status != FP8Q_OK:
        raise Fp8qError(func, status)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _on(device: torch.device):
    """Make the tensors' device current for the C call: the library reads
    the current device for its per-device state (status word, SM count,
    kernel attributes, the no-alloc array's address)."""
    return torch.cuda.device(device)


def _workspace(workspace, M: int, N: int, K: int, blockwise: bool, device: torch.device):
    """(pointer, bytes) of the split-K workspace: "auto" allocates what the
    planned schedule uses (nothing if it does not split K), zero-filled as
    stream-K schedules require; None passes none (K-split partials then go
    through distributed shared memory, and stream-K schedules run split
    along K instead); a uint8 CUDA tensor is used as given (for stream-K it
    must have been zero-filled once: the GEMM leaves it that way)."""
    if workspace is None:
        return None, 0
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError('workspace must be "auto", None or a uint8 CUDA tensor')
        with _on(device):
            nbytes = int(load_library().fp8q_workspace_bytes(M, N, K, int(bool(blockwise))))
        if nbytes == 0:
            return None, 0
        workspace = torch.zeros(nbytes, dtype=torch.uint8, device=device)
    _need(workspace, torch.uint8, "workspace", device)
    if not workspace.is_contiguous():
        raise ValueError("workspace must be contiguous")
    return _ptr(workspace), workspace.numel()


def _need(t: torch.Tensor, dtype, name: str, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _out_code(out_dtype) -> int:
    if out_dtype == torch.bfloat16:
        return FP8Q_OUT_BF16
    if out_dtype == torch.float16:
        return FP8Q_OUT_FP16
    raise TypeError("out_dtype must be torch.bfloat16 or torch.float16")


def ceil_align(m: int, alignment: int) -> int:
    return (m + alignment - 1) // alignment * alignment


# ---------------------------------------------------------------------------
# quantizers
# ---------------------------------------------------------------------------

def fp8q_quant_per_token(x: torch.Tensor, eps: float = 1e-10, xq: torch.Tensor | None = None,
                         x_scale: torch.Tensor | None = None):
    """bf16 [M, K] -> (e4m3 [M, K], fp32 [M]): one scale per token."""
    L = load_library()
    _need(x, torch.bfloat16, "x")
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with contiguous rows")
    M, K = x.shape
    xq = torch.empty((M, K), dtype=E4M3, device=x.device) if xq is None else xq
    x_scale = torch.empty((M,), dtype=torch.float32, device=x.device) if x_scale is None else x_scale
    _need(xq, E4M3, "xq", x.device)
    _need(x_scale, torch.float32, "x_scale", x.device)
    if tuple(xq.shape) != (M, K) or not xq.is_contiguous() or x_scale.numel() < M:
        raise ValueError("xq must be a contiguous [M, K] buffer and x_scale hold M floats")
    with _on(x.device):
        _check("fp8q_quant_per_token",
               L.fp8q_quant_per_token(_ptr(x), M, K, x.stride(0), _ptr(xq), _ptr(x_scale), eps, _stream(x.device)))
    return xq, x_scale


FP8Q_QUANT_SCALE_UE8M0 = 1
FP8Q_QUANT_SILU_AND_MUL = 2


def fp8q_quant_per_token_group_row_padded(x: torch.Tensor, group_size: int = 128, eps: float = 1e-10,
                                          row_alignment: int = 4, xq: torch.Tensor | None = None,
                                          x_scale_storage: torch.Tensor | None = None,
                                          scale_ue8m0: bool = False, fuse_silu_and_mul: bool = False):
    """bf16 [M, K] -> (x_q e4m3 [m_pad, K], x_s fp32 (m_pad, K/g) column-major view).

    As on the row-padding page: m_pad = ceil_align(M, row_alignment), x_s is a
    (K/g, m_pad) allocation viewed transposed (stride(0) == 1); rows >= M of
    both buffers are left as allocated (never written).  scale_ue8m0 rounds
    every scale up to a power of two; fuse_silu_and_mul takes x as [M, 2K]
    and quantizes silu(x[:, :K]) * x[:, K:] (computed in fp32)."""
    L = load_library()
    _need(x, torch.bfloat16, "x")
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with contiguous rows")
    M, K = x.shape
    if fuse_silu_and_mul:
        if K % 2 != 0:
            raise ValueError("fuse_silu_and_mul needs an even last dimension (gate, up)")
        K //= 2
    flags = (FP8Q_QUANT_SCALE_UE8M0 if scale_ue8m0 else 0) | (FP8Q_QUANT_SILU_AND_MUL if fuse_silu_and_mul else 0)
    if K % group_size != 0:
        raise ValueError("the last dimension of x must be divisible by group_size")
    m_pad = ceil_align(M, row_alignment)
    if xq is None:
        xq = torch.empty((m_pad, K), dtype=E4M3, device=x.device)
    if x_scale_storage is None:
        x_scale_storage = torch.empty((K // group_size, m_pad), dtype=torch.float32, device=x.device)
    _need(xq, E4M3, "xq", x.device)
    _need(x_scale_storage, torch.float32, "x_scale_storage", x.device)
    m_pad = xq.shape[0]
    if xq.dim() != 2 or xq.shape[1] != K or not xq.is_contiguous():
        raise ValueError("xq must be a contiguous [m_pad, K] buffer")
    if tuple(x_scale_storage.shape) != (K // group_size, m_pad) or not x_scale_storage.is_contiguous():
        raise ValueError("x_scale_storage must be a contiguous [K/g, m_pad] buffer")
    if flags == 0:
        with _on(x.device):
            _check("fp8q_quant_per_token_group_row_padded",
                   L.fp8q_quant_per_token_group_row_padded(_ptr(x), M, K, x.stride(0), group_size, eps, row_alignment,
                                                           _ptr(xq), _ptr(x_scale_storage), m_pad, _stream(x.device)))
    else:
        with _on(x.device):
            _check("fp8q_quant_per_token_group_row_padded_ex",
                   L.fp8q_quant_per_token_group_row_padded_ex(_ptr(x), M, K, x.stride(0), group_size, eps,
                                                              row_alignment, flags, _ptr(xq), _ptr(x_scale_storage),
                                                              m_pad, _stream(x.device)))
    return xq, x_scale_storage.transpose(0, 1)


def fp8q_quant_static_per_tensor(x: torch.Tensor, scale: torch.Tensor, xq: torch.Tensor | None = None,
                                 repeat_scale: bool = False):
    """Static per-tensor quantization: bf16 [M, K] and a one-element fp32
    device tensor s -> (x_q e4m3 [M, K], the scale repeated to fp32 [M] if
    repeat_scale else None).  x_q = e4m3(x / s), saturating."""
    L = load_library()
    _need(x, torch.bfloat16, "x")
    _need(scale, torch.float32, "scale", x.device)
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with contiguous rows")
    if scale.numel() != 1:
        raise ValueError("scale must hold exactly one value")
    M, K = x.shape
    if xq is None:
        xq = torch.empty((M, K), dtype=E4M3, device=x.device)
    _need(xq, E4M3, "xq", x.device)
    if tuple(xq.shape) != (M, K) or not xq.is_contiguous():
        raise ValueError("xq must be a contiguous [M, K] buffer")
    rep = torch.empty(M, dtype=torch.float32, device=x.device) if repeat_scale else None
    with _on(x.device):
        _check("fp8q_quant_static_per_tensor",
               L.fp8q_quant_static_per_tensor(_ptr(x), M, K, x.stride(0), _ptr(scale), _ptr(xq),
                                              None if rep is None else _ptr(rep), _stream(x.device)))
    return xq, rep


def fp8q_quant_weight_block128(w: torch.Tensor, eps: float = 1e-10):
    """bf16 [N, K] -> (e4m3 [N, K], fp32 [N/128, K/128])."""
    L = load_library()
    _need(w, torch.bfloat16, "w")
    if w.dim() != 2 or not w.is_contiguous():
        raise ValueError("w must be a contiguous 2-D tensor")
    N, K = w.shape
    wq = torch.empty((N, K), dtype=E4M3, device=w.device)
    ws = torch.empty((N // 128, K // 128), dtype=torch.float32, device=w.device)
    with _on(w.device):
        _check("fp8q_quant_weight_block128",
               L.fp8q_quant_weight_block128(_ptr(w), N, K, _ptr(wq), _ptr(ws), eps, _stream(w.device)))
    return wq, ws


# ---------------------------------------------------------------------------
# GEMMs
# ---------------------------------------------------------------------------

def fp8q_scaled_mm_channelwise(a: torch.Tensor, b: torch.Tensor, a_scale: torch.Tensor, b_scale: torch.Tensor,
                               bias: torch.Tensor | None = None, out_dtype=torch.bfloat16,
                               out: torch.Tensor | None = None, workspace="auto"):
    """a e4m3 [M, K]; b e4m3 weight given as its [N, K] K-contiguous storage
    (logical [K, N] = b.T); a_scale fp32 [M]; b_scale fp32 [N]; bias bf16 [N].
    Returns out [M, N] of out_dtype.  workspace: see _workspace."""
    L = load_library()
    _need(a, E4M3, "a")
    _need(b, E4M3, "b", a.device)
    _need(a_scale, torch.float32, "a_scale", a.device)
    _need(b_scale, torch.float32, "b_scale", a.device)
    if bias is not None:
        _need(bias, torch.bfloat16, "bias", a.device)
    if a.dim() != 2 or not a.is_contiguous() or b.dim() != 2 or b.stride(1) != 1:
        raise ValueError("a must be contiguous [M, K]; b must be [N, K] with contiguous rows")
    M, K = a.shape
    N = b.shape[0]
    if b.shape[1] != K:
        raise ValueError("a and b disagree on K")
    code = _out_code(out_dtype)
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=a.device)
    _need(out, out_dtype, "out", a.device)
    ws, ws_bytes = _workspace(workspace, M, N, K, False, a.device)
    with _on(a.device):
        _check("fp8q_scaled_mm_channelwise",
               L.fp8q_scaled_mm_channelwise(_ptr(a), _ptr(b), b.stride(0), _ptr(a_scale), _ptr(b_scale), _ptr(bias),
                                            _ptr(out), M, N, K, code, ws, ws_bytes, _stream(a.device)))
    return out


def fp8q_scaled_mm_blockwise(a: torch.Tensor, w: torch.Tensor, a_scale: torch.Tensor, w_scale: torch.Tensor,
                             M: int | None = None, bias: torch.Tensor | None = None, out_dtype=torch.bfloat16,
                             out: torch.Tensor | None = None, workspace="auto"):
    """a e4m3 [m_pad, K] (row-padded); w e4m3 [N, K]; a_scale the (m_pad, K/128)
    column-major view (or its [K/128, m_pad] storage); w_scale fp32 [N/128, K/128].
    Returns out [M, N] (M defaults to m_pad)."""
    L = load_library()
    _need(a, E4M3, "a")
    _need(w, E4M3, "w", a.device)
    _need(a_scale, torch.float32, "a_scale", a.device)
    _need(w_scale, torch.float32, "w_scale", a.device)
    if bias is not None:
        _need(bias, torch.bfloat16, "bias", a.device)
    m_pad, K = a.shape
    N = w.shape[0]
    M = m_pad if M is None else int(M)
    # The (m_pad, K/128) column-major view (stride(0) == 1) or its [K/128,
    # m_pad] contiguous storage; decided by the strides, since the two have
    # the same shape when K/128 == m_pad.
    if a_scale.dim() == 2 and tuple(a_scale.shape) == (m_pad, K // 128) and a_scale.stride(0) == 1 \
            and (a_scale.stride(1) == m_pad or K // 128 == 1):
        storage = a_scale.transpose(0, 1)
    else:
        storage = a_scale
    if tuple(storage.shape) != (K // 128, m_pad) or not storage.is_contiguous():
        raise ValueError("a_scale must be the column-major (m_pad, K/128) scales of the row-padded quantizer")
    if not a.is_contiguous() or not w.is_contiguous() or not w_scale.is_contiguous():
        raise ValueError("a, w and w_scale must be contiguous")
    code = _out_code(out_dtype)
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=a.device)
    _need(out, out_dtype, "out", a.device)
    ws, ws_bytes = _workspace(workspace, M, N, K, True, a.device)
    with _on(a.device):
        _check("fp8q_scaled_mm_blockwise",
               L.fp8q_scaled_mm_blockwise(_ptr(a), _ptr(w), _ptr(storage), _ptr(w_scale), _ptr(bias), _ptr(out),
                                          M, m_pad, N, K, code, ws, ws_bytes, _stream(a.device)))
    return out


def fp8q_linear_channelwise(x: torch.Tensor, b: torch.Tensor, b_scale: torch.Tensor, bias=None,
                            out_dtype=torch.bfloat16, workspace="auto"):
    """Per-token quantization of x followed by the channelwise GEMM."""
    L = load_library()
    _need(x, torch.bfloat16, "x")
    _need(b, E4M3, "b", x.device)
    _need(b_scale, torch.float32, "b_scale", x.device)
    if bias is not None:
        _need(bias, torch.bfloat16, "bias", x.device)
    if x.dim() != 2 or not x.is_contiguous() or b.stride(1) != 1:
        raise ValueError("x must be contiguous [M, K]; b [N, K] with contiguous rows")
    M, K = x.shape
    N = b.shape[0]
    xq = torch.empty((M, K), dtype=E4M3, device=x.device)
    xs = torch.empty((M,), dtype=torch.float32, device=x.device)
    out = torch.empty((M, N), dtype=out_dtype, device=x.device)
    ws, ws_bytes = _workspace(workspace, M, N, K, False, x.device)
    with _on(x.device):
        _check("fp8q_linear_channelwise",
               L.fp8q_linear_channelwise(_ptr(x), _ptr(b), b.stride(0), _ptr(b_scale), _ptr(bias), _ptr(out), M, N,
                                         K, _ptr(xq), _ptr(xs), _out_code(out_dtype), ws, ws_bytes,
                                         _stream(x.device)))
    return out


def fp8q_linear_blockwise(x: torch.Tensor, w: torch.Tensor, w_scale: torch.Tensor, bias=None,
                          out_dtype=torch.bfloat16, workspace="auto"):
    """Row-padded group quantization of x followed by the blockwise GEMM; the
    output has exactly M rows (the padded rows are never materialised)."""
    L = load_library()
    _need(x, torch.bfloat16, "x")
    _need(w, E4M3, "w", x.device)
    _need(w_scale, torch.float32, "w_scale", x.device)
    if bias is not None:
        _need(bias, torch.bfloat16, "bias", x.device)
    if x.dim() != 2 or not x.is_contiguous():
        raise ValueError("x must be contiguous [M, K]")
    M, K = x.shape
    N = w.shape[0]
    m_pad = ceil_align(M, 4)
    xq = torch.empty((m_pad, K), dtype=E4M3, device=x.device)
    xs = torch.empty((K // 128, m_pad), dtype=torch.float32, device=x.device)
    out = torch.empty((M, N), dtype=out_dtype, device=x.device)
    ws, ws_bytes = _workspace(workspace, M, N, K, True, x.device)
    with _on(x.device):
        _check("fp8q_linear_blockwise",
               L.fp8q_linear_blockwise(_ptr(x), _ptr(w), _ptr(w_scale), _ptr(bias), _ptr(out), M, N, K, _ptr(xq),
                                       _ptr(xs), m_pad, _out_code(out_dtype), ws, ws_bytes, _stream(x.device)))
    return out


def fp8q_linear_blockwise_fused(x: torch.Tensor, w: torch.Tensor, w_scale: torch.Tensor, bias=None,
                                out_dtype=torch.bfloat16):
    """The blockwise linear layer in one kernel: group-128 quantization of
    the bf16 activations inside the GEMM (decode sizes whose schedule is the
    16- or 32-token tile; otherwise FP8Q_ERR_UNSUPPORTED).  Bit-identical to
    fp8q_linear_blockwise on the same schedule."""
    L = load_library()
    _need(x, torch.bfloat16, "x")
    _need(w, E4M3, "w", x.device)
    _need(w_scale, torch.float32, "w_scale", x.device)
    if bias is not None:
        _need(bias, torch.bfloat16, "bias", x.device)
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with contiguous rows")
    M, K = x.shape
    N = w.shape[0]
    out = torch.empty((M, N), dtype=out_dtype, device=x.device)
    with _on(x.device):
        _check("fp8q_linear_blockwise_fused",
               L.fp8q_linear_blockwise_fused(_ptr(x), x.stride(0), _ptr(w), _ptr(w_scale), _ptr(bias), _ptr(out), M, N,
                                             K, _out_code(out_dtype), _stream(x.device)))
    return out


def fp8q_scaled_mm_w8a16(x: torch.Tensor, w: torch.Tensor, w_scale: torch.Tensor, bias=None,
                         out_dtype=torch.bfloat16, out: torch.Tensor | None = None):
    """Weight-only FP8 linear: bf16 x [M, K] @ (e4m3 w [N, K] * w_scale[N]).T
    (+ bias) -> [M, N], fp32 accumulation, no activation quantization."""
    L = load_library()
    _need(x, torch.bfloat16, "x")
    _need(w, E4M3, "w", x.device)
    _need(w_scale, torch.float32, "w_scale", x.device)
    if bias is not None:
        _need(bias, torch.bfloat16, "bias", x.device)
    if x.dim() != 2 or x.stride(1) != 1 or w.dim() != 2 or w.stride(1) != 1:
        raise ValueError("x and w must be 2-D with contiguous rows")
    M, K = x.shape
    N = w.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=x.device)
    with _on(x.device):
        _check("fp8q_scaled_mm_w8a16",
               L.fp8q_scaled_mm_w8a16(_ptr(x), x.stride(0), _ptr(w), w.stride(0), _ptr(w_scale), _ptr(bias), _ptr(out),
                                      M, N, K, _out_code(out.dtype), _stream(x.device)))
    return out


def fp8q_linear_channelwise_noalloc(x: torch.Tensor, b: torch.Tensor, b_scale: torch.Tensor, bias=None,
                                    out_dtype=torch.bfloat16, out: torch.Tensor | None = None):
    """fp8q_linear_channelwise without scratch buffers: the quantized
    activations live in the library's fixed device array, so the C call
    allocates nothing (for callers whose device memory is owned by another
    allocator, or that cannot take cudaMalloc's synchronisation).  Only
    ``out`` is the caller's; pass it to keep this wrapper from allocating.
    Limits: M <= NOALLOC_MAX_ROWS and M * K <= NOALLOC_MAX_CODES.  Calls that
    can overlap on the GPU (other streams) share that array and race."""
    L = load_library()
    _need(x, torch.bfloat16, "x")
    _need(b, E4M3, "b", x.device)
    _need(b_scale, torch.float32, "b_scale", x.device)
    if bias is not None:
        _need(bias, torch.bfloat16, "bias", x.device)
    if x.dim() != 2 or not x.is_contiguous() or b.stride(1) != 1:
        raise ValueError("x must be contiguous [M, K]; b [N, K] with contiguous rows")
    M, K = x.shape
    N = b.shape[0]
    if M > NOALLOC_MAX_ROWS or M * K > NOALLOC_MAX_CODES:
        raise ValueError(f"x is {M} x {K}: the no-alloc scratch holds at most {NOALLOC_MAX_ROWS} rows and "
                         f"{NOALLOC_MAX_CODES} elements; use fp8q_linear_channelwise with your own buffers")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=x.device)
    _need(out, out_dtype, "out", x.device)
    if tuple(out.shape) != (M, N) or not out.is_contiguous():
        raise ValueError("out must be a contiguous [M, N] tensor")
    with _on(x.device):
        _check("fp8q_linear_channelwise_noalloc",
               L.fp8q_linear_channelwise_noalloc(_ptr(x), _ptr(b), b.stride(0), _ptr(b_scale), _ptr(bias), _ptr(out),
                                                 M, N, K, _out_code(out_dtype), _stream(x.device)))
    return out


def fp8q_gemm_plan(M: int, N: int, K: int, blockwise: bool = False, num_sms: int = 0) -> dict:
    """The schedule the library would launch for this problem (host only)."""
    L = load_library()
    p = Plan()
    _check("fp8q_gemm_plan", L.fp8q_gemm_plan(M, N, K, int(bool(blockwise)), num_sms, ctypes.byref(p)))
    return p.as_dict()


def fp8q_workspace_bytes(M: int, N: int, K: int, blockwise: bool = False, device=None) -> int:
    """Bytes of split-K workspace the planned GEMM uses on `device` (default:
    the current device); 0 if its schedule does not split K."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with _on(device):
        return int(load_library().fp8q_workspace_bytes(M, N, K, int(bool(blockwise))))


def fp8q_linear_channelwise_launches(M: int, N: int, K: int) -> int:
    """Kernel launches fp8q_linear_channelwise makes for M tokens of K values
    against N output channels (1: the fused one-token form; 2: quantizer +
    GEMM; 0: nothing to do)."""
    return int(load_library().fp8q_linear_channelwise_launches(M, N, K))


def fp8q_linear_blockwise_launches(M: int, K: int) -> int:
    """Kernel launches fp8q_linear_blockwise makes for M tokens of K values
    (1: the fused one-token form; 2: quantizer + GEMM; 0: nothing to do)."""
    return int(load_library().fp8q_linear_blockwise_launches(M, K))


def fp8q_set_plan_override(swap_ab: int, mma_n: int = 0, split_k: int = 1) -> None:
    """Force the GEMM schedule for this process (swap_ab < 0 clears it)."""
    _check("fp8q_set_plan_override", load_library().fp8q_set_plan_override(swap_ab, mma_n, split_k))


def fp8q_device_status(reset: bool = True, device=None) -> int:
    """Synchronize the current stream and return the device status word
    (FP8Q_OK, or FP8Q_ERR_TIMEOUT if a GEMM gave up on a pipeline wait)."""
    L = load_library()
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with _on(device):
        return int(L.fp8q_device_status(_stream(device), int(bool(reset))))


def fp8q_selftest_wait_timeout(device=None) -> None:
    """Enqueue the diagnostics kernel whose bounded pipeline wait runs out
    (about 2 s); fp8q_device_status() then reports FP8Q_ERR_TIMEOUT."""
    L = load_library()
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with _on(device):
        _check("fp8q_selftest_wait_timeout", L.fp8q_selftest_wait_timeout(_stream(device)))


def fp8q_version() -> int:
    return int(load_library().fp8q_version())
