"""Thin Python binding of libkaio_qkv (C ABI in include/kaio_qkv.h).

Argument marshalling only: shape/dtype checks on the torch tensors, output
allocation with torch, and one ctypes call per operation. Every step of the
computation runs in the library's CUDA kernels; there is no CPU path. If the
library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional, Tuple

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkaio_qkv.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "kaio_qkv.h")

KAIO_OK = 0
KAIO_ERR_INVALID_VALUE = 1
KAIO_ERR_MISALIGNED = 2
KAIO_ERR_UNSUPPORTED_DEVICE = 3
KAIO_ERR_CUDA = 4
KAIO_ERR_DEVICE_TIMEOUT = 5

KAIO_DTYPE_F32, KAIO_DTYPE_F64, KAIO_DTYPE_F16, KAIO_DTYPE_BF16, KAIO_DTYPE_S8, KAIO_DTYPE_U8 = range(6)

_lib = None

_vp, _u32, _i32 = ctypes.c_void_p, ctypes.c_uint32, ctypes.c_int
_SIGNATURES = {
    "kaio_qkv_project_int4": ([_vp] * 10 + [_u32, _u32, _u32, _vp], _i32),
    "kaio_qkv_project_int4_noalloc": ([_vp] * 10 + [_u32, _u32, _u32, _vp], _i32),
    "kaio_debug_decode_wait_limit": ([_vp] * 10 + [_u32, _u32, _u32, ctypes.c_uint64, _vp], _i32),
    "kaio_matmul_tc": ([_vp, _vp, _vp, _u32, _u32, _u32, _vp], _i32),
    "kaio_matmul_tc_backward": ([_vp] * 5 + [_u32, _u32, _u32, _vp], _i32),
    "kaio_matmul_tc_f16": ([_vp, _vp, _vp, _u32, _u32, _u32, _vp], _i32),
    "kaio_matmul_tc_backward_f16": ([_vp] * 5 + [_u32, _u32, _u32, _vp], _i32),
    "kaio_dequant_int4_debug": ([_vp, _vp, _vp, _u32, _u32, _i32, _vp], _i32),
    "kaio_dequantize_per_group_backward": ([_i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp], _i32),
    "kaio_dequantize_per_group": ([_i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp], _i32),
    "kaio_qkv_project_int8": ([_vp] * 4 + [ctypes.c_float] * 3 + [_vp] * 3 + [_u32, _u32, _u32, _vp], _i32),
    "kaio_qkv_path": ([_u32], _i32),
    "kaio_last_error": ([], ctypes.c_char_p),
    "kaio_device_status": ([], _i32),
    "kaio_status_string": ([_i32], ctypes.c_char_p),
}


class KaioError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_string(status)}: {message}")
        self.status = status


def lib():
    """Load the shared library (once). Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; g.build()\"`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def header_functions():
    """Names of the functions declared in include/kaio_qkv.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|const char\*)\s+(kaio_\w+)\s*\(", text, re.M)))


def status_string(status: int) -> str:
    try:
        return lib().kaio_status_string(status).decode()
    except Exception:  # pragma: no cover - library missing
        return f"status {status}"


def last_error() -> str:
    return lib().kaio_last_error().decode()


def check(status: int) -> None:
    if status != KAIO_OK:
        raise KaioError(status, last_error())


# ------------------------------------------------------------------ helpers
def _torch():
    import torch
    return torch


def _stream_ptr(stream) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _need(t, name, dtypes, shape=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be on a CUDA device (no CPU fallback)")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (row-major, no strides of its own)")
    if t.dim() != 2:
        raise ValueError(f"{name} must be rank 2, got shape {tuple(t.shape)}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.requires_grad:
        raise ValueError(f"{name} has gradient tracking enabled; these ops are forward-only: detach() it")


_PACKED = None


def _packed_dtypes():
    global _PACKED
    if _PACKED is None:
        torch = _torch()
        _PACKED = (torch.int32, torch.uint32) if hasattr(torch, "uint32") else (torch.int32,)
    return _PACKED


# ------------------------------------------------------------------ public API
def qkv_project_int4(x, w_q_packed, w_k_packed, w_v_packed, scales_q, scales_k, scales_v,
                     out: Optional[Tuple] = None, stream=None):
    """Fused W4A16 QKV projection: returns (q, k, v), each f16 [M, N].

    x f16 [M, K]; w_*_packed int32/uint32 [K/8, N] (8 signed INT4 per word, nibble
    i = K-row 8r+i); scales_* f16 [K/128, N].
    """
    torch = _torch()
    _need(x, "x", (torch.float16,))
    m, k = x.shape
    if k % 128:
        raise ValueError(f"K ({k}) must be a multiple of group_size (128)")
    n = w_q_packed.shape[1] if w_q_packed.dim() == 2 else -1
    for name, t in (("w_q_packed", w_q_packed), ("w_k_packed", w_k_packed), ("w_v_packed", w_v_packed)):
        _need(t, name, _packed_dtypes(), (k // 8, n))
    for name, t in (("scales_q", scales_q), ("scales_k", scales_k), ("scales_v", scales_v)):
        _need(t, name, (torch.float16,), (k // 128, n))
    if out is None:
        out = tuple(torch.empty((m, n), dtype=torch.float16, device=x.device) for _ in range(3))
    for name, t in zip("qkv", out):
        _need(t, name, (torch.float16,), (m, n))
    check(lib().kaio_qkv_project_int4(
        x.data_ptr(), w_q_packed.data_ptr(), w_k_packed.data_ptr(), w_v_packed.data_ptr(),
        scales_q.data_ptr(), scales_k.data_ptr(), scales_v.data_ptr(),
        out[0].data_ptr(), out[1].data_ptr(), out[2].data_ptr(), m, n, k, _stream_ptr(stream)))
    return out


def qkv_project_int8(x, w_q_packed, w_k_packed, w_v_packed, scale_q: float, scale_k: float,
                     scale_v: float, out: Optional[Tuple] = None, stream=None):
    """Fused W8A16 QKV projection: returns (q, k, v), each f16 [M, N].

    x f16 [M, K]; w_*_packed int32/uint32 [K/4, N] (4 signed INT8 per word,
    byte i = K-row 4r+i); scale_* one float per projection (passed as f32).
    """
    torch = _torch()
    _need(x, "x", (torch.float16,))
    m, k = x.shape
    if k % 128:
        raise ValueError(f"K ({k}) must be a multiple of 128")
    n = w_q_packed.shape[1] if w_q_packed.dim() == 2 else -1
    for name, t in (("w_q_packed", w_q_packed), ("w_k_packed", w_k_packed), ("w_v_packed", w_v_packed)):
        _need(t, name, _packed_dtypes(), (k // 4, n))
    if out is None:
        out = tuple(torch.empty((m, n), dtype=torch.float16, device=x.device) for _ in range(3))
    for name, t in zip("qkv", out):
        _need(t, name, (torch.float16,), (m, n))
    check(lib().kaio_qkv_project_int8(
        x.data_ptr(), w_q_packed.data_ptr(), w_k_packed.data_ptr(), w_v_packed.data_ptr(),
        float(scale_q), float(scale_k), float(scale_v),
        out[0].data_ptr(), out[1].data_ptr(), out[2].data_ptr(), m, n, k, _stream_ptr(stream)))
    return out


def matmul_tc(a, b, out=None, stream=None, out_dtype=None):
    """C = A @ B on the tensor cores: a f16 [M, K], b f16 [K, N] -> [M, N] in
    f32 (default) or f16 (rounded in the kernel's epilogue)."""
    torch = _torch()
    _need(a, "a", (torch.float16,))
    _need(b, "b", (torch.float16,))
    m, k = a.shape
    k2, n = b.shape
    if k != k2:
        raise ValueError(f"K mismatch between inputs: a is [{m}, {k}], b is [{k2}, {n}]")
    if out_dtype is None:
        out_dtype = out.dtype if out is not None else torch.float32
    if out_dtype not in (torch.float32, torch.float16):
        raise ValueError(f"out_dtype must be float32 or float16, got {out_dtype}")
    if out is None:
        out = torch.empty((m, n), dtype=out_dtype, device=a.device)
    _need(out, "c", (out_dtype,), (m, n))
    fn = lib().kaio_matmul_tc if out_dtype == torch.float32 else lib().kaio_matmul_tc_f16
    check(fn(a.data_ptr(), b.data_ptr(), out.data_ptr(), m, n, k, _stream_ptr(stream)))
    return out


def matmul_tc_backward(a, b, g, stream=None, out_dtype=None, out=None):
    """(dA, dB) = (G @ B^T, A^T @ G) for C = A @ B, with g f16 [M, N]; the
    results are f32 (default) or f16 (rounded in the kernels' epilogues),
    written into ``out = (da, db)`` when given."""
    torch = _torch()
    _need(a, "a", (torch.float16,))
    _need(b, "b", (torch.float16,))
    m, k = a.shape
    n = b.shape[1]
    _need(b, "b", (torch.float16,), (k, n))
    _need(g, "g", (torch.float16,), (m, n))
    out_dtype = torch.float32 if out_dtype is None else out_dtype
    if out_dtype not in (torch.float32, torch.float16):
        raise ValueError(f"out_dtype must be float32 or float16, got {out_dtype}")
    if out is None:
        da = torch.empty((m, k), dtype=out_dtype, device=a.device)
        db = torch.empty((k, n), dtype=out_dtype, device=a.device)
    else:
        da, db = out
        _need(da, "da", (out_dtype,), (m, k))
        _need(db, "db", (out_dtype,), (k, n))
    fn = lib().kaio_matmul_tc_backward if out_dtype == torch.float32 else lib().kaio_matmul_tc_backward_f16
    check(fn(a.data_ptr(), b.data_ptr(), g.data_ptr(), da.data_ptr(), db.data_ptr(), m, n, k,
             _stream_ptr(stream)))
    return da, db


def dequant_int4_debug(w_packed, scales, variant: int = 0, stream=None):
    """f16 [K, N] dequantised weights, exactly as the kernels build them."""
    torch = _torch()
    _need(w_packed, "w", _packed_dtypes())
    rows, n = w_packed.shape
    k = rows * 8
    _need(scales, "s", (torch.float16,), (k // 128, n))
    out = torch.empty((k, n), dtype=torch.float16, device=w_packed.device)
    check(lib().kaio_dequant_int4_debug(w_packed.data_ptr(), scales.data_ptr(), out.data_ptr(),
                                        k, n, variant, _stream_ptr(stream)))
    return out


def qkv_path(m: int) -> int:
    return lib().kaio_qkv_path(m)


def device_status() -> None:
    """Synchronise and raise if a kernel reported a bounded-wait timeout."""
    check(lib().kaio_device_status())


def _float_code(dtype):
    torch = _torch()
    codes = {torch.float32: KAIO_DTYPE_F32, torch.float64: KAIO_DTYPE_F64,
             torch.float16: KAIO_DTYPE_F16, torch.bfloat16: KAIO_DTYPE_BF16}
    if dtype not in codes:
        raise TypeError(f"dtype {dtype} is not one of float32, float64, float16, bfloat16")
    return codes[dtype]


def dequantize_per_group_backward(dy, scale, group: int, q_dtype=None, out=None, stream=None):
    """dx[i, j] = dy[i, j] * scale[i, j // group] (straight-through backward of
    the per-group dequantisation), for dy [outer, axis] and scale
    [outer, axis // group] of one float type. q_dtype (int8 or uint8, default
    int8) is the forward's quantised type; out may be dy itself (in place)."""
    torch = _torch()
    fdt = (torch.float32, torch.float64, torch.float16, torch.bfloat16)
    _need(dy, "dy", fdt)
    outer, axis = dy.shape
    if group <= 0 or axis % group != 0:
        raise ValueError(f"group ({group}) must be > 0 and divide axis ({axis})")
    _need(scale, "scale", (dy.dtype,), (outer, axis // group))
    q_dtype = torch.int8 if q_dtype is None else q_dtype
    qcode = {torch.int8: KAIO_DTYPE_S8, torch.uint8: KAIO_DTYPE_U8}.get(q_dtype)
    if qcode is None:
        raise TypeError("q_dtype must be torch.int8 or torch.uint8")
    if out is None:
        out = torch.empty_like(dy)
    _need(out, "dx", (dy.dtype,), (outer, axis))
    check(lib().kaio_dequantize_per_group_backward(_float_code(dy.dtype), qcode, outer, axis, group,
                                                   dy.data_ptr(), scale.data_ptr(), out.data_ptr(),
                                                   _stream_ptr(stream)))
    return out


def dequantize_per_group(q, scale, group: int, out=None, stream=None):
    """out[i, j] = T(q[i, j]) * scale[i, j // group] for q int8 or uint8
    [outer, axis] and scale [outer, axis // group] of float type T."""
    torch = _torch()
    _need(q, "q", (torch.int8, torch.uint8))
    outer, axis = q.shape
    if group <= 0 or axis % group != 0:
        raise ValueError(f"group ({group}) must be > 0 and divide axis ({axis})")
    _need(scale, "scale", (torch.float32, torch.float64, torch.float16, torch.bfloat16), (outer, axis // group))
    if out is None:
        out = torch.empty((outer, axis), dtype=scale.dtype, device=q.device)
    _need(out, "out", (scale.dtype,), (outer, axis))
    qcode = KAIO_DTYPE_S8 if q.dtype == torch.int8 else KAIO_DTYPE_U8
    check(lib().kaio_dequantize_per_group(qcode, _float_code(scale.dtype), outer, axis, group,
                                          q.data_ptr(), scale.data_ptr(), out.data_ptr(), _stream_ptr(stream)))
    return out
