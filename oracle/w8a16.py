"""Plain definition of the W8A16 fused QKV projection (the INT8 sibling).

TEST INFRASTRUCTURE ONLY (see the package docstring). Literal on purpose:
unpack -> dequantise -> float64 matrix product. NumPy's float64 matmul is the
only library primitive used, as the contraction step.

Source: "kaio-candle -- src/qkv_project_int4.rs", module doc. The INT4 op is
described there as following the same direct-call pattern as its INT8 sibling
``qkv_project_int8``, differing in that it takes seven input tensors
(activations, three packed INT4 weight tensors and three f16 group-scale
tensors); the INT8 op likewise returns f16 converted from f32 inside the
kernel. The pages show nothing else of the INT8 op.

Readings where the pages are silent (stated conventions):

- weights are packed like the INT4 ones with 8-bit fields: ``u32[K/4, N]``,
  byte i (bits 8i..8i+7) of word ``P[r, n]`` holds K-row ``4r + i`` as a
  signed two's-complement integer in [-128, 127]; no zero point.
- the "but with seven tensors" contrast is read as: the INT8 op takes no
  group-scale tensors. Each projection has one f32 scale ``s_p`` (per
  tensor), passed by value, so the dequantised weight is ``s_p * w``.
- the reference result is the exact-as-float64 ``sum_k x[m,k] * (s_p *
  w[k,n])``; the f16 output is ``RN_f16`` of it. ``s_p * w`` is exact in
  float64 (a 24-bit significand times an 8-bit integer).
"""
from __future__ import annotations

import numpy as np

from .w4a16 import rn_f16  # noqa: F401  (same f16 rounding of the outputs)


def unpack_int8(packed: np.ndarray) -> np.ndarray:
    """``u32[K/4, N]`` -> ``int8[K, N]``; K-row ``4r+i`` is byte i of row r."""
    p = np.asarray(packed, dtype=np.uint32)
    rows, n = p.shape
    out = np.empty((rows * 4, n), dtype=np.int8)
    for i in range(4):
        byte = ((p >> np.uint32(8 * i)) & np.uint32(0xFF)).astype(np.int16)
        out[i::4, :] = np.where(byte >= 128, byte - 256, byte).astype(np.int8)
    return out


def pack_int8(w: np.ndarray) -> np.ndarray:
    """``int[K, N]`` with values in [-128, 127] -> ``u32[K/4, N]`` (inverse of unpack)."""
    w = np.asarray(w)
    if w.shape[0] % 4:
        raise ValueError("K must be a multiple of 4")
    if w.min(initial=0) < -128 or w.max(initial=0) > 127:
        raise ValueError("INT8 values must lie in [-128, 127]")
    k, n = w.shape
    bits = (w.astype(np.int64) & 0xFF).astype(np.uint32)
    out = np.zeros((k // 4, n), dtype=np.uint32)
    for i in range(4):
        out |= bits[i::4, :] << np.uint32(8 * i)
    return out


def dequant_int8(packed: np.ndarray, scale) -> np.ndarray:
    """``Wd[k, n] = s * int8(W[k, n])`` as float64 (exact), ``s`` one f32 scale."""
    s = float(np.float32(scale))
    return unpack_int8(packed).astype(np.float64) * s


def qkv_project_int8_ref(x, wq, wk, wv, sq, sk, sv):
    """Float64 reference of the fused W8A16 projection: three ``f64[M, N]``.

    ``ref_p = x @ dequant(W_p, s_p)`` with every operand widened to float64.
    Round with ``rn_f16`` to get the f16 outputs.
    """
    x64 = np.asarray(x, dtype=np.float16).astype(np.float64)
    if x64.shape[1] != 4 * np.asarray(wq).shape[0]:
        raise ValueError("x is [M, K] and the packed weights [K/4, N]")
    return tuple(x64 @ dequant_int8(w, s) for w, s in ((wq, sq), (wk, sk), (wv, sv)))


def qkv_project_int8_rows(x, wq, wk, wv, sq, sk, sv, rows):
    """The reference restricted to output rows ``rows`` (for sampled checks)."""
    return qkv_project_int8_ref(np.asarray(x)[np.asarray(rows)], wq, wk, wv, sq, sk, sv)
