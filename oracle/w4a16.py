"""Plain definitions of what the W4A16 QKV projection and the dense matmul compute.

TEST INFRASTRUCTURE ONLY (see the package docstring). Slow and literal on
purpose: unpack -> dequantise -> float64 matrix product. NumPy's float64 matmul
is the only library primitive used, as the contraction step.

Sources (docs.rs pages of the ``kaio-candle`` crate):

- "kaio-candle -- src/qkv_project_int4.rs", doc comment of ``qkv_project_int4``:
  x is ``f16[M, K]``; ``w_q_packed``/``w_k_packed``/``w_v_packed`` are
  ``u32[K/8, N]`` with 8 INT4 values packed per ``u32``; ``scales_*`` are
  ``f16[K/128, N]``, one scale per group of 128 elements; outputs are three
  ``f16[M, N]``; ``K`` must be a multiple of 128 (``GROUP_SIZE`` is locked).
- same page, module doc "Output dtype": the kernel accumulates in f32 and
  converts f32 to f16 inside the kernel.
- "kaio-candle 0.2.0 -- src/matmul_tc_async.rs", module doc: f16 x f16 -> f32
  tensor-core matmul; ``MatmulTcAsyncOp::bwd`` doc: dA = grad @ B^T,
  dB = A^T @ grad.

Readings where the pages are silent (each is a stated convention, not a guess
about hidden code):

- nibble i of packed word ``P[r, n]`` is bits ``4i..4i+3`` and holds K-row
  ``8r + i``; the nibble is a signed two's-complement integer in [-8, 7]; there
  is no zero point (the op takes exactly seven inputs).
- group of K-row k is ``k // 128``; scale ``s[k // 128, n]`` multiplies
  column n.
- the dequantised weight is ``RN_f16(w * s)``: the exact product rounded once,
  to nearest-even, to f16 (the tensor-core operand is f16).
- the reference result is the exact-as-float64 sum ``sum_k x[m,k] * Wd[k,n]``;
  the f16 output is ``RN_f16`` of it.
"""
from __future__ import annotations

import numpy as np

GROUP_SIZE = 128


def unpack_int4(packed: np.ndarray) -> np.ndarray:
    """``u32[K/8, N]`` -> ``int8[K, N]``; K-row ``8r+i`` is nibble i of row r."""
    p = np.asarray(packed, dtype=np.uint32)
    rows, n = p.shape
    out = np.empty((rows * 8, n), dtype=np.int8)
    for i in range(8):
        nib = ((p >> np.uint32(4 * i)) & np.uint32(0xF)).astype(np.int16)
        signed = np.where(nib >= 8, nib - 16, nib)
        out[i::8, :] = signed.astype(np.int8)
    return out


def pack_int4(w: np.ndarray) -> np.ndarray:
    """``int[K, N]`` with values in [-8, 7] -> ``u32[K/8, N]`` (inverse of unpack)."""
    w = np.asarray(w)
    if w.shape[0] % 8:
        raise ValueError("K must be a multiple of 8")
    if w.min(initial=0) < -8 or w.max(initial=0) > 7:
        raise ValueError("INT4 values must lie in [-8, 7]")
    k, n = w.shape
    bits = (w.astype(np.int64) & 0xF).astype(np.uint32)
    out = np.zeros((k // 8, n), dtype=np.uint32)
    for i in range(8):
        out |= bits[i::8, :] << np.uint32(4 * i)
    return out


def rn_f16(v) -> np.ndarray:
    """Round float64 values to the nearest f16, ties to even (IEEE 754 binary16)."""
    with np.errstate(over="ignore"):          # |v| >= 65520 rounds to +/-inf
        return np.asarray(v, dtype=np.float64).astype(np.float16)


def dequant_int4(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """``Wd[k, n] = RN_f16(int4(W[k, n]) * s[k // 128, n])`` as ``f16[K, N]``."""
    w = unpack_int4(packed).astype(np.float64)
    s = np.asarray(scales, dtype=np.float16).astype(np.float64)
    k = w.shape[0]
    if k % GROUP_SIZE:
        raise ValueError("K must be a multiple of 128")
    if s.shape != (k // GROUP_SIZE, w.shape[1]):
        raise ValueError("scales must be [K/128, N]")
    s_rows = np.repeat(s, GROUP_SIZE, axis=0)   # row k holds s[k // 128, :]
    return rn_f16(w * s_rows)


def qkv_project_int4_ref(x, wq, wk, wv, sq, sk, sv):
    """Float64 reference of the fused projection: three ``f64[M, N]``.

    ``ref_p = x @ dequant(W_p, s_p)`` with every operand widened to float64.
    Round with :func:`rn_f16` to get the f16 outputs.
    """
    x64 = np.asarray(x, dtype=np.float16).astype(np.float64)
    outs = []
    for w, s in ((wq, sq), (wk, sk), (wv, sv)):
        wd = dequant_int4(w, s).astype(np.float64)
        outs.append(x64 @ wd)
    return tuple(outs)


def qkv_project_int4_rows(x, wq, wk, wv, sq, sk, sv, rows):
    """The reference restricted to output rows ``rows`` (for sampled checks)."""
    x_rows = np.asarray(x)[np.asarray(rows)]
    return qkv_project_int4_ref(x_rows, wq, wk, wv, sq, sk, sv)


def matmul_ref(a, b):
    """Dense ``C = A @ B`` in float64 from f16 operands (``C`` is ``[M, N]``)."""
    return (np.asarray(a, dtype=np.float16).astype(np.float64)
            @ np.asarray(b, dtype=np.float16).astype(np.float64))


def matmul_rows(a, b, rows):
    """Rows ``rows`` of :func:`matmul_ref`."""
    return matmul_ref(np.asarray(a)[np.asarray(rows)], b)


def matmul_backward_ref(a, b, g):
    """Backward of ``C = A @ B``: ``dA = G @ B^T`` and ``dB = A^T @ G`` (float64)."""
    a64 = np.asarray(a, dtype=np.float16).astype(np.float64)
    b64 = np.asarray(b, dtype=np.float16).astype(np.float64)
    g64 = np.asarray(g, dtype=np.float16).astype(np.float64)
    return g64 @ b64.T, a64.T @ g64


def ulp_f16(v) -> np.ndarray:
    """Spacing of f16 numbers at |v|: ``2**(e-10)`` for normal |v| in
    ``[2**e, 2**(e+1))``, and ``2**-24`` in the subnormal range."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, ex = np.frexp(a)               # a = f * 2**ex with f in [0.5, 1)
    e = np.maximum(ex.astype(np.float64) - 1.0, -14.0)
    return np.where(a > 0, np.exp2(e - 10.0), 2.0 ** -24)
