"""Plain definitions of the per-group dequantisation and its backward.

TEST INFRASTRUCTURE ONLY (see the package docstring). Elementwise and literal:
each result is the exact product of two values, rounded once to the element
type.

Source ("baracuda-kernels -- src/quantize/dequantize_per_group_backward.rs",
module doc and the doc of ``DequantizePerGroupBackwardPlan``):

- straight-through backward ``dq[i, j] = dy[i, j] * scale[i, j / group_size]``;
- tensors are rank 2: ``dy`` and ``dq`` are ``[outer, axis_size]``, ``scale``
  is ``[outer, axis_size / group_size]`` (groups run along the last axis);
- gradients are f32, f64, f16 or bf16; ``axis_size % group_size == 0``,
  ``group_size > 0``, non-negative sizes; an empty problem is a no-op;
- deterministic and bit-stable.

Readings where the page is silent:

- the product is rounded once, to nearest-even, to the gradient's type. For
  f16 and bf16 operands the product is exact in f32 and f64, so this is also
  what computing in f32 and rounding gives.
- forward (the plan is named but not shown): ``out[i, j] = T(q[i, j]) *
  scale[i, j / group_size]`` for ``q`` int8 or uint8 (the page's ``TOut``), no
  zero point, rounded once to ``T``.
"""
import numpy as np

FLOAT_TYPES = ("f32", "f64", "f16", "bf16")
INT_TYPES = ("s8", "u8")


def rn_bf16_bits(v) -> np.ndarray:
    """Round float64 values to bfloat16 (nearest, ties to even) and return the
    16-bit patterns. bfloat16 is the top half of a binary32 with 8 significand
    bits; the values passed here are exact in binary32, so rounding the
    binary32 pattern's low 16 bits is the single rounding of the exact value.
    """
    f = np.asarray(v, dtype=np.float64).astype(np.float32)
    if not np.array_equal(f.astype(np.float64), np.asarray(v, dtype=np.float64), equal_nan=True):
        raise ValueError("rn_bf16_bits expects values exact in binary32")
    u = f.view(np.uint32).astype(np.uint64)
    is_nan = np.isnan(f)
    lower = u & 0xFFFF
    upper = u >> 16
    half = 0x8000
    round_up = (lower > half) | ((lower == half) & ((upper & 1) == 1))
    out = (upper + round_up.astype(np.uint64)) & 0xFFFF
    out = np.where(is_nan, (upper | 0x40) & 0xFFFF, out)   # keep NaN a (quiet) NaN
    return out.astype(np.uint16)


def bf16_to_f64(bits) -> np.ndarray:
    """Value of bfloat16 bit patterns."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def to_f64(a, dtype: str) -> np.ndarray:
    """Values of an array stored as ``dtype`` (bf16 given as uint16 patterns)."""
    if dtype == "bf16":
        return bf16_to_f64(a)
    return np.asarray(a).astype(np.float64)


def round_to(v, dtype: str) -> np.ndarray:
    """Round exact float64 values once to ``dtype`` (bf16 as uint16 patterns)."""
    v = np.asarray(v, dtype=np.float64)
    if dtype == "f64":
        return v.copy()
    if dtype == "f32":
        return v.astype(np.float32)
    if dtype == "f16":
        return v.astype(np.float16)
    if dtype == "bf16":
        return rn_bf16_bits(v)
    raise ValueError(f"unsupported type {dtype}")


def _expand_scale(scale64: np.ndarray, axis: int, group: int) -> np.ndarray:
    outer, ng = scale64.shape
    if group <= 0 or axis % group != 0 or ng != axis // group:
        raise ValueError("scale must be [outer, axis / group] with group > 0 dividing axis")
    # column j of the result takes scale column j // group
    idx = np.arange(axis) // group
    return scale64[:, idx]


def dequantize_per_group_backward_ref(dy, scale, group: int, dtype: str):
    """dq[i, j] = RN_dtype(dy[i, j] * scale[i, j // group])."""
    dy64 = to_f64(dy, dtype)
    sc64 = to_f64(scale, dtype)
    outer, axis = dy64.shape
    prod = dy64 * _expand_scale(sc64, axis, group)
    if dtype == "f64":
        return prod   # one float64 multiply, rounded once by the hardware
    return round_to(prod, dtype)   # exact for f32, f16, bf16 operands


def dequantize_per_group_ref(q, scale, group: int, dtype: str):
    """out[i, j] = RN_dtype(q[i, j] * scale[i, j // group]), q int8 or uint8."""
    q = np.asarray(q)
    if q.dtype not in (np.int8, np.uint8):
        raise ValueError("q must be int8 or uint8")
    sc64 = to_f64(scale, dtype)
    outer, axis = q.shape
    prod = q.astype(np.float64) * _expand_scale(sc64, axis, group)
    if dtype == "f64":
        return prod
    return round_to(prod, dtype)
