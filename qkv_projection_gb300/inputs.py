"""Seeded synthetic inputs for the W4A16 / W8A16 QKV projections, the dense f16
matmul and the per-group dequantisation.

This module only draws random numbers. It holds none of the method's
arithmetic: packed weights are drawn as uniformly random 32-bit words, which is
the same thing as drawing the eight 4-bit fields of each word independently and
uniformly (every 4-bit pattern, i.e. every signed value in [-8, 7], is equally
likely). Unpacking, dequantisation and the products live elsewhere.

Distributions (workload shapes of the W4A16 projection and the dense matmul):

- ``x``: f16, standard normal, rounded to f16 by the dtype cast.
- ``wq``/``wk``/``wv``: uint32 ``[K/8, N]``, uniform over all 2**32 words.
- ``sq``/``sk``/``sv``: f16 ``[K/128, N]``, uniform in [0.005, 0.02].
- W8A16 (``qkv_int8_inputs``): ``x`` as above; packed ``u32[K/4, N]`` words
  uniform over all 2**32 words (every int8 byte equally likely); the three
  per-projection f32 scales uniform in [5e-4, 2e-3].
- dense ``a``/``b``: f16, uniform in [-1, 1]; backward ``g``: f16 standard normal.

One ``numpy.random.Generator`` (PCG64) per call, seeded by ``seed``; tensors
are drawn in the fixed order x, wq, wk, wv, sq, sk, sv.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

GROUP_SIZE = 128


@dataclass
class QKVInputs:
    x: np.ndarray   # f16 [M, K]
    wq: np.ndarray  # u32 [K/8, N]
    wk: np.ndarray
    wv: np.ndarray
    sq: np.ndarray  # f16 [K/128, N]
    sk: np.ndarray
    sv: np.ndarray

    @property
    def shape(self):
        m, k = self.x.shape
        return m, self.wq.shape[1], k

    def weights(self):
        return (self.wq, self.wk, self.wv)

    def scales(self):
        return (self.sq, self.sk, self.sv)


def qkv_inputs(m: int, n: int, k: int, seed: int = 0,
               scale_lo: float = 0.005, scale_hi: float = 0.02) -> QKVInputs:
    """Draw one W4A16 problem of shape (M, N, K)."""
    if k % GROUP_SIZE:
        raise ValueError(f"K={k} is not a multiple of {GROUP_SIZE}")
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((m, k), dtype=np.float32).astype(np.float16)
    w = [rng.integers(0, 2**32, size=(k // 8, n), dtype=np.uint32) for _ in range(3)]
    s = [rng.uniform(scale_lo, scale_hi, size=(k // GROUP_SIZE, n)).astype(np.float16)
         for _ in range(3)]
    return QKVInputs(x, w[0], w[1], w[2], s[0], s[1], s[2])


def weight_sets(n: int, k: int, count: int, seed: int = 1):
    """``count`` distinct (wq, wk, wv, sq, sk, sv) sets, used to rotate weights
    between timed launches so that every launch streams its weights from HBM."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(count):
        w = [rng.integers(0, 2**32, size=(k // 8, n), dtype=np.uint32) for _ in range(3)]
        s = [rng.uniform(0.005, 0.02, size=(k // GROUP_SIZE, n)).astype(np.float16)
             for _ in range(3)]
        out.append((*w, *s))
    return out


@dataclass
class QKV8Inputs:
    x: np.ndarray   # f16 [M, K]
    wq: np.ndarray  # u32 [K/4, N]
    wk: np.ndarray
    wv: np.ndarray
    sq: float       # f32 scale of each projection
    sk: float
    sv: float

    def weights(self):
        return (self.wq, self.wk, self.wv)

    def scales(self):
        return (self.sq, self.sk, self.sv)

    def args(self):
        return (self.x, self.wq, self.wk, self.wv, self.sq, self.sk, self.sv)


def qkv_int8_inputs(m: int, n: int, k: int, seed: int = 0) -> QKV8Inputs:
    """Draw one W8A16 problem of shape (M, N, K); x, wq, wk, wv, sq, sk, sv in order."""
    if k % 4:
        raise ValueError(f"K={k} is not a multiple of 4")
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((m, k), dtype=np.float32).astype(np.float16)
    w = [rng.integers(0, 2**32, size=(k // 4, n), dtype=np.uint32) for _ in range(3)]
    s = [float(np.float32(rng.uniform(5e-4, 2e-3))) for _ in range(3)]
    return QKV8Inputs(x, w[0], w[1], w[2], s[0], s[1], s[2])


def weight_sets_int8(n: int, k: int, count: int, seed: int = 1):
    """``count`` distinct packed (wq, wk, wv) INT8 weight sets (rotated between
    timed launches so that every launch streams its weights from HBM)."""
    rng = np.random.default_rng(seed)
    return [tuple(rng.integers(0, 2**32, size=(k // 4, n), dtype=np.uint32) for _ in range(3))
            for _ in range(count)]


def dense_inputs(m: int, n: int, k: int, seed: int = 0):
    """A f16[M,K], B f16[K,N] uniform in [-1,1] and G f16[M,N] ~ N(0,1)."""
    rng = np.random.default_rng(seed)
    a = rng.uniform(-1.0, 1.0, size=(m, k)).astype(np.float16)
    b = rng.uniform(-1.0, 1.0, size=(k, n)).astype(np.float16)
    g = rng.standard_normal((m, n), dtype=np.float32).astype(np.float16)
    return a, b, g


def dequant_group_inputs(outer: int, axis: int, group: int, dtype: str, seed: int = 0, q_dtype: str = "s8"):
    """Seeded inputs of the per-group dequantisation and its backward.

    Returns (dy, q, scale) as numpy arrays: dy [outer, axis] and scale
    [outer, axis // group] in ``dtype`` (bf16 as uint16 bit patterns: the upper
    half of a float32 draw), dy ~ N(0, 1), scale uniform in [0.005, 0.02];
    q [outer, axis] uniform over all int8 (or uint8) values.
    """
    rng = np.random.default_rng(seed)
    dy = rng.standard_normal((outer, axis))
    sc = rng.uniform(0.005, 0.02, size=(outer, axis // group))
    qd = np.int8 if q_dtype == "s8" else np.uint8
    info = np.iinfo(qd)
    q = rng.integers(info.min, info.max + 1, size=(outer, axis), dtype=np.int64).astype(qd)

    def cast(a):
        if dtype == "bf16":
            return (a.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        return a.astype({"f32": np.float32, "f64": np.float64, "f16": np.float16}[dtype])

    return cast(dy), q, cast(sc)
