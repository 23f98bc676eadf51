"""Pins for the per-group dequantisation oracle (CPU only).

Each expected value is written by hand from the definitions (exact products,
binary16 / bfloat16 round-to-nearest-even), or checked against independent
exact rational arithmetic.
"""
from fractions import Fraction

import numpy as np
import pytest

from oracle import dequant_group as dg


def test_backward_hand_example_f32():
    # dq[i, j] = dy[i, j] * scale[i, j // 2]
    dy = np.array([[1, 2, 3, 4], [-1, 0.5, 8, -2]], dtype=np.float32)
    sc = np.array([[0.5, 2], [4, -0.25]], dtype=np.float32)
    got = dg.dequantize_per_group_backward_ref(dy, sc, 2, "f32")
    assert got.dtype == np.float32
    assert got.tolist() == [[0.5, 1.0, 6.0, 8.0], [-4.0, 2.0, -2.0, 0.5]]


def test_group_columns_closed_form():
    # with group 4 and axis 8, scale column g touches exactly columns 4g .. 4g+3
    dy = np.ones((3, 8), dtype=np.float64)
    sc = np.array([[1.0, 10.0]] * 3)
    got = dg.dequantize_per_group_backward_ref(dy, sc, 4, "f64")
    assert got.tolist() == [[1.0] * 4 + [10.0] * 4] * 3


def test_f16_product_rounding_hand_value():
    # (1 + 2^-10)^2 = 1 + 2^-9 + 2^-20: nearest binary16 is 1 + 2^-9
    v = np.array([[1 + 2 ** -10]], dtype=np.float16)
    got = dg.dequantize_per_group_backward_ref(v, v, 1, "f16")
    assert got.dtype == np.float16 and float(got[0, 0]) == 1 + 2 ** -9


@pytest.mark.parametrize("value,bits", [
    (1.0, 0x3F80),
    (-1.5, 0xBFC0),
    (1 + 2 ** -8, 0x3F80),             # tie between 0x3F80 and 0x3F81: even is 0x3F80
    (1 + 3 * 2 ** -8, 0x3F82),         # tie between 0x3F81 and 0x3F82: even is 0x3F82
    (1 + 2 ** -8 + 2 ** -20, 0x3F81),  # just above the tie: up
    (2.0 ** -133, 0x0001),             # the smallest subnormal, 2^-126 * 2^-7
    (2.0 ** -134, 0x0000),             # half of it: a tie between 0 and 0x0001, even is 0
    (3.0 * 2 ** -135, 0x0001),         # three quarters of it: up
    (3.0 * 2 ** -134, 0x0002),         # 1.5 times it: a tie between 0x0001 and 0x0002, even
])
def test_bf16_rounding_hand_patterns(value, bits):
    assert int(dg.rn_bf16_bits(np.array([value]))[0]) == bits


def test_bf16_product_hand_value():
    # bf16 0x3F81 = 1 + 2^-7; its square 1.01568603515625 is nearest to 1 + 2^-6 (0x3F82)
    b = np.array([[0x3F81]], dtype=np.uint16)
    got = dg.dequantize_per_group_backward_ref(b, b, 1, "bf16")
    assert int(got[0, 0]) == 0x3F82
    assert dg.bf16_to_f64(got)[0, 0] == 1 + 2 ** -6


def test_forward_hand_examples():
    q = np.array([[-128, 127, 0, 5]], dtype=np.int8)
    sc = np.array([[0.5, 0.25]], dtype=np.float16)
    assert dg.dequantize_per_group_ref(q, sc, 2, "f16").astype(np.float64).tolist() == [[-64, 63.5, 0, 1.25]]
    qu = np.array([[0, 255, 128, 1]], dtype=np.uint8)
    scu = np.array([[2.0, 0.5]], dtype=np.float32)
    assert dg.dequantize_per_group_ref(qu, scu, 2, "f32").tolist() == [[0.0, 510.0, 64.0, 0.5]]


def _rne_binary16(fr: Fraction) -> Fraction:
    """Round an exact rational to binary16 (normal range), nearest, ties to even,
    from the format's definition: 11 significand bits."""
    if fr == 0:
        return Fraction(0)
    sign = -1 if fr < 0 else 1
    a = abs(fr)
    e = 0
    while a >= 2:
        a /= 2
        e += 1
    while a < 1:
        a *= 2
        e -= 1
    scaled = a * 1024                      # 10 fraction bits
    lo = scaled.numerator // scaled.denominator
    rem = scaled - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    return sign * Fraction(lo, 1024) * Fraction(2) ** e


def test_f16_backward_matches_exact_rationals():
    rng = np.random.default_rng(5)
    dy = rng.uniform(-4, 4, size=(3, 12)).astype(np.float16)
    sc = rng.uniform(0.01, 3, size=(3, 3)).astype(np.float16)
    got = dg.dequantize_per_group_backward_ref(dy, sc, 4, "f16")
    for i in range(3):
        for j in range(12):
            exact = Fraction(float(dy[i, j])) * Fraction(float(sc[i, j // 4]))
            assert Fraction(float(got[i, j])) == _rne_binary16(exact), (i, j)


def test_mistakes_are_caught():
    """Plausible mistakes, each applied to a pinned input, fail that pin."""
    dy = np.array([[1, 2, 3, 4], [-1, 0.5, 8, -2]], dtype=np.float32)
    sc = np.array([[0.5, 2], [4, -0.25]], dtype=np.float32)
    good = [[0.5, 1.0, 6.0, 8.0], [-4.0, 2.0, -2.0, 0.5]]
    # group index j % num_groups instead of j // group
    wrong_group = (dy.astype(np.float64) * sc[:, np.arange(4) % 2]).astype(np.float32)
    assert wrong_group.tolist() != good
    # every row using the first row's scales
    wrong_row = (dy.astype(np.float64) * sc[0, np.arange(4) // 2]).astype(np.float32)
    assert wrong_row.tolist() != good

    def bf16_truncate(v):
        return (np.asarray(v, np.float64).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)

    def bf16_ties_away(v):
        u = np.asarray(v, np.float64).astype(np.float32).view(np.uint32).astype(np.uint64)
        return (((u + 0x8000) >> 16) & 0xFFFF).astype(np.uint16)

    assert int(bf16_truncate([1 + 2 ** -8 + 2 ** -20])[0]) != 0x3F81          # pinned: 0x3F81
    assert int(bf16_ties_away([1 + 2 ** -8])[0]) != 0x3F80                    # pinned: 0x3F80
    assert int(dg.rn_bf16_bits(np.array([1 + 2 ** -8 + 2 ** -20]))[0]) == 0x3F81
    assert int(dg.rn_bf16_bits(np.array([1 + 2 ** -8]))[0]) == 0x3F80


def test_rejects_bad_group_and_shapes():
    with pytest.raises(ValueError):
        dg.dequantize_per_group_backward_ref(np.zeros((2, 6), np.float32), np.zeros((2, 2), np.float32), 4, "f32")
    with pytest.raises(ValueError):
        dg.dequantize_per_group_backward_ref(np.zeros((2, 4), np.float32), np.zeros((2, 2), np.float32), 0, "f32")
    with pytest.raises(ValueError):
        dg.dequantize_per_group_ref(np.zeros((1, 4), np.int16), np.zeros((1, 2), np.float32), 2, "f32")
