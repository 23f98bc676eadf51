"""Pins for the CPU oracle (no GPU).

The oracle is checked against facts that do not come from it:
hand-written bit patterns (tests/golden), exact rational arithmetic on tiny
problems (pure-Python ints and fractions.Fraction, with an f16 rounding written
here from the IEEE 754 binary16 definition), identity / one-hot / scale-doubling
closed forms and the transpose identities of the matmul backward.

Each pin is written as a check function that takes an oracle implementation, so
the same check is also run against deliberately broken copies of the oracle
(wrong nibble order, unsigned nibbles, wrong group index, no dequant rounding,
transposed weights): a pin that cannot tell them apart is no pin.
"""
import math
import os
from fractions import Fraction
from types import SimpleNamespace

import numpy as np
import pytest

import oracle
from oracle import w4a16 as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# Independent exact arithmetic (pure Python), written from the definitions.
# --------------------------------------------------------------------------

def rne_f16_exact(q: Fraction):
    """Round a rational to the nearest binary16 value, ties to even.

    Returns a Fraction, or +/-inf (float) on overflow. Binary16 has 11
    significant bits; normal exponents -14..15, subnormal quantum 2**-24.
    """
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -14)
    quantum = Fraction(2) ** (e - 10)
    m = a / quantum
    lo = m.numerator // m.denominator
    rem = m - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    r = lo * quantum
    if r >= 65536:
        return sign * math.inf
    return sign * r


def nibble_signed(word: int, i: int) -> int:
    v = (word >> (4 * i)) & 0xF
    return v - 16 if v >= 8 else v


def brute_qkv_exact(x, packed, scales):
    """Exact sum_k x[m,k] * RN_f16(w[k,n] * s[k//128, n]) as Fractions."""
    m_rows, k = x.shape
    n_cols = packed.shape[1]
    out = [[Fraction(0)] * n_cols for _ in range(m_rows)]
    for n in range(n_cols):
        wd = []
        for kk in range(k):
            w = nibble_signed(int(packed[kk // 8, n]), kk % 8)
            s = Fraction(float(scales[kk // 128, n]))
            wd.append(rne_f16_exact(w * s))
        for m in range(m_rows):
            acc = Fraction(0)
            for kk in range(k):
                acc += Fraction(float(x[m, kk])) * wd[kk]
            out[m][n] = acc
    return out


# --------------------------------------------------------------------------
# Broken copies of the oracle, to show the pins are discriminating.
# --------------------------------------------------------------------------

def _unpack_reversed(p):
    p = np.asarray(p, dtype=np.uint32)
    out = np.empty((p.shape[0] * 8, p.shape[1]), dtype=np.int8)
    for i in range(8):
        nib = ((p >> np.uint32(4 * (7 - i))) & np.uint32(0xF)).astype(np.int16)
        out[i::8] = np.where(nib >= 8, nib - 16, nib)
    return out


def _unpack_unsigned(p):
    p = np.asarray(p, dtype=np.uint32)
    out = np.empty((p.shape[0] * 8, p.shape[1]), dtype=np.int16)
    for i in range(8):
        out[i::8] = ((p >> np.uint32(4 * i)) & np.uint32(0xF)).astype(np.int16)
    return out


def _make_variant(name):
    """A namespace with the oracle's API and one planted mistake."""
    unpack = W.unpack_int4
    if name == "reversed_nibbles":
        unpack = _unpack_reversed
    elif name == "unsigned_nibbles":
        unpack = _unpack_unsigned

    def dequant(packed, scales):
        w = unpack(packed).astype(np.float64)
        s = np.asarray(scales, dtype=np.float16).astype(np.float64)
        k = w.shape[0]
        if name == "group_mod":
            rows = s[np.arange(k) % s.shape[0]]
        else:
            rows = np.repeat(s, 128, axis=0)
        prod = w * rows
        if name == "no_dequant_rounding":
            return prod
        return W.rn_f16(prod)

    def qkv(x, wq, wk, wv, sq, sk, sv):
        x64 = np.asarray(x, dtype=np.float16).astype(np.float64)
        outs = []
        for w, s in ((wq, sq), (wk, sk), (wv, sv)):
            wd = np.asarray(dequant(w, s), dtype=np.float64)
            if name == "transposed_weights":
                wd = wd.T if wd.shape[0] == wd.shape[1] else wd[::-1]
            outs.append(x64 @ wd)
        return tuple(outs)

    return SimpleNamespace(unpack_int4=unpack, dequant_int4=dequant, qkv_project_int4_ref=qkv)


REAL = SimpleNamespace(unpack_int4=W.unpack_int4, dequant_int4=W.dequant_int4,
                       qkv_project_int4_ref=W.qkv_project_int4_ref)
MUTANTS = ["reversed_nibbles", "unsigned_nibbles", "group_mod",
           "no_dequant_rounding", "transposed_weights"]


# --------------------------------------------------------------------------
# Pin checks (each returns True when the implementation satisfies the pin).
# --------------------------------------------------------------------------

def _golden_nibbles():
    rows = []
    with open(os.path.join(GOLDEN, "int4_nibbles.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            word, vals = line.split(":")
            rows.append((int(word, 16), [int(v) for v in vals.split()]))
    return rows


def check_golden_nibbles(impl) -> bool:
    for word, vals in _golden_nibbles():
        got = impl.unpack_int4(np.array([[word]], dtype=np.uint32))[:, 0]
        if list(map(int, got)) != vals:
            return False
    return True


def check_brute_force(impl, shapes=((1, 8, 128), (3, 8, 256), (2, 16, 128)), seed=7) -> bool:
    from qkv_projection_gb300.inputs import qkv_inputs
    for (m, n, k) in shapes:
        # scales spanning two binades so that RN_f16(w*s) really rounds
        inp = qkv_inputs(m, n, k, seed=seed, scale_lo=0.003, scale_hi=0.03)
        refs = impl.qkv_project_int4_ref(*inp.__dict__.values())
        for ref, packed, scales in zip(refs, inp.weights(), inp.scales()):
            exact = brute_qkv_exact(inp.x, packed, scales)
            ex = np.array([[float(v) for v in row] for row in exact])
            bound = 1e-12 * max(1.0, np.abs(ex).max())
            if not np.all(np.abs(np.asarray(ref) - ex) <= bound):
                return False
    return True


def check_one_hot(impl) -> bool:
    m, n, k = 4, 16, 256
    rng = np.random.default_rng(3)
    x = rng.standard_normal((m, k)).astype(np.float16)
    k0, n0, c = 130, 5, -7             # K-row 130 lies in group 1, nibble 2 of row 16
    w = np.zeros((k, n), dtype=np.int8)
    w[k0, n0] = c
    packed = W.pack_int4(w)
    s = np.full((k // 128, n), 0.25, dtype=np.float16)
    s[1, n0] = np.float16(0.0123)     # c*s is not an f16 number: the dequant rounds
    zero_p = np.zeros_like(packed)
    refs = impl.qkv_project_int4_ref(x, packed, zero_p, zero_p, s, s, s)
    wd = rne_f16_exact(c * Fraction(float(s[1, n0])))
    expect = np.zeros((m, n))
    expect[:, n0] = [float(Fraction(float(v)) * wd) for v in x[:, k0]]
    return (np.array_equal(np.asarray(refs[0]), expect)
            and not np.any(refs[1]) and not np.any(refs[2]))


def check_identity(impl) -> bool:
    k = n = 256
    rng = np.random.default_rng(4)
    x = rng.standard_normal((5, k)).astype(np.float16)
    packed = W.pack_int4(np.eye(k, dtype=np.int8))
    s = np.ones((k // 128, n), dtype=np.float16)
    q, _, _ = impl.qkv_project_int4_ref(x, packed, packed, packed, s, s, s)
    return np.array_equal(np.asarray(q), x.astype(np.float64))


def check_scale_doubling(impl) -> bool:
    m, n, k = 3, 8, 384
    from qkv_projection_gb300.inputs import qkv_inputs
    inp = qkv_inputs(m, n, k, seed=11)
    g, col = 1, 6
    s2 = inp.sq.copy()
    s2[g, col] = s2[g, col] * np.float16(2)       # exact in f16
    base = impl.qkv_project_int4_ref(inp.x, inp.wq, inp.wq, inp.wq, inp.sq, inp.sq, inp.sq)[0]
    dbl = impl.qkv_project_int4_ref(inp.x, inp.wq, inp.wq, inp.wq, s2, s2, s2)[0]
    # exactly that group's contribution, computed with exact rationals
    contrib = []
    for r in range(m):
        acc = Fraction(0)
        for kk in range(g * 128, (g + 1) * 128):
            wv = nibble_signed(int(inp.wq[kk // 8, col]), kk % 8)
            acc += Fraction(float(inp.x[r, kk])) * rne_f16_exact(wv * Fraction(float(inp.sq[g, col])))
        contrib.append(float(acc))
    diff = np.asarray(dbl) - np.asarray(base)
    others = np.delete(diff, col, axis=1)
    tol = 1e-12 * max(1.0, np.abs(np.asarray(base)).max())
    return (np.all(np.abs(others) == 0)
            and np.all(np.abs(diff[:, col] - np.array(contrib)) <= tol))


PINS = [check_golden_nibbles, check_brute_force, check_one_hot, check_identity,
        check_scale_doubling]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_oracle_satisfies_pin(pin):
    assert pin(REAL)


@pytest.mark.parametrize("mutant", MUTANTS)
def test_pins_reject_planted_mistake(mutant):
    impl = _make_variant(mutant)
    failed = [p.__name__ for p in PINS if not p(impl)]
    assert failed, f"no pin detects the planted mistake {mutant!r}"


# --------------------------------------------------------------------------
# Direct pins of the individual pieces.
# --------------------------------------------------------------------------

def test_golden_words_pack_back():
    for word, vals in _golden_nibbles():
        packed = oracle.pack_int4(np.array(vals, dtype=np.int8).reshape(8, 1))
        assert int(packed[0, 0]) == word


def test_pack_roundtrip_every_value_every_position():
    for v in range(-8, 8):
        for i in range(8):
            w = np.zeros((8, 1), dtype=np.int8)
            w[i, 0] = v
            p = oracle.pack_int4(w)
            assert int(p[0, 0]) == (v & 0xF) << (4 * i)
            assert np.array_equal(oracle.unpack_int4(p), w)


def test_unpack_is_a_bijection_on_random_words():
    rng = np.random.default_rng(5)
    p = rng.integers(0, 2**32, size=(64, 40), dtype=np.uint32)
    w = oracle.unpack_int4(p)
    assert w.min() >= -8 and w.max() <= 7
    assert np.array_equal(oracle.pack_int4(w), p)


def test_pack_rejects_out_of_range():
    with pytest.raises(ValueError):
        oracle.pack_int4(np.full((8, 1), 8))
    with pytest.raises(ValueError):
        oracle.pack_int4(np.full((7, 1), 0))


def test_rn_f16_golden_and_exact_rounding_agree():
    with open(os.path.join(GOLDEN, "f16_rounding.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            val, bits = line.split(":")
            v = float.fromhex(val.strip())
            want = int(bits, 16)
            got = int(oracle.rn_f16(np.array([v])).view(np.uint16)[0])
            assert got == want, (val, hex(got), hex(want))
            ex = rne_f16_exact(Fraction(v))
            if want == 0x7C00:
                assert ex == math.inf
            else:
                assert float(ex) == float(np.array([want], dtype=np.uint16).view(np.float16)[0])


def test_ulp_f16_closed_forms():
    cases = {1.0: 2.0**-10, 1.5: 2.0**-10, 2.0: 2.0**-9, 0.0: 2.0**-24,
             6e-5: 2.0**-24, 2.0**-14: 2.0**-24, 65504.0: 32.0, -3.0: 2.0**-9,
             np.nextafter(2.0, 0.0): 2.0**-10}
    for v, u in cases.items():
        assert float(oracle.ulp_f16(v)) == u, v


def test_dequant_matches_exact_rounding():
    rng = np.random.default_rng(6)
    k, n = 256, 12
    p = rng.integers(0, 2**32, size=(k // 8, n), dtype=np.uint32)
    s = rng.uniform(0.001, 3.0, size=(k // 128, n)).astype(np.float16)
    wd = oracle.dequant_int4(p, s)
    assert wd.dtype == np.float16
    for kk in range(k):
        for c in range(n):
            e = rne_f16_exact(nibble_signed(int(p[kk // 8, c]), kk % 8) * Fraction(float(s[kk // 128, c])))
            assert float(wd[kk, c]) == float(e)


def test_group_boundaries_closed_form():
    # every nibble 1, group 0 scale 1 and group 1 scale 2:
    # ref[m, n] = sum_{k<128} x[m,k] + 2 * sum_{128<=k<256} x[m,k]
    k, n = 256, 8
    x = np.arange(2 * k, dtype=np.float64).reshape(2, k).astype(np.float16) / np.float16(64)
    packed = oracle.pack_int4(np.ones((k, n), dtype=np.int8))
    s = np.ones((2, n), dtype=np.float16)
    s[1] = 2
    q, _, _ = oracle.qkv_project_int4_ref(x, packed, packed, packed, s, s, s)
    xs = x.astype(np.float64)
    want = xs[:, :128].sum(axis=1) + 2 * xs[:, 128:].sum(axis=1)
    assert np.array_equal(q, np.repeat(want[:, None], n, axis=1))


def test_library_matmul_matches_plain_loop():
    rng = np.random.default_rng(8)
    a = rng.uniform(-1, 1, size=(5, 33)).astype(np.float16)
    b = rng.uniform(-1, 1, size=(33, 7)).astype(np.float16)
    c = oracle.matmul_ref(a, b)
    for i in range(5):
        for j in range(7):
            exact = sum(Fraction(float(a[i, t])) * Fraction(float(b[t, j])) for t in range(33))
            assert abs(c[i, j] - float(exact)) <= 1e-12


def test_matmul_backward_identities():
    rng = np.random.default_rng(9)
    n = 24
    g = rng.standard_normal((n, n)).astype(np.float16)
    b = rng.uniform(-1, 1, size=(n, n)).astype(np.float16)
    eye = np.eye(n, dtype=np.float16)
    d_a, d_b = oracle.matmul_backward_ref(eye, b, g)      # A = I  ->  dB = G
    assert np.array_equal(d_b, g.astype(np.float64))
    d_a, d_b = oracle.matmul_backward_ref(b, eye, g)      # B = I  ->  dA = G
    assert np.array_equal(d_a, g.astype(np.float64))
    # non-square shapes: dA is [M, K] and dB is [K, N]
    a = rng.uniform(-1, 1, size=(6, 10)).astype(np.float16)
    b = rng.uniform(-1, 1, size=(10, 4)).astype(np.float16)
    g = rng.standard_normal((6, 4)).astype(np.float16)
    d_a, d_b = oracle.matmul_backward_ref(a, b, g)
    assert d_a.shape == (6, 10) and d_b.shape == (10, 4)
    exact = sum(Fraction(float(g[2, j])) * Fraction(float(b[3, j])) for j in range(4))
    assert abs(d_a[2, 3] - float(exact)) <= 1e-12


def test_sampled_rows_equal_full_reference():
    from qkv_projection_gb300.inputs import qkv_inputs
    inp = qkv_inputs(20, 16, 256, seed=2)
    full = oracle.qkv_project_int4_ref(*inp.__dict__.values())
    rows = [0, 3, 19]
    part = oracle.qkv_project_int4_rows(*inp.__dict__.values(), rows)
    for f, p in zip(full, part):
        assert np.array_equal(f[rows], p)
