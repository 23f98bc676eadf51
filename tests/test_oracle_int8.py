"""Pins for the W8A16 oracle (no GPU).

Checked against facts that do not come from the oracle: hand-written words
(tests/golden/int8_bytes.txt), exact rational arithmetic on tiny problems,
one-hot / identity closed forms and exact power-of-two scale relations. Each
pin is a check function run against the oracle and against copies of it with
one planted mistake; every mistake must fail at least one pin.
"""
import os
from fractions import Fraction
from types import SimpleNamespace

import numpy as np
import pytest

import oracle
from oracle import w8a16 as W8
from qkv_projection_gb300.inputs import qkv_int8_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def byte_signed(word: int, i: int) -> int:
    v = (word >> (8 * i)) & 0xFF
    return v - 256 if v >= 128 else v


def brute_exact(x, packed, scale):
    """sum_k x[m,k] * (s * w[k,n]) as exact Fractions (pure Python)."""
    m_rows, k = x.shape
    s = Fraction(float(np.float32(scale)))
    out = []
    for m in range(m_rows):
        row = []
        for n in range(packed.shape[1]):
            acc = Fraction(0)
            for kk in range(k):
                acc += Fraction(float(x[m, kk])) * s * byte_signed(int(packed[kk // 4, n]), kk % 4)
            row.append(acc)
        out.append(row)
    return out


# --------------------------------------------------------------------------
# Copies of the oracle with one planted mistake each.
# --------------------------------------------------------------------------

def _make_variant(name):
    def unpack(p):
        p = np.asarray(p, dtype=np.uint32)
        rows, n = p.shape
        out = np.empty((rows * 4, n), dtype=np.int16)
        for i in range(4):
            shift = 8 * (3 - i) if name == "reversed_bytes" else 8 * i
            b = ((p >> np.uint32(shift)) & np.uint32(0xFF)).astype(np.int16)
            v = b if name == "unsigned_bytes" else np.where(b >= 128, b - 256, b)
            if name == "planar_rows":            # K-row i*(K/4) + r instead of 4r + i
                out[i * rows:(i + 1) * rows] = v
            else:
                out[i::4] = v
        return out

    def qkv(x, wq, wk, wv, sq, sk, sv):
        x64 = np.asarray(x, dtype=np.float16).astype(np.float64)
        outs = []
        for w, s in ((wq, sq), (wk, sk), (wv, sv)):
            if name == "no_scale":
                s = 1.0
            elif name == "first_scale_for_all":
                s = sq
            wd = unpack(w).astype(np.float64) * float(np.float32(s))
            if name == "transposed_weights":
                wd = wd.T if wd.shape[0] == wd.shape[1] else wd[::-1]
            outs.append(x64 @ wd)
        return tuple(outs)

    return SimpleNamespace(unpack_int8=unpack, qkv_project_int8_ref=qkv)


REAL = SimpleNamespace(unpack_int8=W8.unpack_int8, qkv_project_int8_ref=W8.qkv_project_int8_ref)
MUTANTS = ["reversed_bytes", "unsigned_bytes", "planar_rows", "no_scale", "first_scale_for_all",
           "transposed_weights"]


def _golden_words():
    rows = []
    with open(os.path.join(GOLDEN, "int8_bytes.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            word, vals = line.split(":")
            rows.append((int(word, 16), [int(v) for v in vals.split()]))
    return rows


def check_golden_bytes(impl) -> bool:
    for word, vals in _golden_words():
        if list(map(int, impl.unpack_int8(np.array([[word]], dtype=np.uint32))[:, 0])) != vals:
            return False
    return True


def check_brute_force(impl, shapes=((1, 6, 16), (3, 5, 24), (2, 4, 128)), seed=7) -> bool:
    for (m, n, k) in shapes:
        inp = qkv_int8_inputs(m, n, k, seed=seed)
        refs = impl.qkv_project_int8_ref(*inp.args())
        for ref, packed, s in zip(refs, inp.weights(), inp.scales()):
            ex = np.array([[float(v) for v in row] for row in brute_exact(inp.x, packed, s)])
            if not np.all(np.abs(np.asarray(ref) - ex) <= 1e-12 * max(1.0, np.abs(ex).max())):
                return False
    return True


def check_one_hot(impl) -> bool:
    m, n, k = 3, 12, 64
    x = np.random.default_rng(3).standard_normal((m, k)).astype(np.float16)
    k0, n0, c = 42, 7, -77                     # K-row 42 = byte 2 of packed row 10
    w = np.zeros((k, n), dtype=np.int16)
    w[k0, n0] = c
    packed = W8.pack_int8(w)
    zero = np.zeros_like(packed)
    s = 0.0123                                 # any f32 value: s * c * x is exact in float64
    refs = impl.qkv_project_int8_ref(x, packed, zero, zero, s, s, s)
    expect = np.zeros((m, n))
    sf = Fraction(float(np.float32(s)))
    expect[:, n0] = [float(sf * c * Fraction(float(v))) for v in x[:, k0]]
    return np.array_equal(np.asarray(refs[0]), expect) and not np.any(refs[1]) and not np.any(refs[2])


def check_identity(impl) -> bool:
    k = n = 64
    x = np.random.default_rng(4).standard_normal((5, k)).astype(np.float16)
    packed = W8.pack_int8(np.eye(k, dtype=np.int16))
    q, _, _ = impl.qkv_project_int8_ref(x, packed, packed, packed, 1.0, 1.0, 1.0)
    return np.array_equal(np.asarray(q), x.astype(np.float64))


def check_projection_scales(impl) -> bool:
    # the same weights under scales 1, 2 and 0.5: k = 2 q and v = q / 2 exactly
    inp = qkv_int8_inputs(4, 8, 32, seed=9)
    q, k, v = impl.qkv_project_int8_ref(inp.x, inp.wq, inp.wq, inp.wq, 1.0, 2.0, 0.5)
    q, k, v = (np.asarray(a) for a in (q, k, v))
    return np.any(q) and np.array_equal(k, 2 * q) and np.array_equal(v, q / 2)


PINS = [check_golden_bytes, check_brute_force, check_one_hot, check_identity, check_projection_scales]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_oracle_satisfies_pin(pin):
    assert pin(REAL)


@pytest.mark.parametrize("mutant", MUTANTS)
def test_pins_reject_planted_mistake(mutant):
    impl = _make_variant(mutant)
    failed = [p.__name__ for p in PINS if not p(impl)]
    assert failed, f"no pin detects the planted mistake {mutant!r}"


def test_golden_words_pack_back():
    for word, vals in _golden_words():
        assert int(oracle.pack_int8(np.array(vals).reshape(4, 1))[0, 0]) == word


def test_pack_roundtrip_every_value_every_position():
    for v in range(-128, 128):
        for i in range(4):
            w = np.zeros((4, 1), dtype=np.int16)
            w[i, 0] = v
            p = oracle.pack_int8(w)
            assert int(p[0, 0]) == (v & 0xFF) << (8 * i)
            assert np.array_equal(oracle.unpack_int8(p), w)


def test_unpack_is_a_bijection_on_random_words():
    p = np.random.default_rng(5).integers(0, 2**32, size=(32, 20), dtype=np.uint32)
    w = oracle.unpack_int8(p)
    assert w.dtype == np.int8
    assert np.array_equal(oracle.pack_int8(w), p)


def test_pack_rejects_out_of_range_and_ragged_k():
    with pytest.raises(ValueError):
        oracle.pack_int8(np.full((4, 1), 128))
    with pytest.raises(ValueError):
        oracle.pack_int8(np.full((4, 1), -129))
    with pytest.raises(ValueError):
        oracle.pack_int8(np.zeros((6, 1)))


def test_dequant_is_the_exact_product():
    p = np.random.default_rng(6).integers(0, 2**32, size=(8, 5), dtype=np.uint32)
    s = 0.000987654
    wd = oracle.dequant_int8(p, s)
    sf = Fraction(float(np.float32(s)))
    for kk in range(32):
        for c in range(5):
            assert Fraction(float(wd[kk, c])) == sf * byte_signed(int(p[kk // 4, c]), kk % 4)


def test_sampled_rows_equal_full_reference():
    inp = qkv_int8_inputs(12, 8, 64, seed=2)
    full = oracle.qkv_project_int8_ref(*inp.args())
    rows = [0, 5, 11]
    for f, p in zip(full, oracle.qkv_project_int8_rows(*inp.args(), rows)):
        assert np.array_equal(f[rows], p)


def test_rejects_mismatched_k():
    inp = qkv_int8_inputs(2, 4, 16, seed=1)
    with pytest.raises(ValueError):
        oracle.qkv_project_int8_ref(inp.x[:, :12], *inp.args()[1:])
