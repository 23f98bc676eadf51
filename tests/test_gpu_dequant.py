"""Dequantised weights must equal the oracle's bit for bit (GPU)."""
import numpy as np
import pytest

import oracle
from qkv_projection_gb300 import kaio
from qkv_projection_gb300.inputs import qkv_inputs

from gpu_helpers import to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("variant", [0, 1, 2])
@pytest.mark.parametrize("k,n", [(128, 8), (256, 40), (1024, 264), (4096, 4096)])
def test_dequant_bit_exact(variant, k, n):
    inp = qkv_inputs(1, n, k, seed=k + n)
    got = to_host(kaio.dequant_int4_debug(to_dev(inp.wq), to_dev(inp.sq), variant))
    want = oracle.dequant_int4(inp.wq, inp.sq)
    assert np.array_equal(got.view(np.uint16), want.view(np.uint16))


@pytest.mark.parametrize("variant", [0, 1, 2])
def test_dequant_bit_exact_wide_scale_range(variant):
    # every nibble value against scales spanning the f16 range: subnormal
    # products, exact and inexact roundings, overflow to +/-inf, zero and
    # negative scales
    k, n = 128, 64
    rng = np.random.default_rng(1)
    # column c holds every value -8..7 along K, rotated by c
    w = np.tile(np.arange(-8, 8, dtype=np.int8).reshape(16, 1), (k // 16, n))
    w = np.stack([np.roll(w[:, c], c) for c in range(n)], axis=1)
    packed = oracle.pack_int4(w)
    s = np.empty((1, n), dtype=np.float16)
    specials = np.array([0.0, -0.0, 6e-8, 1e-5, 6.1e-5, 0.5, 1.0, -1.0, 3.14, 1000.0, 8190.0,
                         8192.0, 65504.0, -65504.0, 0.0123, -0.007], dtype=np.float16)
    s[0, :len(specials)] = specials
    s[0, len(specials):] = (np.sign(rng.standard_normal(n - len(specials)))
                            * np.exp2(rng.uniform(-24, 15, n - len(specials)))).astype(np.float16)
    got = to_host(kaio.dequant_int4_debug(to_dev(packed), to_dev(s), variant))
    want = oracle.dequant_int4(packed, s)
    g16, w16 = got.view(np.uint16), want.view(np.uint16)
    # +0 and -0 are both a correct f16 zero for a zero product; compare the rest bitwise
    zero = (want == 0)
    assert np.array_equal(g16[~zero], w16[~zero])
    assert np.all(got[zero] == 0)


def test_two_instruction_routine_at_its_scale_bounds():
    # variant 2 takes the two-instruction routine for 0 < s <= 65504 * 2^-20
    # (f16 bits 0x0001 .. 0x2BFF): every nibble value against the scales at
    # and around both ends of that range, every subnormal scale class and the
    # scales just outside it (0, -0, negative, 0x2C00 and up).
    k = 128
    bits = np.array([0x0001, 0x0002, 0x0003, 0x00FF, 0x0200, 0x03FF, 0x0400, 0x0401, 0x07FF,
                     0x1000, 0x2000, 0x2400, 0x2800, 0x2BFE, 0x2BFF, 0x2C00, 0x2C01, 0x3C00,
                     0x0000, 0x8000, 0x8001, 0xABFF, 0x7BFF], dtype=np.uint16)
    n = 8 * ((len(bits) + 7) // 8)
    s = np.full((1, n), 0x2000, dtype=np.uint16)
    s[0, :len(bits)] = bits
    s = s.view(np.float16)
    w = np.tile(np.arange(-8, 8, dtype=np.int8).reshape(16, 1), (k // 16, n))
    w = np.stack([np.roll(w[:, c], 3 * c) for c in range(n)], axis=1)
    packed = oracle.pack_int4(w)
    got = to_host(kaio.dequant_int4_debug(to_dev(packed), to_dev(s), 2))
    want = oracle.dequant_int4(packed, s)
    assert np.array_equal(got.view(np.uint16), want.view(np.uint16))
