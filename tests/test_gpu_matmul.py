"""Dense tcgen05 matmul and its backward against the CPU oracle (GPU)."""
import numpy as np
import pytest

import oracle
from qkv_projection_gb300 import kaio
from qkv_projection_gb300.inputs import dense_inputs

from gpu_helpers import rel_frobenius, to_dev, to_host

pytestmark = pytest.mark.gpu

TOL = 1e-3


# Tiles are computed by CTA pairs (two vertically adjacent 128-row blocks share
# the B tile): shapes with an odd number of row blocks leave the last pair
# half out of range, and (2432, 4096, 128) -- 19 row blocks, 160 pair tiles --
# also makes the persistent loop wrap.
@pytest.mark.parametrize("m,n,k", [(128, 256, 64), (1, 8, 8), (130, 264, 136), (257, 520, 1000),
                                   (64, 64, 4096), (300, 1024, 256), (512, 512, 512),
                                   (2432, 4096, 128)])
def test_forward_small(m, n, k):
    a, b, _ = dense_inputs(m, n, k, seed=m + n + k)
    c = to_host(kaio.matmul_tc(to_dev(a), to_dev(b)))
    assert rel_frobenius(c, oracle.matmul_ref(a, b)) <= TOL


def test_forward_4096_sampled_rows():
    a, b, _ = dense_inputs(4096, 4096, 4096, seed=0)
    c = to_host(kaio.matmul_tc(to_dev(a), to_dev(b)))
    rows = np.unique(np.concatenate([np.random.default_rng(1).choice(4096, 64, replace=False),
                                     [0, 1, 127, 128, 4095]]))
    assert rel_frobenius(c[rows], oracle.matmul_rows(a, b, rows)) <= TOL


@pytest.mark.parametrize("m,n,k", [(128, 256, 64), (136, 264, 200), (520, 256, 384), (64, 8, 8)])
def test_backward_small(m, n, k):
    a, b, g = dense_inputs(m, n, k, seed=3 * m + n)
    da, db = kaio.matmul_tc_backward(to_dev(a), to_dev(b), to_dev(g))
    ra, rb = oracle.matmul_backward_ref(a, b, g)
    assert rel_frobenius(to_host(da), ra) <= TOL
    assert rel_frobenius(to_host(db), rb) <= TOL


def test_backward_4096_sampled():
    a, b, g = dense_inputs(4096, 4096, 4096, seed=0)
    da, db = kaio.matmul_tc_backward(to_dev(a), to_dev(b), to_dev(g))
    da, db = to_host(da), to_host(db)
    rows = np.unique(np.concatenate([np.random.default_rng(2).choice(4096, 48, replace=False),
                                     [0, 127, 128, 4095]]))
    g64, b64, a64 = (np.asarray(t, dtype=np.float64) for t in (g, b, a))
    # dA rows = G[rows] @ B^T ; dB rows = A[:, rows]^T @ G
    ra = oracle.matmul_backward_ref(a[rows], b, g[rows])[0]
    assert rel_frobenius(da[rows], ra) <= TOL
    rb = a64[:, rows].T @ g64
    assert rel_frobenius(db[rows], rb) <= TOL


def test_backward_transpose_identities():
    # A = I  ->  dB = A^T G = G exactly;  B = I  ->  dA = G B^T = G exactly
    n = 256
    _, b, g = dense_inputs(n, n, n, seed=4)
    eye = np.eye(n, dtype=np.float16)
    _, db = kaio.matmul_tc_backward(to_dev(eye), to_dev(b), to_dev(g))
    assert np.array_equal(to_host(db), g.astype(np.float32))
    da, _ = kaio.matmul_tc_backward(to_dev(b), to_dev(eye), to_dev(g))
    assert np.array_equal(to_host(da), g.astype(np.float32))


def test_forward_identity_exact():
    a, _, _ = dense_inputs(200, 256, 256, seed=6)
    eye = np.eye(256, dtype=np.float16)
    c = to_host(kaio.matmul_tc(to_dev(a), to_dev(eye)))
    assert np.array_equal(c, a.astype(np.float32))


def test_no_device_timeouts_reported():
    kaio.device_status()


@pytest.mark.parametrize("m,n,k", [(128, 256, 64), (1, 8, 8), (130, 264, 136), (257, 520, 1000),
                                   (512, 512, 512)])
def test_forward_f16_output(m, n, k):
    """The f16-output variant stores RN_f16 of the same f32 accumulator the f32
    variant stores (bit for bit), and stays within the matmul tolerance."""
    import torch
    a, b, _ = dense_inputs(m, n, k, seed=m + 2 * n + k)
    ad, bd = to_dev(a), to_dev(b)
    c32 = to_host(kaio.matmul_tc(ad, bd))
    c16 = kaio.matmul_tc(ad, bd, out_dtype=torch.float16)
    assert c16.dtype == torch.float16
    c16 = to_host(c16)
    assert np.array_equal(c16.view(np.uint16), c32.astype(np.float16).view(np.uint16))
    assert rel_frobenius(c16.astype(np.float64), oracle.matmul_ref(a, b)) <= TOL


@pytest.mark.parametrize("m,n,k", [(128, 256, 64), (136, 264, 200), (64, 8, 8)])
def test_backward_f16_output(m, n, k):
    import torch
    a, b, g = dense_inputs(m, n, k, seed=5 * m + n)
    ad, bd, gd = to_dev(a), to_dev(b), to_dev(g)
    da32, db32 = (to_host(t) for t in kaio.matmul_tc_backward(ad, bd, gd))
    da16, db16 = (to_host(t) for t in kaio.matmul_tc_backward(ad, bd, gd, out_dtype=torch.float16))
    assert np.array_equal(da16.view(np.uint16), da32.astype(np.float16).view(np.uint16))
    assert np.array_equal(db16.view(np.uint16), db32.astype(np.float16).view(np.uint16))
    ra, rb = oracle.matmul_backward_ref(a, b, g)
    assert rel_frobenius(da16.astype(np.float64), ra) <= TOL
    assert rel_frobenius(db16.astype(np.float64), rb) <= TOL


def test_f16_output_4096_sampled_rows():
    import torch
    a, b, _ = dense_inputs(4096, 4096, 4096, seed=0)
    c = to_host(kaio.matmul_tc(to_dev(a), to_dev(b), out_dtype=torch.float16))
    rows = np.unique(np.concatenate([np.random.default_rng(3).choice(4096, 48, replace=False),
                                     [0, 127, 128, 4095]]))
    assert rel_frobenius(c[rows].astype(np.float64), oracle.matmul_rows(a, b, rows)) <= TOL


def test_backward_into_given_outputs():
    import torch
    a, b, g = dense_inputs(136, 264, 200, seed=11)
    ad, bd, gd = to_dev(a), to_dev(b), to_dev(g)
    da, db = kaio.matmul_tc_backward(ad, bd, gd)
    oa = torch.full_like(da, float("nan"))
    ob = torch.full_like(db, float("nan"))
    ra, rb = kaio.matmul_tc_backward(ad, bd, gd, out=(oa, ob))
    assert ra is oa and rb is ob
    assert np.array_equal(to_host(oa), to_host(da)) and np.array_equal(to_host(ob), to_host(db))
    with pytest.raises(ValueError):
        kaio.matmul_tc_backward(ad, bd, gd, out=(ob, oa))   # shapes swapped


# Wide (512-column) pair tiles are used when they fill a wave of resident CTA
# pairs: (2432, 4232, 64) gives 10 x 9 = 90 of them, with a half-empty last
# pair of row blocks and a last column block 136 wide, whose chunks beyond N
# the epilogue skips.
def test_forward_wide_tiles_ragged_edges():
    import torch
    a, b, _ = dense_inputs(2432, 4232, 64, seed=5)
    ad, bd = to_dev(a), to_dev(b)
    c = to_host(kaio.matmul_tc(ad, bd))
    ref = oracle.matmul_ref(a, b)
    assert rel_frobenius(c, ref) <= TOL
    assert rel_frobenius(c[:, 4096:], ref[:, 4096:]) <= TOL      # the ragged column block
    assert rel_frobenius(c[2304:], ref[2304:]) <= TOL            # the half-empty row pair
    c16 = to_host(kaio.matmul_tc(ad, bd, out_dtype=torch.float16))
    assert np.array_equal(c16.view(np.uint16), c.astype(np.float16).view(np.uint16))
