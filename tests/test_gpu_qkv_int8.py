"""W8A16 fused QKV projection on the GPU against the CPU oracle."""
import numpy as np
import pytest

import oracle
from qkv_projection_gb300 import kaio
from qkv_projection_gb300.inputs import qkv_int8_inputs

from gpu_helpers import assert_qkv_close, to_dev, to_host

pytestmark = pytest.mark.gpu


def dev_args(inp):
    return [to_dev(inp.x)] + [to_dev(w) for w in inp.weights()] + list(inp.scales())


def run(inp, stream=None, out=None):
    outs = kaio.qkv_project_int8(*dev_args(inp), out=out, stream=stream)
    return [to_host(o) for o in outs]


def check_full(inp, what):
    got = run(inp)
    for g, r, name in zip(got, oracle.qkv_project_int8_ref(*inp.args()), "QKV"):
        assert_qkv_close(g, r, f"{what} {name}")
    return got


# Several tiles and ragged tails on both paths: M <= 16 (cluster split-K
# decode kernel) and M >= 17 (tile kernel); N not a multiple of 128, K from
# one 128-group up.
SHAPES = [
    (1, 8, 128), (2, 40, 128), (3, 136, 256), (7, 264, 384), (8, 256, 512), (9, 520, 256),
    (15, 72, 1024), (16, 128, 256), (16, 1032, 640), (1, 136, 2176),
    (17, 128, 128), (33, 264, 256), (63, 136, 384), (64, 256, 512), (65, 392, 256),
    (128, 128, 128), (129, 520, 640), (200, 264, 1024), (257, 136, 256),
]


@pytest.mark.parametrize("m,n,k", SHAPES)
def test_small_shapes(m, n, k):
    check_full(qkv_int8_inputs(m, n, k, seed=m * 7 + n + k), f"M={m} N={n} K={k}")


def test_decode_m1_k4096_n4096_full():
    check_full(qkv_int8_inputs(1, 4096, 4096, seed=0), "decode M=1")


def test_batched_decode_m16_k8192_n8192_sampled_columns():
    inp = qkv_int8_inputs(16, 8192, 8192, seed=0)
    got = run(inp)
    cols = np.sort(np.random.default_rng(0).choice(8192, 384, replace=False))
    cols = np.unique(np.concatenate([cols, [0, 1, 127, 128, 8191]]))
    refs = oracle.qkv_project_int8_ref(inp.x, *[w[:, cols] for w in inp.weights()], *inp.scales())
    for g, r, name in zip(got, refs, "QKV"):
        assert_qkv_close(g[:, cols], r, f"M=16 K=8192 {name}")


def test_prefill_4096_sampled_rows():
    inp = qkv_int8_inputs(4096, 4096, 4096, seed=0)
    got = run(inp)
    rows = np.sort(np.random.default_rng(0).choice(4096, 64, replace=False))
    rows = np.unique(np.concatenate([rows, [0, 1, 127, 128, 4095]]))
    for g, r, name in zip(got, oracle.qkv_project_int8_rows(*inp.args(), rows), "QKV"):
        assert_qkv_close(g[rows], r, f"prefill {name}")


@pytest.mark.parametrize("m", [1, 16, 17, 200])
def test_extreme_bytes_are_exact(m):
    # Bytes -128, 127, -1, 0 and x in {-1, 0.5, 1}: every partial sum is an
    # exact f32 number, the power-of-two scale is exact, and the results are
    # f16 numbers, so the kernel must reproduce the oracle bit for bit.
    n, k = 264, 512
    rng = np.random.default_rng(m)
    w = rng.choice(np.array([-128, 127, -1, 0]), size=(k, n))
    x = rng.choice(np.array([-1.0, 0.5, 1.0]), size=(m, k)).astype(np.float16)
    packed = oracle.pack_int8(w)
    scales = (2.0 ** -9, 2.0 ** -8, 2.0 ** -10)
    got = kaio.qkv_project_int8(to_dev(x), to_dev(packed), to_dev(packed), to_dev(packed), *scales)
    refs = oracle.qkv_project_int8_ref(x, packed, packed, packed, *scales)
    for g, r in zip(got, refs):
        assert np.array_equal(to_host(g), oracle.rn_f16(r))


@pytest.mark.parametrize("m", [4, 96])
def test_scale_semantics(m):
    inp = qkv_int8_inputs(m, 136, 384, seed=4)
    x, wq = to_dev(inp.x), to_dev(inp.wq)
    q, k, v = (to_host(t) for t in kaio.qkv_project_int8(x, wq, wq, wq, 1.0 / 64, 1.0 / 32, -1.0 / 64))
    assert np.any(q)
    assert np.array_equal(k, (q.astype(np.float64) * 2).astype(np.float16))   # exact: power of two
    assert np.array_equal(v, -q)
    q0, _, vn = (to_host(t) for t in kaio.qkv_project_int8(x, wq, wq, wq, 0.0, 1.0, float("nan")))
    assert not np.any(q0) and np.isnan(vn).all()


@pytest.mark.parametrize("m", [4, 16, 96])
def test_deterministic(m):
    inp = qkv_int8_inputs(m, 1032, 2048, seed=5)
    a, b = run(inp), run(inp)
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint16), y.view(np.uint16))


@pytest.mark.parametrize("m,n,k", [(5, 264, 256), (40, 136, 384)])
def test_guard_bands_untouched(m, n, k):
    import torch
    inp = qkv_int8_inputs(m, n, k, seed=3)
    pad = 64
    bufs = [torch.full((m * n + 2 * pad,), float("nan"), dtype=torch.float16, device="cuda")
            for _ in range(3)]
    outs = [b[pad:pad + m * n].view(m, n) for b in bufs]
    kaio.qkv_project_int8(*dev_args(inp), out=outs)
    torch.cuda.synchronize()
    for b, r in zip(bufs, oracle.qkv_project_int8_ref(*inp.args())):
        h = to_host(b)
        assert np.isnan(h[:pad]).all() and np.isnan(h[pad + m * n:]).all()
        assert_qkv_close(h[pad:pad + m * n].reshape(m, n), r, "guarded")


def test_aliased_weight_inputs_and_side_stream():
    import torch
    inp = qkv_int8_inputs(12, 264, 256, seed=9)
    x, wq = to_dev(inp.x), to_dev(inp.wq)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        outs = kaio.qkv_project_int8(x, wq, wq, wq, inp.sq, inp.sq, inp.sq, stream=s)
    s.synchronize()
    ref = oracle.qkv_project_int8_ref(inp.x, inp.wq, inp.wq, inp.wq, inp.sq, inp.sq, inp.sq)[0]
    for o in outs:
        assert_qkv_close(to_host(o), ref, "aliased")


def test_empty_and_zero_k():
    import torch
    lib = kaio.lib()
    bufs = [torch.full((3, 16), 7.0, dtype=torch.float16, device="cuda") for _ in range(4)]
    w = torch.zeros((32, 16), dtype=torch.int32, device="cuda")
    p = [b.data_ptr() for b in bufs]
    # M = 0: nothing written
    assert lib.kaio_qkv_project_int8(p[0], w.data_ptr(), w.data_ptr(), w.data_ptr(), 1.0, 1.0, 1.0,
                                     p[1], p[2], p[3], 0, 16, 128, None) == kaio.KAIO_OK
    torch.cuda.synchronize()
    assert all((b == 7).all() for b in bufs[1:])
    # K = 0: the empty sum, every output element 0
    assert lib.kaio_qkv_project_int8(p[0], w.data_ptr(), w.data_ptr(), w.data_ptr(), 1.0, 1.0, 1.0,
                                     p[1], p[2], p[3], 3, 16, 0, None) == kaio.KAIO_OK
    torch.cuda.synchronize()
    assert all((b == 0).all() for b in bufs[1:])


@pytest.mark.parametrize("m", [1, 16, 40])
def test_input_written_by_the_preceding_kernel(m):
    # x is produced on the same stream by a PyTorch kernel just before the
    # call, with no host synchronisation in between.
    import torch
    inp = qkv_int8_inputs(m, 520, 1024, seed=13)
    x = to_dev(inp.x)
    ws = [to_dev(w) for w in inp.weights()]
    stream = torch.cuda.current_stream()
    x2 = torch.empty_like(x)
    for _ in range(3):
        x2.zero_()
        x2.copy_(x * 2)                  # exact in f16
        outs = kaio.qkv_project_int8(x2, *ws, *inp.scales(), stream=stream)
    refs = oracle.qkv_project_int8_ref(inp.x.astype(np.float64) * 2, *inp.weights(), *inp.scales())
    for o, r in zip(outs, refs):
        assert_qkv_close(to_host(o), r, "x from preceding kernel")


@pytest.mark.parametrize("m,n,k", [(1, 1032, 12416), (5, 264, 5760), (16, 136, 8576)])
def test_decode_x_ring_wraps(m, n, k):
    # M <= 16 keeps x in a ring of its own, four slots beside two weight
    # stages: here each CTA's K range spans more stages than the x ring has
    # slots, and K / 128 (97, 45, 67) is odd, so ranges end on half stages.
    check_full(qkv_int8_inputs(m, n, k, seed=m + n + k), f"M={m} N={n} K={k}")


@pytest.mark.parametrize("m", [1, 16])
def test_decode_more_ctas_than_sms(m):
    # 160 column tiles of single-CTA clusters: two waves on a 152-SM GPU
    check_full(qkv_int8_inputs(m, 20480, 384, seed=20480 + m), f"M={m} N=20480 K=384")


def test_no_device_timeouts_reported():
    kaio.device_status()
