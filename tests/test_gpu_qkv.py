"""W4A16 fused QKV projection on the GPU against the CPU oracle."""
import numpy as np
import pytest

import oracle
from qkv_projection_gb300 import kaio
from qkv_projection_gb300.inputs import qkv_inputs

from gpu_helpers import assert_qkv_close, qkv_to_dev, to_dev, to_host

pytestmark = pytest.mark.gpu


def run(inp, stream=None):
    outs = kaio.qkv_project_int4(*qkv_to_dev(inp), stream=stream)
    return [to_host(o) for o in outs]


def check_full(inp, what):
    got = run(inp)
    refs = oracle.qkv_project_int4_ref(*inp.__dict__.values())
    for g, r, name in zip(got, refs, "QKV"):
        assert_qkv_close(g, r, f"{what} {name}")
    return got


# Small shapes spanning several tiles and ragged tails on both paths:
# M <= 16 (decode kernel) and M >= 17 (tcgen05 kernel).
SHAPES = [
    (1, 8, 128), (2, 40, 128), (3, 136, 256), (7, 264, 384), (8, 256, 512), (9, 520, 256),
    (15, 72, 1024), (16, 128, 256), (16, 1032, 640),
    (17, 128, 128), (33, 264, 256), (63, 136, 384), (64, 256, 512), (65, 392, 256),
    (128, 128, 128), (129, 520, 640), (200, 264, 1024), (257, 136, 256),
]


@pytest.mark.parametrize("m,n,k", SHAPES)
def test_small_shapes(m, n, k):
    check_full(qkv_inputs(m, n, k, seed=m * 7 + n + k), f"M={m} N={n} K={k}")


def test_config_m16_k256_n128_seed0():
    check_full(qkv_inputs(16, 128, 256, seed=0), "c1")


def test_decode_m1_k4096_n4096_full():
    check_full(qkv_inputs(1, 4096, 4096, seed=0), "decode M=1")


def test_batched_decode_m16_k8192_n8192_sampled_columns():
    inp = qkv_inputs(16, 8192, 8192, seed=0)
    got = run(inp)
    cols = np.sort(np.random.default_rng(0).choice(8192, 384, replace=False))
    cols = np.unique(np.concatenate([cols, [0, 1, 255, 256, 8191]]))
    sub = [inp.x] + [w[:, cols] for w in inp.weights()] + [s[:, cols] for s in inp.scales()]
    refs = oracle.qkv_project_int4_ref(*sub)
    for g, r, name in zip(got, refs, "QKV"):
        assert_qkv_close(g[:, cols], r, f"M=16 K=8192 {name}")


def test_prefill_4096_sampled_rows():
    inp = qkv_inputs(4096, 4096, 4096, seed=0)
    got = run(inp)
    rows = np.sort(np.random.default_rng(0).choice(4096, 64, replace=False))
    rows = np.unique(np.concatenate([rows, [0, 1, 127, 128, 4095]]))
    refs = oracle.qkv_project_int4_rows(*inp.__dict__.values(), rows)
    for g, r, name in zip(got, refs, "QKV"):
        assert_qkv_close(g[rows], r, f"prefill {name}")


@pytest.mark.parametrize("m", [4, 16, 96])
def test_deterministic(m):
    inp = qkv_inputs(m, 1032, 2048, seed=5)
    a = run(inp)
    b = run(inp)
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint16), y.view(np.uint16))


@pytest.mark.parametrize("m,n,k", [(5, 264, 256), (40, 136, 384)])
def test_guard_bands_untouched(m, n, k):
    import torch
    inp = qkv_inputs(m, n, k, seed=3)
    ins = qkv_to_dev(inp)
    pad = 64  # elements of f16 before and after each output
    bufs = [torch.full((m * n + 2 * pad,), float("nan"), dtype=torch.float16, device="cuda")
            for _ in range(3)]
    outs = [b[pad:pad + m * n].view(m, n) for b in bufs]
    kaio.qkv_project_int4(*ins, out=outs)
    torch.cuda.synchronize()
    refs = oracle.qkv_project_int4_ref(*inp.__dict__.values())
    for b, r in zip(bufs, refs):
        h = to_host(b)
        assert np.isnan(h[:pad]).all() and np.isnan(h[pad + m * n:]).all()
        assert_qkv_close(h[pad:pad + m * n].reshape(m, n), r, "guarded")


def test_aliased_weight_inputs_and_side_stream():
    import torch
    inp = qkv_inputs(12, 264, 256, seed=9)
    x, wq, _, _, sq, _, _ = qkv_to_dev(inp)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        outs = kaio.qkv_project_int4(x, wq, wq, wq, sq, sq, sq, stream=s)
    s.synchronize()
    ref = oracle.qkv_project_int4_ref(inp.x, inp.wq, inp.wq, inp.wq, inp.sq, inp.sq, inp.sq)[0]
    for o in outs:
        assert_qkv_close(to_host(o), ref, "aliased")


def test_empty_and_zero_k():
    import torch
    lib = kaio.lib()
    bufs = [torch.full((3, 16), 7.0, dtype=torch.float16, device="cuda") for _ in range(4)]
    w = torch.zeros((16, 16), dtype=torch.int32, device="cuda")
    p = [b.data_ptr() for b in bufs]
    # M == 0: nothing to compute, nothing written
    st = lib.kaio_qkv_project_int4(p[3], w.data_ptr(), w.data_ptr(), w.data_ptr(), p[3], p[3], p[3],
                                   p[0], p[1], p[2], 0, 16, 128, None)
    assert st == kaio.KAIO_OK, kaio.last_error()
    torch.cuda.synchronize()
    assert all((to_host(b) == 7).all() for b in bufs[:3])
    # K == 0: the empty sum; the outputs become zeros (inputs span no bytes)
    st = lib.kaio_qkv_project_int4(p[3], p[3], p[3], p[3], p[3], p[3], p[3],
                                   p[0], p[1], p[2], 3, 16, 0, None)
    assert st == kaio.KAIO_OK, kaio.last_error()
    torch.cuda.synchronize()
    assert all((to_host(b) == 0).all() for b in bufs[:3])


def test_misaligned_device_pointer_rejected():
    import torch
    inp = qkv_inputs(4, 64, 128, seed=1)
    x, wq, wk, wv, sq, sk, sv = qkv_to_dev(inp)
    big = torch.zeros(4 * 64 + 8, dtype=torch.float16, device="cuda")
    st = kaio.lib().kaio_qkv_project_int4(x.data_ptr(), wq.data_ptr(), wk.data_ptr(), wv.data_ptr(),
                                          sq.data_ptr(), sk.data_ptr(), sv.data_ptr(),
                                          big.data_ptr() + 2, big.data_ptr() + 2, big.data_ptr() + 2,
                                          4, 64, 128, None)
    assert st == kaio.KAIO_ERR_MISALIGNED


def test_host_pointer_rejected():
    import torch
    inp = qkv_inputs(4, 64, 128, seed=1)
    x, wq, wk, wv, sq, sk, sv = qkv_to_dev(inp)
    host = torch.zeros((4, 128), dtype=torch.float16).pin_memory()
    q, k, v = (torch.empty((4, 64), dtype=torch.float16, device="cuda") for _ in range(3))
    st = kaio.lib().kaio_qkv_project_int4(host.data_ptr(), wq.data_ptr(), wk.data_ptr(), wv.data_ptr(),
                                          sq.data_ptr(), sk.data_ptr(), sv.data_ptr(),
                                          q.data_ptr(), k.data_ptr(), v.data_ptr(), 4, 64, 128, None)
    assert st == kaio.KAIO_ERR_INVALID_VALUE
    assert "device memory" in kaio.last_error()


def test_decode_shared_memory_sizes_in_any_order():
    # Decode launches size their shared memory by K; a small launch between two
    # large ones must not leave the kernel's limit below what the large one needs.
    for m, n, k in [(1, 4096, 4096), (5, 264, 128), (1, 4096, 4096), (12, 256, 256), (16, 1032, 8192)]:
        check_full(qkv_inputs(m, n, k, seed=k), f"sequence M={m} K={k}")


def test_no_device_timeouts_reported():
    kaio.device_status()


@pytest.mark.parametrize("m", [1, 16])
def test_input_written_by_the_preceding_kernel(m):
    """A call must read x as left by the kernel just before it in the stream
    (the decode kernel may start early under programmatic dependent launch and
    must wait for its predecessor before reading): x is produced on the device
    by a PyTorch kernel, in a chain of calls with no host synchronisation."""
    import torch
    n = k = 1024
    inp = qkv_inputs(m, n, k, seed=31 + m)
    x, wq, wk, wv, sq, sk, sv = qkv_to_dev(inp)
    x_buf = torch.zeros_like(x)
    outs = None
    for step in range(3):
        x_buf.copy_(x * (step + 1))        # a kernel writing x right before the call
        outs = kaio.qkv_project_int4(x_buf, wq, wk, wv, sq, sk, sv)
    torch.cuda.synchronize()
    x3 = (inp.x.astype(np.float64) * 3).astype(np.float16)
    refs = oracle.qkv_project_int4_ref(x3, inp.wq, inp.wk, inp.wv, inp.sq, inp.sk, inp.sv)
    for o, r, name in zip(outs, refs, "QKV"):
        assert_qkv_close(to_host(o), r, f"preceding-kernel x {name}")


def test_chained_calls_read_the_previous_calls_output():
    """Call 2 takes call 1's Q output as its x (K = N) with no host
    synchronisation between them: it must see all of call 1's output."""
    import torch
    m, n = 4, 512
    inp = qkv_inputs(m, n, n, seed=77)
    x, wq, wk, wv, sq, sk, sv = qkv_to_dev(inp)
    q1, _, _ = kaio.qkv_project_int4(x, wq, wk, wv, sq, sk, sv)
    q2, k2, v2 = kaio.qkv_project_int4(q1, wq, wk, wv, sq, sk, sv)
    torch.cuda.synchronize()
    q1_host = to_host(q1)
    refs = oracle.qkv_project_int4_ref(q1_host, inp.wq, inp.wk, inp.wv, inp.sq, inp.sk, inp.sv)
    for o, r, name in zip((q2, k2, v2), refs, "QKV"):
        assert_qkv_close(to_host(o), r, f"chained {name}")


@pytest.mark.parametrize("m", [1, 16, 64, 200])
def test_mixed_scale_classes(m):
    # Scales of every class in one problem, per lane and per group: a large
    # scale at one column of group 1, negative scales over the second column
    # tile, subnormal ones over the third, ordinary ones elsewhere.
    n, k = 392, 512
    inp = qkv_inputs(m, n, k, seed=m + 11)
    for s in inp.scales():
        s[1, 40] = np.float16(0.5)
        s[:, 128:256] = -s[:, 128:256]
        s[:, 256:384] = (s[:, 256:384].astype(np.float32) * np.float32(2.0 ** -12)).astype(np.float16)
    check_full(inp, f"mixed scale classes M={m}")


@pytest.mark.parametrize("m", [2, 5, 11])
def test_decode_rows_not_a_multiple_of_the_cluster(m):
    # The cluster's ranks finish batch rows m = rank, rank + S, ...: with M not a
    # multiple of S some ranks finish fewer rows than others (here K = 8192 over
    # 64 groups and a ragged last column tile).
    check_full(qkv_inputs(m, 1032, 8192, seed=100 + m), f"M={m} N=1032 K=8192")


@pytest.mark.parametrize("m", [1, 16])
def test_decode_more_ctas_than_sms(m):
    # N = 20480 is 160 column tiles: with K = 384 the planner runs them as 160
    # single-CTA clusters, more than the GPU's 152 SMs hold at once, so CTAs of
    # a second wave start as the first ones finish (and programmatic launch
    # lets the next call's CTAs wait on this one's).
    inp = qkv_inputs(m, 20480, 384, seed=20480 + m)
    got = run(inp)
    got2 = run(inp)
    for g, g2, r, name in zip(got, got2, oracle.qkv_project_int4_ref(*inp.__dict__.values()), "QKV"):
        assert_qkv_close(g, r, f"M={m} N=20480 {name}")
        assert np.array_equal(g.view(np.uint16), g2.view(np.uint16))
