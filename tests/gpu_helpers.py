"""Helpers shared by the GPU parity tests (tensor transfer and tolerances)."""
import numpy as np

import oracle


def to_dev(a):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a).cuda()


def to_host(t):
    return t.detach().cpu().numpy()


def qkv_to_dev(inp):
    return [to_dev(v) for v in (inp.x, inp.wq, inp.wk, inp.wv, inp.sq, inp.sk, inp.sv)]


def assert_qkv_close(got_f16, ref_f64, what=""):
    """|gpu - ref| <= ulp_f16(ref) + 2e-3 * max|ref|, per projection."""
    got = np.asarray(got_f16, dtype=np.float16).astype(np.float64)
    ref = np.asarray(ref_f64, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if ref.size == 0:
        return
    bound = oracle.ulp_f16(ref) + 2e-3 * np.abs(ref).max()
    err = np.abs(got - ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst at {i}: "
                             f"gpu={got[i]!r} ref={ref[i]!r} bound={bound[i]!r}")


def rel_frobenius(got, ref):
    ref = np.asarray(ref, dtype=np.float64)
    got = np.asarray(got, dtype=np.float64)
    den = np.linalg.norm(ref)
    return np.linalg.norm(got - ref) / (den if den > 0 else 1.0)
