"""The allocation-free decode entry point (kaio_qkv_project_int4_noalloc).

It serves callers that cannot allocate device memory (engines and plugin hosts
that own all device memory, fully reserved processes, latency-critical paths):
its stream-K kernel keeps its split-K scratch in a fixed array inside the
library and allocates nothing. Its results must match both the regular entry
point and the CPU oracle within the projection tolerance, element by element,
on consecutive calls that share that array.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes when run on its own.
"""
import ctypes

import numpy as np
import pytest

import oracle
from qkv_projection_gb300 import kaio
from qkv_projection_gb300.inputs import qkv_inputs

from gpu_helpers import qkv_to_dev, to_host

pytestmark = pytest.mark.gpu


def _call(fn, ins, outs, m, n, k):
    st = fn(*(t.data_ptr() for t in ins), *(o.data_ptr() for o in outs), m, n, k, None)
    assert st == kaio.KAIO_OK, kaio.last_error()


def _close(got, ref):
    got = got.astype(np.float64)
    ref = ref.astype(np.float64)
    bound = oracle.ulp_f16(ref) + 2e-3 * np.abs(ref).max()
    assert np.all(np.abs(got - ref) <= bound)


@pytest.mark.parametrize("m,n,k", [(16, 1032, 640), (1, 4096, 4096), (5, 264, 384)])
def test_noalloc_matches_regular_entry_and_oracle_twice(m, n, k):
    import torch
    lib = kaio.lib()
    inp = qkv_inputs(m, n, k, seed=m + n + k)
    ins = qkv_to_dev(inp)
    ref_out = [torch.empty((m, n), dtype=torch.float16, device="cuda") for _ in range(3)]
    _call(lib.kaio_qkv_project_int4, ins, ref_out, m, n, k)
    torch.cuda.synchronize()
    regular = [to_host(o) for o in ref_out]
    exact = oracle.qkv_project_int4_ref(*inp.__dict__.values())
    for _ in range(2):                       # two calls in a row share the scratch array
        out = [torch.full((m, n), float("nan"), dtype=torch.float16, device="cuda") for _ in range(3)]
        _call(lib.kaio_qkv_project_int4_noalloc, ins, out, m, n, k)
        torch.cuda.synchronize()
        for o, r, e in zip(out, regular, exact):
            got = to_host(o)
            _close(got, r)                   # the regular entry point's result
            _close(got, e)                   # the oracle's f64 result


def test_noalloc_rejects_sizes_beyond_its_limits():
    import torch
    lib = kaio.lib()
    ins = qkv_to_dev(qkv_inputs(17, 64, 128, seed=1))
    out = [torch.empty((17, 64), dtype=torch.float16, device="cuda") for _ in range(3)]
    st = lib.kaio_qkv_project_int4_noalloc(*(t.data_ptr() for t in ins), *(o.data_ptr() for o in out),
                                           17, 64, 128, None)
    assert st == kaio.KAIO_ERR_INVALID_VALUE
    assert "M (17) exceeds 16" in kaio.last_error()
    big_n = 5462 * 256          # 3 * 5462 column groups > 16384
    st = lib.kaio_qkv_project_int4_noalloc(*(t.data_ptr() for t in ins), *(o.data_ptr() for o in out),
                                           1, big_n, 128, None)
    assert st == kaio.KAIO_ERR_INVALID_VALUE
    assert "allocation-free limit" in kaio.last_error()
