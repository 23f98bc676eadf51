"""Failure detection of the decode kernel's bounded waits, on the GPU.

Every wait in the kernels' pipelines gives up after a limit instead of
hanging; the kernel then records the timeout in a device error word, lets the
copies and MMAs it has in flight finish, frees its tensor memory and returns.
Here a test entry runs the decode kernel with that limit set to zero, so the
first pipeline wait that finds its phase unfinished (the MMA warps' first
wait needs converted weights, which take thousands of cycles) gives up. The
host must then read KAIO_ERR_DEVICE_TIMEOUT from kaio_device_status(), the
error must be cleared by that read, and the context must stay usable: the
next regular call matches the oracle.
"""
import numpy as np
import pytest

import oracle
from qkv_projection_gb300 import kaio
from qkv_projection_gb300.inputs import qkv_inputs

from gpu_helpers import assert_qkv_close, qkv_to_dev, to_host

pytestmark = pytest.mark.gpu


def _regular(ins, inp, what):
    outs = kaio.qkv_project_int4(*ins)
    refs = oracle.qkv_project_int4_ref(*inp.__dict__.values())
    for o, r, name in zip(outs, refs, "QKV"):
        assert_qkv_close(to_host(o), r, f"{what} {name}")


@pytest.mark.parametrize("m,n,k", [(1, 256, 1024), (16, 1032, 640)])
def test_zero_wait_limit_reports_timeout_and_context_survives(m, n, k):
    import torch
    inp = qkv_inputs(m, n, k, seed=11 + m)
    ins = qkv_to_dev(inp)
    kaio.device_status()                                   # start from a clear error word
    _regular(ins, inp, "before")
    outs = [torch.empty((m, n), dtype=torch.float16, device="cuda") for _ in range(3)]
    st = kaio.lib().kaio_debug_decode_wait_limit(*(t.data_ptr() for t in ins), *(o.data_ptr() for o in outs),
                                                 m, n, k, 0, None)
    assert st == kaio.KAIO_OK, kaio.last_error()
    assert kaio.lib().kaio_device_status() == kaio.KAIO_ERR_DEVICE_TIMEOUT
    assert "bounded wait" in kaio.last_error()
    assert kaio.lib().kaio_device_status() == kaio.KAIO_OK   # the read cleared it
    _regular(ins, inp, "after")
    assert kaio.lib().kaio_device_status() == kaio.KAIO_OK


def test_normal_wait_limit_through_the_test_entry_matches_the_oracle():
    import torch
    m, n, k = 5, 264, 384
    inp = qkv_inputs(m, n, k, seed=5)
    ins = qkv_to_dev(inp)
    outs = [torch.empty((m, n), dtype=torch.float16, device="cuda") for _ in range(3)]
    st = kaio.lib().kaio_debug_decode_wait_limit(*(t.data_ptr() for t in ins), *(o.data_ptr() for o in outs),
                                                 m, n, k, 2_000_000_000, None)
    assert st == kaio.KAIO_OK, kaio.last_error()
    torch.cuda.synchronize()
    refs = oracle.qkv_project_int4_ref(*inp.__dict__.values())
    for o, r, name in zip(outs, refs, "QKV"):
        assert_qkv_close(to_host(o), r, f"2 s limit {name}")
    assert kaio.lib().kaio_device_status() == kaio.KAIO_OK
