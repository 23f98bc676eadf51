"""Per-group dequantisation and its backward on the GPU against the oracle.

Every element is a single product rounded once to the element type, so the
results must match the oracle bit for bit, on the vector kernel (aligned rows
split into 16-byte vectors) and on the scalar kernel (any other shape).
"""
import numpy as np
import pytest

from oracle import dequant_group as dg
from qkv_projection_gb300 import kaio
from qkv_projection_gb300.inputs import dequant_group_inputs

pytestmark = pytest.mark.gpu

DTYPES = ["f32", "f64", "f16", "bf16"]


def _torch_dtype(d):
    import torch
    return {"f32": torch.float32, "f64": torch.float64, "f16": torch.float16, "bf16": torch.bfloat16}[d]


def to_dev(a, d):
    """numpy array (bf16 as uint16 patterns) -> CUDA tensor of type d."""
    import torch
    if d == "bf16":
        return torch.from_numpy(a.view(np.int16).copy()).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bits(t, d):
    """CUDA tensor -> numpy bit patterns for exact comparison."""
    import torch
    if d == "bf16":
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    a = t.cpu().numpy()
    return a.view({"f32": np.uint32, "f64": np.uint64, "f16": np.uint16}[d])


def ref_bits(r, d):
    if d == "bf16":
        return np.asarray(r, dtype=np.uint16)
    return np.asarray(r).view({"f32": np.uint32, "f64": np.uint64, "f16": np.uint16}[d])


# (outer, axis, group): vector path with whole-vector groups, vector path with
# groups smaller than or straddling a vector, and shapes only the scalar
# kernel takes (axis not a multiple of the vector length).
SHAPES = [(3, 256, 128), (5, 1024, 32), (7, 96, 2), (4, 48, 6), (6, 30, 3), (1, 8, 8), (9, 130, 13)]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("outer,axis,group", SHAPES)
def test_backward_bit_exact(dtype, outer, axis, group):
    dy, _, sc = dequant_group_inputs(outer, axis, group, dtype, seed=outer * 7 + axis)
    got = kaio.dequantize_per_group_backward(to_dev(dy, dtype), to_dev(sc, dtype), group)
    assert got.dtype == _torch_dtype(dtype)
    ref = dg.dequantize_per_group_backward_ref(dy, sc, group, dtype)
    assert np.array_equal(bits(got, dtype), ref_bits(ref, dtype))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("q_dtype", ["s8", "u8"])
@pytest.mark.parametrize("outer,axis,group", SHAPES)
def test_forward_bit_exact(dtype, q_dtype, outer, axis, group):
    import torch
    _, q, sc = dequant_group_inputs(outer, axis, group, dtype, seed=outer + axis, q_dtype=q_dtype)
    got = kaio.dequantize_per_group(torch.from_numpy(q).cuda(), to_dev(sc, dtype), group)
    ref = dg.dequantize_per_group_ref(q, sc, group, dtype)
    assert np.array_equal(bits(got, dtype), ref_bits(ref, dtype))


@pytest.mark.parametrize("dtype", ["f16", "f32", "bf16"])
def test_backward_misaligned_views_use_the_scalar_kernel(dtype):
    # views starting one element into their buffers: element-aligned but not
    # 16-byte aligned, so the scalar kernel runs
    import torch
    outer, axis, group = 4, 64, 16
    dy, _, sc = dequant_group_inputs(outer, axis, group, dtype, seed=3)
    flat = torch.empty(outer * axis + 1, dtype=_torch_dtype(dtype), device="cuda")
    view = flat[1:].view(outer, axis)
    view.copy_(to_dev(dy, dtype))
    out_flat = torch.empty(outer * axis + 1, dtype=_torch_dtype(dtype), device="cuda")
    out_view = out_flat[1:].view(outer, axis)
    kaio.dequantize_per_group_backward(view, to_dev(sc, dtype), group, out=out_view)
    ref = dg.dequantize_per_group_backward_ref(dy, sc, group, dtype)
    assert np.array_equal(bits(out_view, dtype), ref_bits(ref, dtype))


@pytest.mark.parametrize("dtype", DTYPES)
def test_backward_in_place(dtype):
    outer, axis, group = 8, 512, 64
    dy, _, sc = dequant_group_inputs(outer, axis, group, dtype, seed=11)
    t = to_dev(dy, dtype)
    out = kaio.dequantize_per_group_backward(t, to_dev(sc, dtype), group, out=t)
    assert out.data_ptr() == t.data_ptr()
    ref = dg.dequantize_per_group_backward_ref(dy, sc, group, dtype)
    assert np.array_equal(bits(t, dtype), ref_bits(ref, dtype))


def test_empty_problems_are_no_ops():
    import torch
    lib = kaio.lib()
    # null pointers are fine when there is nothing to do, as on the page
    assert lib.kaio_dequantize_per_group_backward(kaio.KAIO_DTYPE_F16, kaio.KAIO_DTYPE_S8, 0, 128, 32,
                                                  None, None, None, None) == kaio.KAIO_OK
    assert lib.kaio_dequantize_per_group(kaio.KAIO_DTYPE_S8, kaio.KAIO_DTYPE_F32, 4, 0, 32,
                                         None, None, None, None) == kaio.KAIO_OK
    x = torch.zeros((0, 64), dtype=torch.float16, device="cuda")
    s = torch.zeros((0, 2), dtype=torch.float16, device="cuda")
    assert kaio.dequantize_per_group_backward(x, s, 32).shape == (0, 64)


def test_backward_large_sampled_rows():
    # 10.5 M vectors of 8 elements: more than the capped grid (64 CTAs of 256
    # threads x 4 vectors per SM on 152 SMs), so the grid-stride loop wraps
    outer, axis, group = 8192, 10240, 128
    dy, _, sc = dequant_group_inputs(outer, axis, group, "bf16", seed=21)
    got = bits(kaio.dequantize_per_group_backward(to_dev(dy, "bf16"), to_dev(sc, "bf16"), group), "bf16")
    rows = np.unique(np.concatenate([np.random.default_rng(5).choice(outer, 64, replace=False), [0, outer - 1]]))
    ref = dg.dequantize_per_group_backward_ref(dy[rows], sc[rows], group, "bf16")
    assert np.array_equal(got[rows], ref_bits(ref, "bf16"))


def test_forward_large_sampled_rows():
    import torch
    outer, axis, group = 8192, 10240, 64
    _, q, sc = dequant_group_inputs(outer, axis, group, "f16", seed=22, q_dtype="u8")
    got = bits(kaio.dequantize_per_group(torch.from_numpy(q).cuda(), to_dev(sc, "f16"), group), "f16")
    rows = np.unique(np.concatenate([np.random.default_rng(6).choice(outer, 64, replace=False), [0, outer - 1]]))
    ref = dg.dequantize_per_group_ref(q[rows], sc[rows], group, "f16")
    assert np.array_equal(got[rows], ref_bits(ref, "f16"))


def test_no_device_timeouts_or_errors():
    kaio.device_status()   # raises if any kernel reported an error
