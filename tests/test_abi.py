"""Host-side checks of the C ABI (no GPU needed).

The library must load on a machine without a GPU, export every function that
include/kaio_qkv.h declares, and reject bad arguments with the documented
status before it touches CUDA. These calls use made-up pointer values: the
validation that runs first (null pointers, K and N rules, alignment, overlap)
never dereferences them.
"""
import ctypes

import pytest

from qkv_projection_gb300 import kaio

INVALID, MISALIGNED, CUDA_ERR, UNSUPPORTED = (kaio.KAIO_ERR_INVALID_VALUE, kaio.KAIO_ERR_MISALIGNED,
                                              kaio.KAIO_ERR_CUDA, kaio.KAIO_ERR_UNSUPPORTED_DEVICE)


@pytest.fixture(scope="module")
def L():
    return kaio.lib()


def test_library_exports_every_declared_symbol(L):
    names = kaio.header_functions()
    assert {"kaio_qkv_project_int4", "kaio_matmul_tc", "kaio_matmul_tc_backward",
            "kaio_dequant_int4_debug", "kaio_last_error", "kaio_device_status",
            "kaio_status_string", "kaio_qkv_path"} <= set(names)
    for name in names:
        assert hasattr(L, name), name


def test_status_strings(L):
    for code, name in [(0, "KAIO_OK"), (1, "KAIO_ERR_INVALID_VALUE"), (2, "KAIO_ERR_MISALIGNED"),
                       (3, "KAIO_ERR_UNSUPPORTED_DEVICE"), (4, "KAIO_ERR_CUDA"),
                       (5, "KAIO_ERR_DEVICE_TIMEOUT")]:
        assert L.kaio_status_string(code).decode() == name


def test_path_selection(L):
    assert [L.kaio_qkv_path(m) for m in (0, 1, 8, 16, 17, 64, 4096)] == [0, 0, 0, 0, 1, 1, 1]


# distinct, 16-byte aligned fake device addresses, far apart
BASE = 1 << 40
def ptr(i, off=0):
    return BASE + i * (1 << 32) + off


def qkv(L, M=16, N=128, K=256, ptrs=None, stream=None):
    p = list(ptrs) if ptrs is not None else [ptr(i) for i in range(10)]
    return L.kaio_qkv_project_int4(*p, M, N, K, stream)


def test_qkv_rejects_null_pointers(L):
    for i in range(10):
        p = [ptr(j) for j in range(10)]
        p[i] = None
        assert qkv(L, ptrs=p) == INVALID
        assert "null" in kaio.last_error()


def test_qkv_rejects_k_not_multiple_of_group(L):
    for K in (64, 130, 200, 8):
        assert qkv(L, K=K) == INVALID
        assert "group_size (128)" in kaio.last_error()


def test_qkv_rejects_n_not_multiple_of_8(L):
    for N in (1, 4, 12, 130):
        assert qkv(L, N=N) == INVALID
        assert "N (" in kaio.last_error()


def test_qkv_rejects_misaligned(L):
    for i in range(10):
        p = [ptr(j) for j in range(10)]
        p[i] += 8
        assert qkv(L, ptrs=p) == MISALIGNED


def test_qkv_rejects_overlap(L):
    M, N, K = 16, 128, 256
    # q overlapping x
    p = [ptr(j) for j in range(10)]
    p[7] = p[0] + 16
    assert qkv(L, M, N, K, ptrs=p) == INVALID
    assert "overlaps input x" in kaio.last_error()
    # k overlapping q
    p = [ptr(j) for j in range(10)]
    p[8] = p[7] + 32
    assert qkv(L, M, N, K, ptrs=p) == INVALID
    assert "overlap" in kaio.last_error()
    # inputs may alias each other (read-only): same packed buffer for q/k/v weights
    p = [ptr(j) for j in range(10)]
    p[2] = p[3] = p[1]
    st = qkv(L, M, N, K, ptrs=p)
    assert st not in (INVALID, MISALIGNED)


def test_valid_call_without_gpu_fails_loudly(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # Arguments pass validation; the first CUDA call finds no device and the
    # library reports it instead of computing anything on the host.
    assert qkv(L) in (CUDA_ERR, UNSUPPORTED)
    assert kaio.last_error()


def test_matmul_validation(L):
    a, b, c = ptr(0), ptr(1), ptr(2)
    assert L.kaio_matmul_tc(None, b, c, 64, 64, 64, None) == INVALID
    assert L.kaio_matmul_tc(a, b, c, 64, 60, 64, None) == INVALID      # N % 8
    assert L.kaio_matmul_tc(a, b, c, 64, 64, 60, None) == INVALID      # K % 8
    assert L.kaio_matmul_tc(a + 4, b, c, 64, 64, 64, None) == MISALIGNED
    assert L.kaio_matmul_tc(a, b, a + 64, 64, 64, 64, None) == INVALID  # c overlaps a
    assert L.kaio_matmul_tc_backward(a, b, ptr(3), ptr(4), ptr(4) + 16, 64, 64, 64, None) == INVALID
    assert L.kaio_matmul_tc_backward(a, b, None, ptr(4), ptr(5), 64, 64, 64, None) == INVALID


def test_dequant_debug_validation(L):
    assert L.kaio_dequant_int4_debug(ptr(0), ptr(1), ptr(2), 128, 64, 3, None) == INVALID
    assert L.kaio_dequant_int4_debug(ptr(0), ptr(1), ptr(2), 128, 64, -1, None) == INVALID
    assert L.kaio_dequant_int4_debug(ptr(0), ptr(1), ptr(2), 100, 64, 0, None) == INVALID
    assert L.kaio_dequant_int4_debug(ptr(0), ptr(1), ptr(0), 128, 64, 0, None) == INVALID


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(4, 128, dtype=torch.float16)
    w = torch.zeros(16, 8, dtype=torch.int32)
    s = torch.zeros(1, 8, dtype=torch.float16)
    with pytest.raises(ValueError, match="CUDA device"):
        kaio.qkv_project_int4(x, w, w, w, s, s, s)
    with pytest.raises(ValueError, match="CUDA device"):
        kaio.matmul_tc(torch.zeros(8, 8, dtype=torch.float16), torch.zeros(8, 8, dtype=torch.float16))


def test_noalloc_entry_validation(L):
    p = [ptr(j) for j in range(10)]
    assert L.kaio_qkv_project_int4_noalloc(*p, 17, 128, 256, None) == INVALID     # M > 16
    assert "exceeds 16" in kaio.last_error()
    assert L.kaio_qkv_project_int4_noalloc(*p, 16, 128, 200, None) == INVALID     # K % 128
    assert L.kaio_qkv_project_int4_noalloc(*p, 16, 5462 * 256, 128, None) == INVALID
    assert "allocation-free limit" in kaio.last_error()
    q = list(p)
    q[4] += 2
    assert L.kaio_qkv_project_int4_noalloc(*q, 16, 128, 256, None) == MISALIGNED


def test_dequant_group_validation_order(L):
    """Checks in the page's order: element types, sizes and group, the empty
    problem (Ok with null pointers), then pointers."""
    F16, F32, F64, BF16, S8, U8 = (kaio.KAIO_DTYPE_F16, kaio.KAIO_DTYPE_F32, kaio.KAIO_DTYPE_F64,
                                   kaio.KAIO_DTYPE_BF16, kaio.KAIO_DTYPE_S8, kaio.KAIO_DTYPE_U8)
    bwd, fwd = L.kaio_dequantize_per_group_backward, L.kaio_dequantize_per_group
    dy, sc, dx = 0x10000000, 0x20000000, 0x30000000
    assert bwd(S8, S8, 2, 8, 4, dy, sc, dx, None) == INVALID and "float type" in kaio.last_error()
    assert bwd(F16, F32, 2, 8, 4, dy, sc, dx, None) == INVALID and "S8 or U8" in kaio.last_error()
    assert bwd(F16, S8, -1, 8, 4, dy, sc, dx, None) == INVALID and "non-negative" in kaio.last_error()
    assert bwd(F16, S8, 2, 8, 0, dy, sc, dx, None) == INVALID and "> 0" in kaio.last_error()
    assert bwd(F16, S8, 2, 10, 4, dy, sc, dx, None) == INVALID and "multiple of group" in kaio.last_error()
    assert bwd(F16, S8, 0, 8, 4, None, None, None, None) == kaio.KAIO_OK
    assert fwd(U8, BF16, 3, 0, 4, None, None, None, None) == kaio.KAIO_OK
    assert bwd(F16, S8, 2, 8, 4, None, sc, dx, None) == INVALID and "null" in kaio.last_error()
    assert bwd(F32, S8, 2, 8, 4, dy + 2, sc, dx, None) == MISALIGNED
    assert bwd(F64, S8, 2, 8, 4, dy, sc + 4, dx, None) == MISALIGNED
    assert fwd(S8, F16, 2, 8, 4, dy + 1, sc, dx, None) != MISALIGNED      # int8 input: any address
    assert bwd(F16, S8, 2, 8, 4, dy, sc, sc + 2, None) == INVALID and "overlaps scale" in kaio.last_error()
    assert bwd(F16, S8, 2, 8, 4, dy, sc, dy + 2, None) == INVALID and "overlaps" in kaio.last_error()
    assert fwd(S8, F16, 2, 8, 4, dy, sc, dy, None) == INVALID and "overlaps" in kaio.last_error()
    # exactly in place passes the argument checks; without a GPU it then fails on CUDA
    st = bwd(F16, S8, 2, 8, 4, dy, sc, dy, None)
    assert st != INVALID or "overlap" not in kaio.last_error()


def qkv8(L, M=16, N=128, K=256, ptrs=None, scales=(1.0, 1.0, 1.0), stream=None):
    p = list(ptrs) if ptrs is not None else [ptr(i) for i in range(7)]
    return L.kaio_qkv_project_int8(*p[:4], *scales, *p[4:], M, N, K, stream)


def test_int8_entry_validation(L):
    for i in range(7):                                   # x, 3 weights, 3 outputs
        p = [ptr(j) for j in range(7)]
        p[i] = None
        assert qkv8(L, ptrs=p) == INVALID and "null" in kaio.last_error()
    for K in (64, 130, 200, 4):
        assert qkv8(L, K=K) == INVALID and "multiple of 128" in kaio.last_error()
    for N in (1, 4, 12, 130):
        assert qkv8(L, N=N) == INVALID and "N (" in kaio.last_error()
    for i in range(7):
        p = [ptr(j) for j in range(7)]
        p[i] += 8
        assert qkv8(L, ptrs=p) == MISALIGNED
    p = [ptr(j) for j in range(7)]
    p[4] = p[0] + 16                                      # q overlaps x
    assert qkv8(L, ptrs=p) == INVALID and "overlaps input x" in kaio.last_error()
    p = [ptr(j) for j in range(7)]
    p[6] = p[1] + 64                                      # v overlaps w_q_packed
    assert qkv8(L, ptrs=p) == INVALID and "w_q_packed" in kaio.last_error()
    # the packed weights are [K/4, N] words: v right after a [K/4, N] w_q is fine
    p = [ptr(j) for j in range(7)]
    p[6] = p[1] + 256 // 4 * 128 * 4
    assert qkv8(L, ptrs=p) not in (INVALID, MISALIGNED)
    # scales are passed by value and not validated
    assert qkv8(L, scales=(float("nan"), 0.0, -1.0)) not in (INVALID, MISALIGNED)


def test_int8_binding_checks_shapes():
    import torch
    x = torch.zeros(4, 128, dtype=torch.float16)
    with pytest.raises(ValueError, match="CUDA device"):
        w = torch.zeros(32, 8, dtype=torch.int32)
        kaio.qkv_project_int8(x, w, w, w, 1.0, 1.0, 1.0)
    with pytest.raises(ValueError):
        kaio.qkv_project_int8(torch.zeros(4, 100, dtype=torch.float16), w, w, w, 1.0, 1.0, 1.0)


def test_wait_limit_entry_validates_before_touching_cuda(L):
    p = [ptr(i) for i in range(10)]
    assert L.kaio_debug_decode_wait_limit(*p, 17, 128, 256, 0, None) == INVALID   # decode shapes only
    assert "1..16" in kaio.last_error()
    assert L.kaio_debug_decode_wait_limit(*p, 4, 128, 200, 0, None) == INVALID   # K % 128
    q = list(p)
    q[3] = None
    assert L.kaio_debug_decode_wait_limit(*q, 4, 128, 256, 0, None) == INVALID
    assert "null" in kaio.last_error()
