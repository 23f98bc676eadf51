import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_100 family) and the built library")


def pytest_collection_modifyitems(config, items):
    # GPU tests need both a device and the compiled library; on a machine
    # without a GPU they are skipped rather than failed.
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session", autouse=True)
def _library_built():
    """Compile the C-ABI library once if it is not there yet (nvcc cross-compiles
    for sm_103a without a GPU), so host-side tests of the boundary can load it."""
    from qkv_projection_gb300 import build
    if not os.path.exists(build.LIB):
        build.build()
    yield
