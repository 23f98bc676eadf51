"""CPU oracle for the W4A16 and W8A16 fused QKV projections and the dense f16 matmul.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use it. It shares no code with the CUDA library.

Every function here is pinned by tests under ``tests/test_oracle*.py`` against
facts that do not come from the oracle itself (hand-written bit patterns,
exact rational arithmetic, identities and closed forms).
"""
from .w4a16 import (  # noqa: F401
    GROUP_SIZE,
    unpack_int4,
    pack_int4,
    rn_f16,
    dequant_int4,
    qkv_project_int4_ref,
    qkv_project_int4_rows,
    matmul_ref,
    matmul_rows,
    matmul_backward_ref,
    ulp_f16,
)
from .w8a16 import (  # noqa: F401
    unpack_int8,
    pack_int8,
    dequant_int8,
    qkv_project_int8_ref,
    qkv_project_int8_rows,
)
