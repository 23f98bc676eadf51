"""GB300-native W4A16 fused QKV projection and dense f16 tensor-core matmul.

The compute lives in ``libkaio_qkv.so`` (hand-written CUDA for sm_103a) behind
a C ABI declared in ``include/kaio_qkv.h``. ``qkv_projection_gb300.kaio`` is the
thin Python binding (argument marshalling only).
"""
