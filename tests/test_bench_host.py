"""Host-side checks of bench.py (no GPU): the oracle arm on every workload kind
and the work each oracle sample claims."""
import os
import sys
from types import SimpleNamespace

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


@pytest.mark.parametrize("cfg", ["qkv8_decode_m1_k4096_n4096", "dequant_fwd_s8_f16_outer8192_axis8192_g128",
                                 "matmul_f16_m4096_n4096_k4096_fwd_bwd"])
def test_reference_arm_line(cfg):
    kind = bench.CONFIGS[cfg][0]
    args = SimpleNamespace(steps=1, warmup=3, ref_seconds=0.5)
    d = bench.run_reference(args, cfg, 1, 0)
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["metric"] == bench.METRICS[kind]
    assert d["unit"] == ("TFLOP/s" if kind in ("matmul", "matmul16") else "GB/s")
    assert d["config"]["workload"] == cfg
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["unit"] == d["unit"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert bench.run_reference(args, cfg, 2, 1) is None          # only rank 0 reports


def test_oracle_sample_amounts():
    # projections: weight bytes of the sampled columns
    _, amount, n, extent, noun, unit = bench.oracle_sample("qkv_m16_k256_n128", 0.5)
    assert (n, extent, noun, unit) == (64, 128, "columns", "GB/s")
    assert amount == 3 * (256 // 8) * 64 * 4 + 3 * (256 // 128) * 64 * 2
    _, amount, n, _, _, _ = bench.oracle_sample("qkv8_decode_m1_k4096_n4096", 1 / 64)
    assert amount == 3 * (4096 // 4) * n * 4
    # dequantisation: all bytes of the sampled rows
    _, amount, n, extent, noun, _ = bench.oracle_sample("dequant_bwd_bf16_outer8192_axis8192_g128", 1 / 1024)
    assert (n, extent, noun) == (8, 8192, "rows")
    assert amount == 8 * 8192 * (2 + 2) + 8 * 64 * 2
    # dense: FLOPs of the sampled rows of C and dA and columns of dB
    _, amount, n, extent, _, unit = bench.oracle_sample("matmul_f16_m4096_n4096_k4096_fwd_bwd", 1 / 512)
    assert (n, extent, unit) == (8, 4096, "TFLOP/s")
    assert amount == 2 * 8 * 4096 * 4096 * 3
