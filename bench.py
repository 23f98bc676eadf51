"""Benchmark of the W4A16 fused QKV projection (and the dense tensor-core matmul).

One step = one pass of the hot path over one batch: one kaio_qkv_project_int4
call (Q, K and V together) on the chosen workload. Default workload: the
largest configuration, the prefill projection M = N = K = 4096 (412.3 GFLOP
per step, tensor-core bound); the decode shapes are selected with --config.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl kaio|reference]

Timing: the K steps are captured in one CUDA graph; that window of K steps is
replayed back to back for at least --min-seconds, each replay bracketed by CUDA
events on the launching stream, and the per-step time is that of the median
window (min and max are reported beside it).

Prints one JSON line (rank 0). Under torchrun (N > 1) every rank runs an
independent replica on its own GPU (the projection has no exchange step) and
the value is the total over ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_STEPS = {
    "qkv_decode_m1_k4096_n4096": 200,
    "qkv_m16_k256_n128": 200,
    "qkv_batched_decode_m16_k8192_n8192": 100,
    "qkv_prefill_m4096_k4096_n4096": 20,
    "matmul_f16_m4096_n4096_k4096_fwd_bwd": 20,
    "matmul_f16out_m4096_n4096_k4096_fwd_bwd": 20,
    "qkv8_decode_m1_k4096_n4096": 200,
    "qkv8_batched_decode_m16_k8192_n8192": 100,
    "qkv8_prefill_m4096_k4096_n4096": 20,
    "dequant_bwd_bf16_outer8192_axis8192_g128": 50,
    "dequant_fwd_s8_f16_outer8192_axis8192_g128": 50,
}
CONFIGS = {
    # name: (kind, M, N, K)
    "qkv_decode_m1_k4096_n4096": ("qkv", 1, 4096, 4096),
    "qkv_m16_k256_n128": ("qkv", 16, 128, 256),
    "qkv_batched_decode_m16_k8192_n8192": ("qkv", 16, 8192, 8192),
    "qkv_prefill_m4096_k4096_n4096": ("qkv", 4096, 4096, 4096),
    "matmul_f16_m4096_n4096_k4096_fwd_bwd": ("matmul", 4096, 4096, 4096),
    # the same three GEMMs with the results rounded to f16 in the epilogue
    "matmul_f16out_m4096_n4096_k4096_fwd_bwd": ("matmul16", 4096, 4096, 4096),
    # W8A16 (INT8 weights, one f32 scale per projection)
    "qkv8_decode_m1_k4096_n4096": ("qkv8", 1, 4096, 4096),
    "qkv8_batched_decode_m16_k8192_n8192": ("qkv8", 16, 8192, 8192),
    "qkv8_prefill_m4096_k4096_n4096": ("qkv8", 4096, 4096, 4096),
    # per-group dequantisation: (kind, outer, axis, group)
    "dequant_bwd_bf16_outer8192_axis8192_g128": ("dqbwd", 8192, 8192, 128),
    "dequant_fwd_s8_f16_outer8192_axis8192_g128": ("dqfwd", 8192, 8192, 128),
}
# element types of the per-group dequantisation workloads: (float type, quantised type)
DEQUANT_TYPES = {"dqbwd": ("bf16", "s8"), "dqfwd": ("f16", "s8")}
DEFAULT_CONFIG = "qkv_prefill_m4096_k4096_n4096"
METRIC = "W4A16 QKV TFLOP/s and weight GB/s (1xGB300) as % of roofline"
METRICS = {
    "qkv": METRIC,
    "qkv8": "W8A16 QKV TFLOP/s and weight GB/s (1xGB300) as % of roofline",
    "matmul": "dense f16 tensor-core matmul fwd+bwd TFLOP/s",
    "matmul16": "dense f16 tensor-core matmul fwd+bwd, f16 results, TFLOP/s",
    "dqbwd": "per-group dequantisation backward GB/s (dy + scale read, dx written)",
    "dqfwd": "per-group dequantisation GB/s (q + scale read, out written)",
}


def config_shape(kind, a, b, c):
    if kind in DEQUANT_TYPES:
        return {"outer": a, "axis": b, "group": c}
    return {"M": a, "N": b, "K": c}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1024 * 1024


def qkv_bytes(m, n, k):
    weights = 3 * (k // 8) * n * 4 + 3 * (k // 128) * n * 2     # packed + scales
    other = m * k * 2 + 3 * m * n * 2                             # x in, q/k/v out
    return weights, other


def qkv8_bytes(m, n, k):
    weights = 3 * (k // 4) * n * 4                                # packed INT8 words
    other = m * k * 2 + 3 * m * n * 2
    return weights, other


def qkv_flops(m, n, k):
    return 3 * 2 * m * n * k


def dequant_bytes(kind, outer, axis, group):
    """Algorithmic bytes of one per-group dequantisation call: the input and
    the scales read once, the output written once."""
    fdt, _ = DEQUANT_TYPES[kind]
    fsz = {"f32": 4, "f64": 8, "f16": 2, "bf16": 2}[fdt]
    in_sz = fsz if kind == "dqbwd" else 1
    return outer * axis * (in_sz + fsz) + outer * (axis // group) * fsz


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


KERNEL_HEADERS = ("kaio_device.cuh", "kaio_internal.h")


def kernel_source_sha(kernel_file: str) -> str:
    """First 16 hex digits of the sha256 over a kernel's source file followed by
    the device headers every kernel file includes."""
    csrc = os.path.join(ROOT, "qkv_projection_gb300", "csrc")
    h = hashlib.sha256()
    for f in (kernel_file,) + KERNEL_HEADERS:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profile_traffic(kernel_file: str, config: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, if that summary was taken from the current kernel source."""
    csrc = os.path.join(ROOT, "qkv_projection_gb300", "csrc")
    srcs = [os.path.join(csrc, f) for f in (kernel_file,) + KERNEL_HEADERS]
    summary = os.path.join(ROOT, "profiles", f"{config}.md")
    if not (all(os.path.exists(f) for f in srcs) and os.path.exists(summary)):
        return None
    sha = kernel_source_sha(kernel_file)
    text = open(summary).read()
    m_sha = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]{16})", text)
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_sha or not m_b or m_sha.group(1) != sha:
        return None
    return float(m_b.group(1))


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu),
                 "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                 "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                 "clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        w0, w1 = getattr(self, "window", (float("-inf"), float("inf")))
        inside = [l for t, l in self.lines if w0 <= t <= w1]
        for line in inside or [l for _, l in self.lines]:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 6:
                continue
            try:
                mhz.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for name, v in zip(names, parts[2:6]):
                if v.lower() == "active":
                    reasons.add(name)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        mhz.sort()
        return {"sm_mhz": mhz[len(mhz) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(mhz)}


# ---------------------------------------------------------------- distributed
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_init(ws):
    if ws <= 1:
        return None
    import torch.distributed as dist
    backend = "nccl"
    try:
        import torch
        if not torch.cuda.is_available():
            backend = "gloo"
    except Exception:
        backend = "gloo"
    dist.init_process_group(backend=backend)
    return dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, value, device):
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- kaio arm
def run_kaio(args, cfg_name, ws, rank, local, dist):
    import numpy as np
    import torch

    from qkv_projection_gb300 import kaio
    from qkv_projection_gb300.inputs import dense_inputs, qkv_inputs, weight_sets

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    kind, M, N, K = CONFIGS[cfg_name]
    peaks, peak_src = load_peaks()
    stream = torch.cuda.Stream(device=device)

    def dev(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint32:
            a = a.view(np.int32)
        return torch.from_numpy(a).to(device)

    if kind == "qkv":
        wbytes, obytes = qkv_bytes(M, N, K)
        inp = qkv_inputs(M, N, K, seed=0)
        # Rotate among weight sets totalling >= 3x L2 so each launch streams its
        # weights from HBM (and at least 2 sets even when one set exceeds L2).
        nsets = max(2, -(-3 * L2_BYTES // wbytes))
        sets = [tuple(dev(a) for a in (inp.wq, inp.wk, inp.wv, inp.sq, inp.sk, inp.sv))]
        for ws_ in weight_sets(N, K, nsets - 1, seed=1):
            sets.append(tuple(dev(a) for a in ws_))
        x = dev(inp.x)
        # Q, K and V as three views of one [3, M, N] buffer, so that the e2e
        # step reads the whole result back with one copy.
        out_buf = torch.empty((3, M, N), dtype=torch.float16, device=device)
        outs = [out_buf[j] for j in range(3)]
        lib = kaio.lib()
        ptr_sets = [[t.data_ptr() for t in s] for s in sets]
        xo = [x.data_ptr()] + [o.data_ptr() for o in outs]
        sp = int(stream.cuda_stream)

        def step(i):
            w = ptr_sets[i % len(ptr_sets)]
            st = lib.kaio_qkv_project_int4(xo[0], w[0], w[1], w[2], w[3], w[4], w[5],
                                           xo[1], xo[2], xo[3], M, N, K, sp)
            if st:
                raise kaio.KaioError(st, kaio.last_error())

        def e2e_outs():
            buf = torch.empty((3, M, N), dtype=torch.float16, device=device)
            return [buf, [buf[j] for j in range(3)]]   # read back buf; the call writes its views

        def e2e_call(i, ins, res):
            kaio.qkv_project_int4(ins[0], *sets[i % len(sets)], out=res[1], stream=stream)
        e2e_case = ([x], e2e_outs, e2e_call, {"weights_resident": True})

        units_bytes = wbytes
        alg_bytes = wbytes + obytes
        flops = qkv_flops(M, N, K)
        kernel_file = "tc_decode.cu" if kaio.qkv_path(M) == 0 else "tc_kernels.cu"
        bound = "hbm" if M <= 16 else "tensor"
        launches_per_step = 1
    elif kind == "qkv8":
        from qkv_projection_gb300.inputs import qkv_int8_inputs, weight_sets_int8
        wbytes, obytes = qkv8_bytes(M, N, K)
        inp = qkv_int8_inputs(M, N, K, seed=0)
        nsets = max(2, -(-3 * L2_BYTES // wbytes))
        sets = [tuple(dev(w) for w in inp.weights())]
        for ws_ in weight_sets_int8(N, K, nsets - 1, seed=1):
            sets.append(tuple(dev(w) for w in ws_))
        x = dev(inp.x)
        out_buf = torch.empty((3, M, N), dtype=torch.float16, device=device)
        outs = [out_buf[j] for j in range(3)]
        lib = kaio.lib()
        ptr_sets = [[t.data_ptr() for t in s_] for s_ in sets]
        xo = [x.data_ptr()] + [o.data_ptr() for o in outs]
        sc = inp.scales()
        sp = int(stream.cuda_stream)

        def step(i):
            w = ptr_sets[i % len(ptr_sets)]
            kaio.check(lib.kaio_qkv_project_int8(xo[0], w[0], w[1], w[2], sc[0], sc[1], sc[2],
                                                 xo[1], xo[2], xo[3], M, N, K, sp))

        def e2e_outs():
            buf = torch.empty((3, M, N), dtype=torch.float16, device=device)
            return [buf, [buf[j] for j in range(3)]]   # read back buf; the call writes its views

        def e2e_call(i, ins, res):
            kaio.qkv_project_int8(ins[0], *sets[i % len(sets)], *sc, out=res[1], stream=stream)
        e2e_case = ([x], e2e_outs, e2e_call, {"weights_resident": True})

        units_bytes = wbytes
        alg_bytes = wbytes + obytes
        flops = qkv_flops(M, N, K)
        kernel_file = "tc_decode.cu" if M <= 16 else "tc_kernels.cu"
        bound = "hbm" if M <= 16 else "tensor"
        launches_per_step = 1
    elif kind in DEQUANT_TYPES:
        from qkv_projection_gb300.inputs import dequant_group_inputs
        outer, axis, group = M, N, K
        fdt, qdt = DEQUANT_TYPES[kind]
        dy, q, sc = dequant_group_inputs(outer, axis, group, fdt, seed=0, q_dtype=qdt)
        tdt = {"f32": torch.float32, "f64": torch.float64, "f16": torch.float16, "bf16": torch.bfloat16}[fdt]

        def fdev(a):
            return dev(a.view(np.int16)).view(tdt) if fdt == "bf16" else dev(a)
        # Two input/output sets, alternated, so that every call streams from HBM
        # (each set alone is at least L2-sized).
        src = fdev(dy) if kind == "dqbwd" else dev(q)
        S = fdev(sc)
        srcs = [src, src.clone()]
        outs = [torch.empty((outer, axis), dtype=tdt, device=device) for _ in range(2)]
        lib = kaio.lib()
        sp = int(stream.cuda_stream)
        fcode = kaio._float_code(tdt)
        qcode = kaio.KAIO_DTYPE_S8 if qdt == "s8" else kaio.KAIO_DTYPE_U8

        def step(i):
            a, o = srcs[i % 2], outs[i % 2]
            if kind == "dqbwd":
                kaio.check(lib.kaio_dequantize_per_group_backward(fcode, qcode, outer, axis, group, a.data_ptr(),
                                                                  S.data_ptr(), o.data_ptr(), sp))
            else:
                kaio.check(lib.kaio_dequantize_per_group(qcode, fcode, outer, axis, group, a.data_ptr(),
                                                         S.data_ptr(), o.data_ptr(), sp))

        def e2e_outs():
            return [torch.empty_like(outs[0])]

        def e2e_call(i, ins, res):
            if kind == "dqbwd":
                kaio.dequantize_per_group_backward(ins[0], ins[1], group, out=res[0], stream=stream)
            else:
                kaio.dequantize_per_group(ins[0], ins[1], group, out=res[0], stream=stream)
        e2e_case = ([src, S], e2e_outs, e2e_call, {})

        wbytes = 0
        units_bytes = dequant_bytes(kind, outer, axis, group)
        alg_bytes = units_bytes
        flops = outer * axis
        kernel_file = "dequant_group.cu"
        bound = "hbm"
        launches_per_step = 1
    else:
        a, b, g = dense_inputs(M, N, K, seed=0)
        A, B, G = dev(a), dev(b), dev(g)
        out_t = torch.float16 if kind == "matmul16" else torch.float32
        C = torch.empty((M, N), dtype=out_t, device=device)
        dA = torch.empty((M, K), dtype=out_t, device=device)
        dB = torch.empty((K, N), dtype=out_t, device=device)
        lib = kaio.lib()
        sp = int(stream.cuda_stream)
        fwd = lib.kaio_matmul_tc_f16 if kind == "matmul16" else lib.kaio_matmul_tc
        bwd = lib.kaio_matmul_tc_backward_f16 if kind == "matmul16" else lib.kaio_matmul_tc_backward

        def step(i):
            kaio.check(fwd(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, sp))
            kaio.check(bwd(A.data_ptr(), B.data_ptr(), G.data_ptr(), dA.data_ptr(), dB.data_ptr(),
                           M, N, K, sp))

        def e2e_outs():
            return [torch.empty_like(C), torch.empty_like(dA), torch.empty_like(dB)]

        def e2e_call(i, ins, res):
            kaio.matmul_tc(ins[0], ins[1], out=res[0], stream=stream, out_dtype=out_t)
            kaio.matmul_tc_backward(ins[0], ins[1], ins[2], stream=stream, out_dtype=out_t, out=(res[1], res[2]))
        e2e_case = ([A, B, G], e2e_outs, e2e_call, {})

        wbytes = 0
        units_bytes = 0
        alg_bytes = 3 * (2 * M * K * 2 + M * N * (2 if kind == "matmul16" else 4))
        flops = 3 * 2 * M * N * K
        kernel_file = "tc_kernels.cu"
        bound = "tensor"
        launches_per_step = 3

    # Warm-up.
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            step(i)
    stream.synchronize()

    # Host cost of one C-ABI call (validation, residency checks, tensor maps,
    # launch): a host loop of calls with no synchronisation in between.
    host_us = None
    if kind in ("qkv", "qkv8"):
        n_host = 200
        with torch.cuda.stream(stream):
            h0 = time.perf_counter()
            for i in range(n_host):
                step(i)
            h1 = time.perf_counter()
        stream.synchronize()
        host_us = round((h1 - h0) / n_host * 1e6, 2)

    # One window = the K timed steps, captured in one CUDA graph.
    steps = args.steps
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            for i in range(steps):
                step(i)
    stream.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(2):
            graph.replay()
    stream.synchronize()

    # Replay the window back to back for at least --min-seconds (and at least
    # 5 times), each replay bracketed by events on the launching stream.
    probe0 = torch.cuda.Event(enable_timing=True)
    probe1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        probe0.record(stream)
        graph.replay()
        probe1.record(stream)
    probe1.synchronize()
    one_ms = max(probe0.elapsed_time(probe1), 1e-3)
    windows = int(min(20000, max(5, args.min_seconds * 1e3 / one_ms)))
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(windows + 1)]

    barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        time.sleep(0.3)
        w0 = time.perf_counter()
        with torch.cuda.stream(stream):      # replay() launches on the current stream
            evs[0].record(stream)
            for r in range(windows):
                graph.replay()
                evs[r + 1].record(stream)
        evs[-1].synchronize()
        clk.mark(w0, time.perf_counter() + 0.05)
        time.sleep(0.1)
    torch.cuda.synchronize()
    barrier(dist)
    win_ms = sorted(evs[r].elapsed_time(evs[r + 1]) for r in range(windows))
    t_ms = win_ms[len(win_ms) // 2]
    t_max_ms = max_over_ranks(dist, t_ms, device)
    per_step_s = t_max_ms / 1e3 / steps
    window_stats = {"windows": windows, "steps_per_window": steps,
                    "ms_per_step_min": round(win_ms[0] / steps, 6),
                    "ms_per_step_max": round(win_ms[-1] / steps, 6)}

    # End to end through the public API: per step, copy the step's inputs in
    # from pinned host memory, make the call(s), read every result back into
    # pinned host memory. Steps that move many bytes are pipelined the way a
    # serving loop runs them: inputs in on one stream, the calls on the compute
    # stream, results out on a third, with two sets of device buffers and
    # events ordering each buffer's reuse, so step i's copies overlap steps
    # i-1 and i+1. Small steps (decode) run in order on the compute stream:
    # there the per-step host work of the extra streams and events costs more
    # than the copies it would hide.
    e2e = None
    if not args.no_e2e:
        dev_in, make_outs, call, extra = e2e_case
        def tensors(res):
            return [r for r in res if isinstance(r, torch.Tensor)]   # what a step reads back

        step_bytes = sum(t.numel() * t.element_size() for t in dev_in) + \
            sum(t.numel() * t.element_size() for t in tensors(make_outs()))
        pipelined = step_bytes >= (16 << 20)
        nb = 2 if pipelined else 1
        h_in = [t.cpu().pin_memory() for t in dev_in]
        d_in = [[torch.empty_like(t) for t in dev_in] for _ in range(nb)]
        d_out = [make_outs() for _ in range(nb)]
        h_out = [[torch.empty(r.shape, dtype=r.dtype).pin_memory() for r in tensors(d_out[b])] for b in range(nb)]
        r_out = [tensors(d_out[b]) for b in range(nb)]
        s_in, s_out = (torch.cuda.Stream(device), torch.cuda.Stream(device)) if pipelined else (stream, stream)
        ev_in = [torch.cuda.Event() for _ in range(nb)]
        ev_comp = [torch.cuda.Event() for _ in range(nb)]
        ev_out = [torch.cuda.Event() for _ in range(nb)]
        e_steps = max(args.steps, 200 if M <= 16 and kind in ("qkv", "qkv8") else 20)
        h2d = sum(t.numel() * t.element_size() for t in h_in)

        def e2e_step(i):
            if not pipelined:                        # runs inside the compute stream's context
                for d, h in zip(d_in[0], h_in):
                    d.copy_(h, non_blocking=True)
                call(i, d_in[0], d_out[0])
                for h, r in zip(h_out[0], r_out[0]):
                    h.copy_(r, non_blocking=True)
                return
            b = i % nb
            s_in.wait_event(ev_comp[b])              # step i - nb has finished reading d_in[b]
            with torch.cuda.stream(s_in):
                for d, h in zip(d_in[b], h_in):
                    d.copy_(h, non_blocking=True)
                ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            stream.wait_event(ev_out[b])             # step i - nb's results have left d_out[b]
            with torch.cuda.stream(stream):
                call(i, d_in[b], d_out[b])
                ev_comp[b].record(stream)
            s_out.wait_event(ev_comp[b])
            with torch.cuda.stream(s_out):
                for h, r in zip(h_out[b], r_out[b]):
                    h.copy_(r, non_blocking=True)
                ev_out[b].record(s_out)

        with torch.cuda.stream(stream):
            for i in range(3):
                e2e_step(i)
            torch.cuda.synchronize(device)
            barrier(dist)
            t0 = time.perf_counter()
            for i in range(e_steps):
                e2e_step(i)
            torch.cuda.synchronize(device)
            t1 = time.perf_counter()
        te = max_over_ranks(dist, t1 - t0, device)
        d2h = sum(t.numel() * t.element_size() for t in h_out[0])
        if kind in ("matmul", "matmul16") or bound == "tensor":
            e2e = {"value": round(ws * flops * e_steps / te / 1e12, 3), "unit": "TFLOP/s"}
        else:
            e2e = {"value": round(ws * units_bytes * e_steps / te / 1e9, 3), "unit": "GB/s"}
        e2e.update({"h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e_steps,
                    "pipelining": "3 streams (in, compute, out), 2 buffer sets" if pipelined else "none (one stream)",
                    **extra})

    if rank != 0:
        return None

    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    tc_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))   # f16 = bf16 rate
    if bound == "hbm":
        achieved = alg_bytes / per_step_s / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4), "peak_source": peak_src}
    else:
        achieved = flops / per_step_s / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": tc_peak, "unit": "TFLOP/s",
                "frac": round(achieved / tc_peak, 4), "peak_source": peak_src + " bf16 burst (f16 = bf16 rate)"}
    roof["traffic"] = profile_traffic(kernel_file, cfg_name)

    if kind in ("qkv", "qkv8") and bound == "hbm":
        value = ws * wbytes / per_step_s / 1e9
        unit = "GB/s"
    elif kind in DEQUANT_TYPES:
        value = ws * units_bytes / per_step_s / 1e9
        unit = "GB/s"
    else:
        value = ws * flops / per_step_s / 1e12
        unit = "TFLOP/s"
    metric = METRICS[kind]
    dtype = {"qkv": "f16 (int4 weights, f32 accumulate)", "qkv8": "f16 (int8 weights, f32 accumulate)", "matmul": "f16 (f32 accumulate)",
             "matmul16": "f16 (f32 accumulate, f16 results)",
             "dqbwd": "bf16 (products exact in f32, rounded once)",
             "dqfwd": "int8 -> f16 (products exact in f32, rounded once)"}[kind]
    l2 = {"qkv": "inputs larger than L2 (weight sets rotated)",
          "qkv8": "inputs larger than L2 (weight sets rotated)",
          "dqbwd": "two input/output sets of 2x128 MiB alternated (inputs larger than L2)",
          "dqfwd": "two input/output sets of 64+128 MiB alternated (inputs larger than L2)"}.get(
              kind, "operands 32 MiB each; no flush (compute-bound)")
    shape = config_shape(kind, M, N, K)
    line = {
        "metric": metric,
        "value": round(value, 3),
        "unit": unit,
        "n_gpus": ws,
        "steps": steps,
        "warmup": max(args.warmup, 3),
        "ms_per_step": round(per_step_s * 1e3, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dtype,
        "data": "synthetic (seeded; weights rotate over sets totalling >= 3x L2)" if kind in ("qkv", "qkv8") else
                "synthetic (seeded)",
        "config": {"workload": cfg_name, **shape, "parallelism": f"replicas x{ws}", "l2": l2},
        "tflops": round(ws * flops / per_step_s / 1e12, 3) if kind not in DEQUANT_TYPES else None,
        "weight_gbs": round(ws * wbytes / per_step_s / 1e9, 3) if kind in ("qkv", "qkv8") else None,
        # packed words alone (INT4: without the group scales; INT8 has no scale tensors)
        "packed_weight_gbs": (round(ws * 3 * (shape["K"] * (4 if kind == "qkv" else 8) // 32) * shape["N"] * 4
                                    / per_step_s / 1e9, 3) if kind in ("qkv", "qkv8") else None),
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": windows * steps * launches_per_step,
        "timing": {**window_stats, "gpu_launches_per_window": steps * launches_per_step,
                   "note": "ms_per_step is the median window's; gpu_launches counts every window timed"},
        "host_us_per_call": host_us,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline and ws == 1:
        line["cpu_baseline"] = cpu_baseline(cfg_name, budget_s=args.cpu_budget)
    return line


# ---------------------------------------------------------------- oracle arm
def oracle_sample(cfg_name, frac):
    """One oracle evaluation of workload `cfg_name` on a sample of fraction
    `frac`; returns (step, amount, n, extent, noun, unit) where `amount` is the
    work one step does in the metric's unit (bytes for GB/s, FLOPs for
    TFLOP/s) and n of extent `noun`s were sampled."""
    import numpy as np

    import oracle

    kind, M, N, K = CONFIGS[cfg_name]
    if kind in DEQUANT_TYPES:
        from oracle import dequant_group as dg
        from qkv_projection_gb300.inputs import dequant_group_inputs
        fdt, qdt = DEQUANT_TYPES[kind]
        rows = max(1, int(round(M * frac)))
        dy, q, sc = dequant_group_inputs(rows, N, K, fdt, seed=0, q_dtype=qdt)

        def step():
            if kind == "dqbwd":
                dg.dequantize_per_group_backward_ref(dy, sc, K, fdt)
            else:
                dg.dequantize_per_group_ref(q, sc, K, fdt)
        return step, dequant_bytes(kind, rows, N, K), rows, M, "rows", "GB/s"
    if kind in ("matmul", "matmul16"):
        from qkv_projection_gb300.inputs import dense_inputs
        a, b, g = dense_inputs(M, N, K, seed=0)
        r = max(1, int(round(M * frac)))
        c = max(1, int(round(N * frac)))
        rows, cols = np.arange(r), np.arange(c)

        def step():
            oracle.matmul_rows(a, b, rows)                        # rows of C = A B
            oracle.matmul_rows(g, np.ascontiguousarray(b.T), rows)  # rows of dA = G B^T
            oracle.matmul_ref(np.ascontiguousarray(a.T), np.ascontiguousarray(g[:, cols]))  # columns of dB = A^T G
        return step, 2 * r * K * N + 2 * r * N * K + 2 * M * K * c, r, M, "rows (and columns of dB)", "TFLOP/s"
    if M > 16:
        # Tensor-bound shapes: a seeded sample of output rows (always rows 0, 1,
        # 127, 128 and M-1), in FLOPs of the rows computed.
        r = max(5, int(round(M * frac)))
        rows = np.unique(np.concatenate([
            np.random.default_rng(0).choice(M, r, replace=False), [0, 1, 127, 128, M - 1]]))
        if kind == "qkv8":
            from qkv_projection_gb300.inputs import qkv_int8_inputs
            inp8 = qkv_int8_inputs(M, N, K, seed=0)

            def step():
                oracle.qkv_project_int8_rows(*inp8.args(), rows)
        else:
            from qkv_projection_gb300.inputs import qkv_inputs
            inp = qkv_inputs(M, N, K, seed=0)

            def step():
                oracle.qkv_project_int4_rows(*inp.__dict__.values(), rows)
        return step, qkv_flops(len(rows), N, K), len(rows), M, "rows", "TFLOP/s"
    ncols = max(8, int(round(N * frac)) // 8 * 8)
    if kind == "qkv8":
        from qkv_projection_gb300.inputs import qkv_int8_inputs
        inp8 = qkv_int8_inputs(M, N, K, seed=0)
        ws8 = [np.ascontiguousarray(w[:, :ncols]) for w in inp8.weights()]

        def step():
            oracle.qkv_project_int8_ref(inp8.x, *ws8, *inp8.scales())
        return step, qkv8_bytes(M, ncols, K)[0], ncols, N, "columns", "GB/s"
    from qkv_projection_gb300.inputs import qkv_inputs
    inp = qkv_inputs(M, N, K, seed=0)
    sub = [inp.x] + [np.ascontiguousarray(w[:, :ncols]) for w in inp.weights()] + \
          [np.ascontiguousarray(s_[:, :ncols]) for s_ in inp.scales()]

    def step():
        oracle.qkv_project_int4_ref(*sub)
    return step, qkv_bytes(M, ncols, K)[0], ncols, N, "columns", "GB/s"


def _per_unit(amount, unit):
    return amount / (1e12 if unit == "TFLOP/s" else 1e9)


def cpu_baseline(cfg_name, budget_s=15.0):
    kind, M, N, K = CONFIGS[cfg_name]
    frac = (1.0 / 64 if kind in DEQUANT_TYPES else 1.0 / 32 if kind in ("matmul", "matmul16")
            else 1.0 / 64 if M > 16 else 1.0 if N * K <= 4096 * 4096 else 0.125)
    step, amount, n, extent, noun, unit = oracle_sample(cfg_name, frac)
    t0 = time.perf_counter()
    step()
    one = time.perf_counter() - t0
    reps = max(1, int(budget_s / max(one, 1e-6)))
    t0 = time.perf_counter()
    for _ in range(reps):
        step()
    dt = time.perf_counter() - t0
    return {"value": round(_per_unit(amount, unit) * reps / dt, 5), "unit": unit, "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{reps} oracle evaluations of {cfg_name} on {n} of {extent} {noun} "
                      f"(numpy float64; BLAS may use up to {os.cpu_count()} threads)"}


def run_reference(args, cfg_name, ws, rank):
    kind, M, N, K = CONFIGS[cfg_name]
    if rank != 0:
        return None
    # Size each step's sample so that the whole run takes about --ref-seconds.
    total_steps = args.steps + max(args.warmup, 3)
    probe, _, n_probe, extent, _, _ = oracle_sample(cfg_name, 1.0 / 64)
    t0 = time.perf_counter()
    probe()
    per_unit = (time.perf_counter() - t0) / n_probe
    frac = min(1.0, max(8.0 / extent, args.ref_seconds / total_steps / max(per_unit, 1e-9) / extent))
    step, amount, n, extent, noun, unit = oracle_sample(cfg_name, frac)
    for _ in range(max(args.warmup, 3)):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = _per_unit(amount, unit) * args.steps / dt
    sample = f"each step: one oracle evaluation of {cfg_name} on {n} of {extent} {noun} (numpy float64)"
    return {
        "impl": "reference", "metric": METRICS[kind], "value": round(value, 6), "unit": unit,
        "n_gpus": ws, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": round(dt / args.steps * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": cfg_name, **config_shape(kind, M, N, K)},
        "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": os.cpu_count(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["kaio", "reference"], default="kaio")
    ap.add_argument("--config", choices=sorted(CONFIGS), default=DEFAULT_CONFIG)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--min-seconds", type=float, default=2.0,
                    help="replay the K-step window for at least this long (median window reported)")
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="approximate length of the --impl reference run")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = DEFAULT_STEPS[args.config]
    ws, rank, local = dist_env()
    if args.impl == "reference":
        line = run_reference(args, args.config, ws, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    dist = dist_init(ws)
    line = run_kaio(args, args.config, ws, rank, local, dist)
    if line is not None:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
