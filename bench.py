#!/usr/bin/env python
"""Decode-step weight-streaming benchmark on GB300.

A step is one pass of the whole hot path over one decode token: every weight
matrix of the model streamed once by the library's GEMV kernels, each GEMV
with its own activation vector (all calls through the C ABI, captured once
into a CUDA graph and replayed).

Default workload (--workload qwen_bf16): the Qwen2.5-7B-shaped BF16 decode
step at batch 1 -- 28 layers x (qkv 4608x3584, o 3584x3584, gate and up
18944x3584, down 3584x18944) + LM head 152064x3584 = 141 GEMVs and 14.14 GB
of weights per step (about 110x the L2, so no matrix is still cached when the
step reaches it again). Synthetic seeded data (no checkpoint).

The same JSON line carries, under "configs", the other configurations the
metric is quoted on, each on its autotuned plans: the BF16 2048x2048 GEMV,
the four TinyLlama-shaped INT4 group-64 matrices (and the TinyLlama INT4
step), the skinny BF16 GEMM over the Qwen2.5-7B MLP shapes at M = 1 ... 256,
and the AWQ-style INT4 Qwen2.5-7B step at M = 1, 16 and 64 (codes repacked at
load time). --no-extras leaves them out.

Metric: achieved HBM GB/s = algorithmic bytes of the step (weights + scales
+ x) / step time, and the weight-stream ms per token.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Multi-GPU: launched by torchrun, one independent replica per GPU (the GEMV
has no exchange step); the slowest rank's time is used.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import re
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from memory_bound_weight_gb300 import workloads as wl  # noqa: E402

FALLBACK_HBM_GBS = 6778.3  # the machine's measured copy bandwidth, recorded copy
NOMINAL_HBM_GBS = 7900.0  # the GB300's nominal HBM3e bandwidth (context only; fractions use the measured peak)
FALLBACK_BF16_TFLOPS = 1752.2  # the pool's measured sustained cuBLAS bf16, recorded copy
# DRAM bytes (read + write) per launch of the step's dominant kernel from one
# ncu capture, keyed by (kernel source sha, shape, weight format); a changed
# kernel gets traffic = null until it is captured again.
TRAFFIC = {
    # the Qwen2.5-7B gate/up matrices (BF16, 18944x3584), the default step's dominant kernel: gemv_rows
    # (8 warps, 3 stages of 4 KB per warp, 2 CTAs per SM), ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,
    # 1 launch: 135,827,712 + 2,765,568 (profiles/gemv_rows_bf16_18944x3584.md); the tuner's other row-stream
    # instantiations on this shape stream the same rows through the same code
    ("f5ed3ed01133743e", "18944x3584", "bf16"): 138593280,
    # the qwen3_int8 step's dominant kernel: the bulk-fed kernel on the fused gate_up matrices (INT8, 19456x2560),
    # 49,933,824 + 0 (same capture; its ncu summary under profiles/)
    ("f5ed3ed01133743e", "19456x2560", "int8_pc"): 49933824,
    # the TinyLlama INT4 step's dominant kernel: gemv_lat on the fused gate_up matrices (INT4 g64, 11264x2048),
    # dram__bytes_read.sum 12,315,392 + dram__bytes_write.sum 0 (its ncu summary under profiles/)
    ("cf3bf3b20ec9aac8", "11264x2048", "int4_g64"): 12315392,
    # the AWQ batch-1 step's dominant kernel: gemv_mma2 on 18944x3584 (AWQ, repacked codes), 35,341,056 + 0
    # (same capture; its ncu summary under profiles/)
    ("fc44b33cdfecb3fc", "18944x3584", "int4_awq_g128"): 35341056,
}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", default="mbw", choices=["mbw", "reference"])
    p.add_argument("--workload", default="qwen_bf16",
                   choices=["tinyllama_int4", "tinyllama_int4_fusedops", "tinyllama_int4_unfused", "qwen_bf16",
                            "qwen_bf16_fused", "qwen_awq", "qwen_awq_repacked", "qwen_awq_repacked_fused",
                            "qwen_awq_fusedops", "qwen3_int8", "bf16_2048"])
    p.add_argument("--batch", type=int, default=1,
                   help="activation rows per GEMV (qwen_awq: AWQ-style INT4 decode at batch M)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--ref-budget", type=float, default=None,
                   help="--impl reference: oracle seconds per step (default: about 20 s over the whole run)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--per-matrix", action="store_true",
                   help="also time each distinct shape on its own: steady state and cold (L2 flushed per call)")
    p.add_argument("--no-shape-timing", action="store_true",
                   help="skip the per-shape timing behind the dominant-kernel roofline (e.g. under a profiler)")
    p.add_argument("--tune", default="step", choices=["step", "shape"],
                   help="step: per-shape autotune, then refine the plans on the whole step graph (default); "
                        "shape: per-shape autotune only")
    p.add_argument("--plans-out", default=None, help="write the tuned plan index of every shape to this JSON file")
    p.add_argument("--plans-from", default=None, help="restore plans from a --plans-out file instead of tuning")
    p.add_argument("--no-extras", action="store_true",
                   help="leave out the other configurations' figures (configs key of the JSON line)")
    p.add_argument("--extras-tune", default="step", choices=["step", "shape"],
                   help="plan tuning of the extra decode steps (TinyLlama INT4, AWQ): refined on the whole step "
                        "(default; a plan that wins its shape alone can slow its neighbours in the chain) or per "
                        "shape only")
    p.add_argument("--profile-range", action="store_true",
                   help="bracket the timed region with cudaProfilerStart/Stop (for ncu --profile-from-start off)")
    return p.parse_args()


# ------------------------------------------------------------- distributed ----
def dist_setup(backend):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group(backend=backend)
    return rank, ws, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(v, ws, device):
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist

    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- helpers ----
def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json, copy kernel)"
    except Exception:  # noqa: BLE001
        return FALLBACK_HBM_GBS, "measured on this pool (recorded copy; MEASURED_PEAKS.json absent)"


def tensor_peak():
    """bf16 dense tensor peak (TFLOP/s): the pool's sustained cuBLAS figure, the
    one for a kernel timed inside a long step."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops_sustained"]), "measured sustained (MEASURED_PEAKS.json, cuBLAS bf16)"
    except Exception:  # noqa: BLE001
        return FALLBACK_BF16_TFLOPS, "measured on this pool (recorded sustained cuBLAS bf16; MEASURED_PEAKS.json absent)"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms in a thread."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.rows = []
        self.proc = None
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except FileNotFoundError:
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.t:
            self.t.join(timeout=5)

    def summary(self, t0, t1):
        rows = [r for (ts, r) in self.rows if t0 <= ts <= t1 and len(r) >= 9]
        window = "timed region"
        if not rows:  # a very short timed region: take the samples around it
            rows = [r for (ts, r) in self.rows if t0 - 1.0 <= ts <= t1 + 1.0 and len(r) >= 9]
            window = "timed region +/- 1 s"
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "window": window}


KERNEL_SOURCES = {"lat": ("gemv_lat.cu", "device.cuh"), "mma2": ("gemv_mma.cu", "device.cuh"),
                  "mma": ("gemv_mma.cu", "device.cuh"), "simt": ("gemv_simt.cu", "device.cuh"),
                  "tma": ("gemv_tma.cu", "device.cuh"), "tcgen05": ("gemm_tc.cu", "device.cuh"),
                  "awq_mma": ("gemv_awq_batch.cu", "device.cuh"), "rows": ("gemv_tma.cu", "device.cuh"),
                  "bulk": ("gemv_tma.cu", "device.cuh")}


def kernel_source_sha(family):
    h = hashlib.sha256()
    for f in KERNEL_SOURCES.get(family, ("device.cuh",)):
        with open(os.path.join(ROOT, "memory_bound_weight_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# -------------------------------------------------------------- workloads ----
class Step:
    """All matrices of one decode step resident on the device, and the calls
    that stream them (each GEMV with its own activation rows X [M][K])."""

    def __init__(self, name, fmt, mats, seed, device, M=1, repacked=False):
        import torch

        import memory_bound_weight_gb300 as mbw
        from memory_bound_weight_gb300 import inputs as gen
        from memory_bound_weight_gb300 import inputs_gpu

        self.name, self.fmt, self.mats, self.M = name, fmt, mats, M
        self.repacked = repacked  # AWQ codes reordered at load time (mbw.repack_int4)
        self.device = device
        sumK = sum(m.K for m in mats)
        sumN = sum(m.N for m in mats)
        self.x = torch.empty(M * sumK, dtype=torch.bfloat16, device=device)
        self.y = torch.empty(M * sumN, dtype=torch.bfloat16, device=device)
        self.calls = []
        ko = no = 0
        for mi, m in enumerate(mats):
            xv = self.x[ko:ko + M * m.K]
            yv = self.y[no:no + M * m.N]
            inputs_gpu.bf16_normal_(xv, seed, gen.stream_id(mi, gen.KIND_X), gen.X_SIGMA)
            xa = xv if M == 1 else xv.view(M, m.K)
            ya = yv if M == 1 else yv.view(M, m.N)
            self.calls.append(device_call(fmt, seed, mi, m.N, m.K, xa, ya, device, m.fuse, M, repacked))
            ko += M * m.K
            no += M * m.N
        self.op = op_of_fmt(fmt) | (mbw.REPACKED if repacked else 0)
        self.bytes_alg = wl.step_bytes_alg(mats, fmt, M)
        self.flops = sum(wl.call_flops(M, m) for m in mats)
        # e2e: the x vectors and the residuals the calls read come from the host
        self.h2d_bytes = 2 * M * sumK + sum(2 * M * m.N for m in mats if m.fuse & wl.FUSE_RESIDUAL)
        self.d2h_bytes = 2 * M * sumN

    def shapes(self):
        """Distinct call kinds (fusion bits, N, K)."""
        return sorted({(m.fuse, m.N, m.K) for m in self.mats})

    def run(self):
        for fn, args, out in self.calls:
            fn(*args, out=out)


def op_of_fmt(fmt):
    import memory_bound_weight_gb300 as mbw

    return {wl.FMT_INT4_G64: mbw.OP_GEMV_INT4_G64, wl.FMT_INT4_AWQ_G128: mbw.OP_GEMV_INT4_AWQ_G128,
            wl.FMT_BF16: mbw.OP_GEMV_BF16, wl.FMT_INT8_PC: mbw.OP_GEMV_INT8_PC}[fmt]


def skey(kind):
    """String key of a call kind (fusion bits, N, K): "NxK" plus its fusions."""
    fz, N, K = kind
    return f"{N}x{K}" + ("+norm" if fz & wl.FUSE_NORM else "") + ("+glu" if fz & wl.FUSE_GLU else "") + \
        ("+res" if fz & wl.FUSE_RESIDUAL else "")


def device_call(fmt, seed, mi, N, K, x, y, device, fuse=0, M=1, repacked=False):
    """(C-ABI call, its inputs, its output) for matrix `mi` of a workload, with
    the matrix generated on the device. A fused call also gets its up matrix,
    norm weight and residual (seeded like the rest). `repacked` (AWQ): the codes
    are reordered once, in place, by the load-time repack, and the call is the
    repacked one."""
    import functools

    import memory_bound_weight_gb300 as mbw
    from memory_bound_weight_gb300 import inputs as gen
    from memory_bound_weight_gb300 import inputs_gpu

    if fuse and fmt == wl.FMT_INT4_AWQ_G128:
        def awq(m):
            c = inputs_gpu.int4_codes(seed, m, N, K, device)
            if repacked:
                mbw.repack_int4(c, out=c)
            return (c, inputs_gpu.f16_group_scales(seed, m, N, K // 128, device),
                    inputs_gpu.u4_zero_points(seed, m, N, K // 128, device))
        c, s, z = awq(mi)
        kw = {"repacked": repacked}
        if fuse & wl.FUSE_GLU:
            kw["up_weights"], kw["up_scales"], kw["up_zeros"] = awq(50000 + mi)
        if fuse & wl.FUSE_NORM:
            g = torch_empty((K,), device)
            inputs_gpu.bf16_normal_(g, seed, gen.stream_id(60000 + mi, gen.KIND_X), gen.X_SIGMA)
            kw["norm_weight"], kw["norm_eps"] = g, 1e-6
        if fuse & wl.FUSE_RESIDUAL:
            r = torch_empty((M, N) if M > 1 else (N,), device)
            inputs_gpu.bf16_normal_(r.view(-1), seed, gen.stream_id(70000 + mi, gen.KIND_X), gen.X_SIGMA)
            kw["residual"] = r
        return functools.partial(mbw.gemv_fused_awq_g128, c, s, z, x, **kw), (), y

    if fuse:
        base = op_of_fmt(fmt)
        W, sc = device_weights(fmt, seed, mi, N, K, device)
        kw = {}
        if fuse & wl.FUSE_GLU:
            kw["up_weights"], kw["up_scales"] = device_weights(fmt, seed, 50000 + mi, N, K, device)
        if fuse & wl.FUSE_NORM:
            g = torch_empty((K,), device)
            inputs_gpu.bf16_normal_(g, seed, gen.stream_id(60000 + mi, gen.KIND_X), gen.X_SIGMA)
            kw["norm_weight"], kw["norm_eps"] = g, 1e-6
        if fuse & wl.FUSE_RESIDUAL:
            r = torch_empty((M, N) if M > 1 else (N,), device)
            inputs_gpu.bf16_normal_(r.view(-1), seed, gen.stream_id(70000 + mi, gen.KIND_X), gen.X_SIGMA)
            kw["residual"] = r
        return functools.partial(mbw.gemv_fused, base, W, sc, x, **kw), (), y

    if fmt == wl.FMT_INT4_G64:
        c = inputs_gpu.int4_codes(seed, mi, N, K, device)
        s = inputs_gpu.f16_group_scales(seed, mi, N, K // 64, device)
        return mbw.gemv_int4_g64, (c, s, x), y
    if fmt == wl.FMT_INT4_AWQ_G128:
        c = inputs_gpu.int4_codes(seed, mi, N, K, device)
        s = inputs_gpu.f16_group_scales(seed, mi, N, K // 128, device)
        z = inputs_gpu.u4_zero_points(seed, mi, N, K // 128, device)
        if repacked:
            mbw.repack_int4(c, out=c)
            return functools.partial(mbw.gemv_int4_awq_g128, repacked=True), (c, s, z, x), y
        return mbw.gemv_int4_awq_g128, (c, s, z, x), y
    if fmt == wl.FMT_INT8_PC:
        q = inputs_gpu.int8_codes(seed, mi, N, K, device)
        s = inputs_gpu.f32_row_scales(seed, mi, N, device)
        return mbw.gemv_int8_pc, (q, s, x), y
    if fmt == wl.FMT_BF16:
        return mbw.gemv_bf16, (inputs_gpu.bf16_weights(seed, mi, N, K, device), x), y
    raise ValueError(fmt)


def torch_empty(shape, device):
    import torch

    return torch.empty(shape, dtype=torch.bfloat16, device=device)


def device_weights(fmt, seed, mi, N, K, device):
    """(weights, scales) of matrix `mi`, generated on the device (scales None for BF16)."""
    from memory_bound_weight_gb300 import inputs_gpu

    if fmt == wl.FMT_INT4_G64:
        return inputs_gpu.int4_codes(seed, mi, N, K, device), inputs_gpu.f16_group_scales(seed, mi, N, K // 64, device)
    if fmt == wl.FMT_INT8_PC:
        return inputs_gpu.int8_codes(seed, mi, N, K, device), inputs_gpu.f32_row_scales(seed, mi, N, device)
    if fmt == wl.FMT_BF16:
        return inputs_gpu.bf16_weights(seed, mi, N, K, device), None
    raise ValueError(fmt)


WORKLOAD_MATS = {
    "tinyllama_int4": (lambda: wl.tinyllama_step(fused=True), wl.FMT_INT4_G64),
    "tinyllama_int4_fusedops": (lambda: wl.tinyllama_step(fusedops=True), wl.FMT_INT4_G64),
    "tinyllama_int4_unfused": (lambda: wl.tinyllama_step(), wl.FMT_INT4_G64),
    "qwen_bf16": (wl.qwen25_7b_step, wl.FMT_BF16),
    "qwen_bf16_fused": (lambda: wl.qwen25_7b_step(fused=True), wl.FMT_BF16),
    "qwen_awq": (wl.qwen25_7b_step, wl.FMT_INT4_AWQ_G128),
    "qwen_awq_repacked": (wl.qwen25_7b_step, wl.FMT_INT4_AWQ_G128),
    "qwen_awq_repacked_fused": (lambda: wl.qwen25_7b_step(fused=True), wl.FMT_INT4_AWQ_G128),
    "qwen_awq_fusedops": (lambda: wl.qwen25_7b_step(fusedops=True), wl.FMT_INT4_AWQ_G128),
    "qwen3_int8": (wl.qwen3_4b_step, wl.FMT_INT8_PC),
    "bf16_2048": (lambda: [wl.Mat(f"copy{i}", 2048, 2048) for i in range(64)], wl.FMT_BF16),
}


def make_step(workload, seed, device, M=1):
    if workload in ("tinyllama_int4", "tinyllama_int4_unfused", "tinyllama_int4_fusedops"):
        return Step("TinyLlama-1.1B-shaped INT4 g64 decode step, batch 1", wl.FMT_INT4_G64,
                    WORKLOAD_MATS[workload][0](), seed, device)
    if workload == "qwen_bf16":
        return Step("Qwen2.5-7B-shaped BF16 decode step, batch 1", wl.FMT_BF16, wl.qwen25_7b_step(), seed, device)
    if workload == "qwen_bf16_fused":
        return Step("Qwen2.5-7B-shaped BF16 decode step, batch 1, gate and up fused", wl.FMT_BF16,
                    wl.qwen25_7b_step(fused=True), seed, device)
    if workload in ("qwen_awq", "qwen_awq_repacked", "qwen_awq_repacked_fused", "qwen_awq_fusedops"):
        rp = workload != "qwen_awq"
        fo = workload == "qwen_awq_fusedops"
        fu = workload == "qwen_awq_repacked_fused"
        return Step(f"Qwen2.5-7B-shaped AWQ-style INT4 decode step, batch {M}" + (", repacked codes" if rp else "")
                    + (", small ops fused" if fo else "") + (", gate and up fused" if fu else ""),
                    wl.FMT_INT4_AWQ_G128, wl.qwen25_7b_step(fusedops=fo, fused=fu), seed, device, M, repacked=rp)
    if workload == "qwen3_int8":
        return Step(f"Qwen3-4B-shaped symmetric INT8 per-channel decode step, batch {M}", wl.FMT_INT8_PC,
                    wl.qwen3_4b_step(), seed, device, M)
    if workload == "bf16_2048":
        # 2048x2048 BF16 GEMV; 64 distinct copies (537 MB) so that each is evicted before it recurs
        mats = [wl.Mat(f"copy{i}", 2048, 2048) for i in range(64)]
        return Step("BF16 GEMV 2048x2048, batch 1 (64 rotating copies)", wl.FMT_BF16, mats, seed, device)
    raise ValueError(workload)


# ------------------------------------------------------------- cpu oracle ----
_HOST_CACHE = {}  # host copies of the step's matrices, reused across oracle runs
def cpu_baseline(workload, budget_s=10.0, M=1):
    """The fp64 oracle on this host's cores over a bounded sample of the step
    (whole passes over the step's matrices until about `budget_s` of oracle time)."""
    import numpy as np

    import oracle
    from memory_bound_weight_gb300 import inputs as gen

    o = oracle.load()
    if workload == "bf16_2048":
        mats, fmt = [wl.Mat("copy0", 2048, 2048)] * 64, wl.FMT_BF16
    else:
        mk, fmt = WORKLOAD_MATS[workload]
        mats = mk()
    what = f"the step's {len(mats)} matrices"
    if wl.step_weight_bytes(mats, fmt) > 2e9:
        # a multi-GB step: the oracle cycles over the first layer's matrices (the
        # same GEMVs, byte for byte; generating every matrix on the host would
        # take minutes and hold the whole step in host memory)
        nl = sum(1 for m in mats if m.name.startswith("L0."))
        what = f"the first layer's {nl} matrices of the {len(mats)}-matrix step"
        mats = mats[:nl]

    def host_weights(mi, m):
        if fmt == wl.FMT_INT4_G64:
            return gen.int4_codes(0, mi, m.N, m.K), gen.f16_group_scales(0, mi, m.N, m.K // 64), None
        if fmt == wl.FMT_INT8_PC:
            return gen.int8_codes(0, mi, m.N, m.K), gen.f32_row_scales(0, mi, m.N), None
        if fmt == wl.FMT_INT4_AWQ_G128:
            G = m.K // 128
            return (gen.int4_codes(0, mi, m.N, m.K), gen.f16_group_scales(0, mi, m.N, G),
                    gen.u4_zero_points(0, mi, m.N, G))
        return gen.bf16_weights(0, mi, m.N, m.K), None, None

    def gemm(w, X):
        A, B, Z = w
        if fmt == wl.FMT_INT4_G64:
            return o.gemm_int4_g64(A, B, X)[0]
        if fmt == wl.FMT_INT8_PC:
            return o.gemm_int8_pc(A, B, X)[0]
        if fmt == wl.FMT_INT4_AWQ_G128:
            return o.gemm_int4_awq_g128(A, B, Z, X)[0]
        return o.gemm_bf16(A, X)[0]
    done_bytes = 0
    spent = 0.0
    n = 0
    order = [(mi, m) for _ in range(1000) for mi, m in enumerate(mats)]
    cache = _HOST_CACHE.setdefault((workload, M), {})
    cacheable = wl.step_weight_bytes(mats, fmt) < 2e9
    for mi, m in order:
        if mi in cache:
            X, w, wu, G, R = cache[mi]
        else:
            X = gen.bf16_activations(0, mi, M, m.K)
            w = host_weights(mi, m)
            wu = host_weights(50000 + mi, m) if m.fuse & wl.FUSE_GLU else None
            G = gen.bf16_normal(0, gen.stream_id(60000 + mi, gen.KIND_X), m.K, gen.X_SIGMA) \
                if m.fuse & wl.FUSE_NORM else None
            R = gen.bf16_normal(0, gen.stream_id(70000 + mi, gen.KIND_X), M * m.N, gen.X_SIGMA).reshape(M, m.N) \
                if m.fuse & wl.FUSE_RESIDUAL else None
            if cacheable:
                cache[mi] = (X, w, wu, G, R)
        t = time.perf_counter()
        Xn = o.rmsnorm_bf16(X, G, 1e-6) if G is not None else X
        Y = gemm(w, Xn)
        if wu is not None:
            Y = o.swiglu(Y, gemm(wu, Xn))
        if R is not None:
            Y = o.add_residual(Y, R)
        spent += time.perf_counter() - t
        done_bytes += wl.call_bytes(fmt, M, m)
        n += 1
        if spent >= budget_s:
            break
    return {"value": done_bytes / spent / 1e9, "unit": "GB/s", "cores": o.num_threads(), "kind": "oracle",
            "sample": f"{n} matrix GEMVs ({n / len(mats):.2f} passes over {what}, "
                      f"{done_bytes / 1e9:.3f} GB), fp64 C oracle, OpenMP over rows, {spent:.1f} s"}


def cpu_baseline_single_thread(workload, M=1, budget_s=3.0):
    """The same oracle sample on one host thread (the row loop unparallelised)."""
    import oracle

    o = oracle.load()
    n = o.num_threads()
    o.set_num_threads(1)
    try:
        r = cpu_baseline(workload, budget_s=budget_s, M=M)
    finally:
        o.set_num_threads(n)
    return {"value": r["value"], "unit": r["unit"], "cores": 1, "sample": r["sample"].replace("OpenMP over rows",
                                                                                             "one thread")}


def run_reference(args, rank, ws):
    """--impl reference: the oracle, as it stands, on the host cores."""
    if rank != 0:
        return
    per_step = args.ref_budget if args.ref_budget else max(0.5, 20.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        cpu_baseline(args.workload, budget_s=per_step, M=args.batch)
    t0 = time.perf_counter()
    vals = []
    for _ in range(args.steps):
        vals.append(cpu_baseline(args.workload, budget_s=per_step, M=args.batch))
    elapsed = time.perf_counter() - t0
    v = statistics.median(r["value"] for r in vals)
    cb = dict(vals[0])
    cb["value"] = v
    cb["sample"] = f"each step: {per_step:.1f} s of oracle time over the step's matrices in order; first step: " \
                   + vals[0]["sample"]
    mk, fmt = WORKLOAD_MATS[args.workload]
    step_bytes = wl.step_bytes_alg(mk(), fmt, args.batch)
    line = {"impl": "reference", "metric": metric_name(args.workload), "value": v, "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_bytes / (v * 1e9) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_desc(args.workload, args.batch)}, "cpu_baseline": cb,
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def metric_name(workload):
    return "decode GEMV achieved HBM GB/s (% of GB300 peak); weight-stream ms/token"


def workload_desc(workload, batch=1):
    return {"tinyllama_int4": "TinyLlama-1.1B-shaped INT4 group-64 decode step, batch 1, q/k/v and gate/up fused "
                              "(89 GEMVs)",
            "tinyllama_int4_unfused": "TinyLlama-1.1B-shaped INT4 group-64 decode step, batch 1 (155 GEMVs)",
            "tinyllama_int4_fusedops": "TinyLlama-1.1B-shaped INT4 group-64 decode step, batch 1, q/k/v and gate/up "
                                       "fused, with the layer's small ops folded into the GEMVs: RMSNorm prologues "
                                       "(q/k/v, gate/up, head), SwiGLU epilogue (gate/up), residual-add epilogues (o, "
                                       "down) (89 GEMVs)",
            "qwen_bf16": "Qwen2.5-7B-shaped BF16 decode step, batch 1 (141 GEMVs)",
            "qwen_bf16_fused": "Qwen2.5-7B-shaped BF16 decode step, batch 1, gate and up stored as one [Wgate; Wup] "
                               "matrix and streamed by one GEMV per layer (113 GEMVs, the same weights)",
            "qwen_awq": f"Qwen2.5-7B-shaped AWQ-style INT4 decode step (group 128, fp16 scale, uint4 zero point, LM head "
                        f"included), batch {batch} (141 GEMMs)",
            "qwen_awq_repacked": f"Qwen2.5-7B-shaped AWQ-style INT4 decode step (group 128, fp16 scale, uint4 zero "
                                 f"point, LM head included), codes reordered at load time (mbw_repack_int4), batch "
                                 f"{batch} (141 GEMMs)",
            "qwen_awq_repacked_fused": f"Qwen2.5-7B-shaped AWQ-style INT4 decode step (group 128, fp16 scale, uint4 "
                                       f"zero point, LM head included), codes reordered at load time, gate and up "
                                       f"stored as one [Wgate; Wup] matrix, batch {batch} (113 GEMMs, the same weights)",
            "qwen_awq_fusedops": f"Qwen2.5-7B-shaped AWQ-style INT4 decode step (group 128, fp16 scale, uint4 zero "
                                 f"point), codes reordered at load time, with the layer's small ops folded into the "
                                 f"GEMVs: RMSNorm prologues (q/k/v, gate/up, head), SwiGLU epilogue (gate/up), "
                                 f"residual-add epilogues (o, down), batch {batch} (113 GEMVs)",
            "qwen3_int8": f"Qwen3-4B-shaped symmetric INT8 decode step (one fp32 scale per output channel, every "
                          f"linear layer and the LM head, q/k/v and gate/up fused), batch {batch} (145 GEMVs)",
            "bf16_2048": "BF16 GEMV 2048x2048, batch 1, 64 rotating copies"}[workload]


# ------------------------------------------------------- other configs ----
class CallKind:
    """What time_per_shape needs of a step (format, op, batch, code layout),
    for shapes timed without a resident step."""

    def __init__(self, fmt, M=1, repacked=False):
        import memory_bound_weight_gb300 as mbw

        self.fmt, self.M, self.repacked = fmt, M, repacked
        self.op = op_of_fmt(fmt) | (mbw.REPACKED if repacked else 0)

    def shapes(self):
        return []


def hbm_roofline(nbytes, us, peak):
    """HBM roofline fields of one launch: algorithmic bytes / its time."""
    a = nbytes / (us * 1e-6) / 1e9
    return {"bound": "hbm", "achieved": a, "peak": peak, "unit": "GB/s", "frac": a / peak,
            "bytes_alg_per_launch": nbytes, "us_per_launch": us}


def per_matrix_figures(fmt, shapes, device, cold_iters=100):
    """Steady state (PDL chain over copies >= 4x L2) and cold (L2 flushed)
    time of each shape on its autotuned plan, with its roofline."""
    peak, _ = hbm_peak()
    out = time_per_shape(CallKind(fmt), device, shapes=shapes, plans=None, cold_iters=cold_iters)
    for (fz, N, K) in shapes:
        r = out[skey((fz, N, K))]
        r["roofline"] = hbm_roofline(wl.call_bytes(fmt, 1, wl.Mat("", N, K, fz)), r["us"], peak)
    return out


def step_figure(workload, M, device, tune="shape", steps=20):
    """One decode step of `workload` at batch M: plans tuned per shape (or on
    the whole step), one CUDA graph per step, device time of `steps` replays;
    the dominant kernel's roofline as in the headline line."""
    import torch

    import memory_bound_weight_gb300 as mbw

    step = make_step(workload, seed=0, device=device, M=M)
    for fz, N, K in step.shapes():
        mbw.autotune(step.op | fz, M, N, K)
    if tune == "step":
        from memory_bound_weight_gb300.tune import tune_sequence

        tune_sequence(step.run, [(step.op | fz, M, N, K) for fz, N, K in step.shapes()])
    plans = {skey(sh): mbw.plan_describe(step.op | sh[0], M, sh[1], sh[2]) for sh in step.shapes()}
    step_plans = {sh: mbw.plan_index(step.op | sh[0], M, sh[1], sh[2]) for sh in step.shapes()}
    step.run()
    torch.cuda.synchronize()
    cap = torch.cuda.Stream(device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        step.run()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    stream = torch.cuda.current_stream(device)
    e0.record(stream)
    for _ in range(steps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    peak, peak_src = hbm_peak()
    gbs = step.bytes_alg / (ms * 1e-3) / 1e9
    shape_times = time_per_shape(step, device, shapes=step.shapes(), plans=step_plans)
    counts = {}
    for m in step.mats:
        counts[(m.fuse, m.N, m.K)] = counts.get((m.fuse, m.N, m.K), 0) + 1
    dominant = max(step.shapes(), key=lambda sh: counts[sh] * shape_times[skey(sh)]["us"])
    roof = roofline_fields(step, ms, gbs, peak, peak_src, None, plans, len(step.mats), dominant, counts,
                           shape_times)
    out = {"workload": workload_desc(workload, M), "ms_per_step": ms, "GB/s": gbs, "frac_of_peak": gbs / peak,
           "bytes_alg_per_step": step.bytes_alg, "steps": steps, "tune": tune, "plans": plans, "roofline": roof,
           "step_shapes": shape_times}
    del g, step
    torch.cuda.empty_cache()
    return out


def skinny_figures(device, Ms=wl.SKINNY_M, reps=7):
    """gemm_skinny_bf16 over the Qwen2.5-7B MLP shapes at each batch M, on the
    autotuned plan: a CUDA graph of at least 40 calls over distinct copies of
    W >= 4x L2 taken in turn, median of `reps` replays; HBM and tensor
    rooflines, the longer the bound."""
    import torch

    import memory_bound_weight_gb300 as mbw
    from memory_bound_weight_gb300 import inputs_gpu

    peak, _ = hbm_peak()
    tc, tc_src = tensor_peak()
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    op = mbw.OP_GEMM_SKINNY_BF16
    out = {}
    for m in wl.SKINNY_SHAPES:
        N, K = m.N, m.K
        row = {}
        for M in Ms:
            b = wl.bytes_alg(wl.FMT_BF16, M, N, K)
            fl = wl.flops(M, N, K)
            copies = int(max(4, -(-4 * l2 // b)))
            Ws = [inputs_gpu.bf16_weights(0, 2000 + i, N, K, device) for i in range(copies)]
            X = inputs_gpu.bf16_activations(0, 7, M, K, device)
            Ys = [torch.empty((M, N), dtype=torch.bfloat16, device=device) for _ in range(copies)]
            mbw.autotune(op, M, N, K)
            for i in range(copies):
                mbw.gemm_skinny_bf16(X, Ws[i], out=Ys[i])
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            launches = max(copies, 40)  # the copies in turn
            with torch.cuda.graph(g, stream=torch.cuda.Stream(device)):
                for i in range(launches):
                    mbw.gemm_skinny_bf16(X, Ws[i % copies], out=Ys[i % copies])
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            ts = []
            for _ in range(reps):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record()
                g.replay()
                e1.record()
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1) / launches)
            us = statistics.median(ts) * 1e3
            r = hbm_roofline(b, us, peak)
            tflops = fl / (us * 1e-6) / 1e12
            r.update({"hbm_frac": r["frac"], "tensor_frac": tflops / tc, "tensor_peak": tc,
                      "tensor_peak_source": tc_src})
            if fl / (tc * 1e12) > b / (peak * 1e9):
                r.update({"bound": "tensor", "achieved": tflops, "peak": tc, "unit": "TFLOP/s", "frac": tflops / tc})
            row[f"M={M}"] = {"us": us, "GB/s": b / (us * 1e-6) / 1e9, "frac_of_peak": b / (us * 1e-6) / 1e9 / peak,
                             "TFLOP/s": tflops, "copies": copies, "plan": mbw.plan_describe(op, M, N, K),
                             "roofline": r}
            del Ws, Ys, g
            torch.cuda.empty_cache()
        out[f"{N}x{K}"] = row
    return out


def extra_configs(device, main_workload, tune="shape"):
    """The other configurations the metric is quoted on, after the headline
    step (N = 1 only): BF16 GEMV 2048x2048; the four TinyLlama-shaped INT4
    group-64 matrices and the TinyLlama INT4 step; the Qwen2.5-7B BF16 step
    with gate and up stored as one matrix; the skinny BF16 GEMM sweep; the
    AWQ-style INT4 step at M = 1, 16, 64 with repacked codes, and at M = 1 with
    gate and up stored as one matrix."""
    t0 = time.time()
    out = {}
    out["bf16_gemv_2048x2048"] = per_matrix_figures(wl.FMT_BF16, [(0, 2048, 2048)], device)
    out["int4_g64_tinyllama_matrices"] = per_matrix_figures(
        wl.FMT_INT4_G64, [(0, m.N, m.K) for m in wl.TINYLLAMA_TABLE_SHAPES], device)
    if main_workload != "tinyllama_int4":
        out["int4_g64_tinyllama_step"] = step_figure("tinyllama_int4", 1, device, tune)
    if main_workload != "qwen_bf16":
        out["bf16_qwen_step"] = step_figure("qwen_bf16", 1, device, tune)
    if main_workload != "qwen_bf16_fused":
        # the same weights with gate and up stored as one matrix: 113 GEMVs instead of 141
        out["bf16_qwen_step_gate_up_fused"] = step_figure("qwen_bf16_fused", 1, device, tune)
    out["skinny_bf16_qwen_mlp"] = skinny_figures(device)
    out["awq_qwen_step_repacked"] = {f"M={M}": step_figure("qwen_awq_repacked", M, device, tune) for M in wl.AWQ_M}
    # batch 1 with gate and up stored as one matrix (113 GEMVs instead of 141, the same weights)
    out["awq_qwen_step_repacked_gate_up_fused"] = {"M=1": step_figure("qwen_awq_repacked_fused", 1, device, tune)}
    out["seconds"] = time.time() - t0
    return out


# ------------------------------------------------------------------- main ----
def main():
    args = parse_args()
    if args.impl == "reference":
        rank, ws, _ = dist_setup("gloo")
        run_reference(args, rank, ws)
        if ws > 1:
            barrier(ws)
        return

    import torch

    rank, ws, local = dist_setup("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)

    from memory_bound_weight_gb300 import build as mbuild

    if rank == 0 and not os.path.exists(os.path.join(ROOT, "memory_bound_weight_gb300", "libmbw.so")):
        mbuild.build()
    barrier(ws)
    import memory_bound_weight_gb300 as mbw

    step = make_step(args.workload, seed=0, device=device, M=args.batch)
    Mb = step.M
    if args.plans_from:
        with open(args.plans_from) as f:
            saved = json.load(f)
        for fz, N, K in step.shapes():
            mbw.plan_select(step.op | fz, Mb, N, K, int(saved[skey((fz, N, K))]))
    else:
        for fz, N, K in step.shapes():
            mbw.autotune(step.op | fz, Mb, N, K)
        if args.tune == "step":
            from memory_bound_weight_gb300.tune import tune_sequence

            res = tune_sequence(step.run, [(step.op | fz, Mb, N, K) for fz, N, K in step.shapes()],
                                log=(lambda m: print("[tune]", m, file=sys.stderr)))
            print(f"[tune] step {res['_ms'][0]:.4f} -> {res['_ms'][1]:.4f} ms", file=sys.stderr)
    if args.plans_out and rank == 0:
        with open(args.plans_out, "w") as f:
            json.dump({skey(sh): mbw.plan_index(step.op | sh[0], Mb, sh[1], sh[2]) for sh in step.shapes()}, f)
    plans = {skey(sh): mbw.plan_describe(step.op | sh[0], Mb, sh[1], sh[2]) for sh in step.shapes()}
    step.run()
    torch.cuda.synchronize()

    # one CUDA graph per step: the C-ABI calls captured in order
    cap = torch.cuda.Stream(device)
    g = torch.cuda.CUDAGraph()
    n0 = mbw.launch_count()
    with torch.cuda.graph(g, stream=cap):
        step.run()
    launches_per_step = mbw.launch_count() - n0

    stream = torch.cuda.current_stream(device)
    for _ in range(max(3, args.warmup)):
        g.replay()
    torch.cuda.synchronize()
    barrier(ws)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(ws)
    if args.profile_range:
        torch.cuda.profiler.start()
    t0 = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if args.profile_range:
        torch.cuda.profiler.stop()
    barrier(ws)
    sampler.stop()
    ms = e0.elapsed_time(e1)
    ms = max_over_ranks(ms, ws, device)
    ms_step = ms / args.steps
    gbs_rank = step.bytes_alg / (ms_step * 1e-3) / 1e9
    value = gbs_rank * ws

    # end to end: per step, the x vectors go host->device from pinned memory,
    # the step runs, the y vectors come back device->host.
    e2e = None
    if not args.no_e2e:
        xh = torch.empty_like(step.x, device="cpu").pin_memory()
        xh.copy_(step.x)
        yh = torch.empty_like(step.y, device="cpu").pin_memory()
        ke = max(1, min(args.steps, 2000))
        for _ in range(max(3, args.warmup // 10)):
            step.x.copy_(xh, non_blocking=True)
            g.replay()
            yh.copy_(step.y, non_blocking=True)
        torch.cuda.synchronize()
        barrier(ws)
        e0.record(stream)
        for _ in range(ke):
            step.x.copy_(xh, non_blocking=True)
            g.replay()
            yh.copy_(step.y, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        ems = max_over_ranks(e0.elapsed_time(e1), ws, device) / ke
        e2e = {"value": step.bytes_alg / (ems * 1e-3) / 1e9 * ws, "unit": "GB/s",
               "h2d_bytes_per_step": step.h2d_bytes, "d2h_bytes_per_step": step.d2h_bytes,
               "ms_per_step": ems, "steps": ke}

    # per-shape steady state on the step's own plans: the dominant kernel is
    # the shape with the largest share of the step (launches x time per launch)
    step_plans = {sh: mbw.plan_index(step.op | sh[0], Mb, sh[1], sh[2]) for sh in step.shapes()}
    shape_times = {}
    if rank == 0 and not args.no_shape_timing:
        shape_times = time_per_shape(step, device, shapes=step.shapes(), plans=step_plans)
    per_matrix = None
    if args.per_matrix and rank == 0:
        # steady state and cold (L2 flushed before every call), step's own plans
        # for its shapes, autotuned plans for the named extra shapes
        per_matrix = time_per_shape(step, device, plans=step_plans, cold_iters=100,
                                    shapes=list(step_plans) + [sh for sh in named_shapes(step.fmt)
                                                               if sh not in step_plans])

    peak, peak_src = hbm_peak()
    counts = {}
    for m in step.mats:
        counts[(m.fuse, m.N, m.K)] = counts.get((m.fuse, m.N, m.K), 0) + 1
    dominant = None
    if shape_times:
        dominant = max(step.shapes(), key=lambda sh: counts[sh] * shape_times[skey(sh)]["us"])
    family = plans[skey(dominant)].split(" ")[0] if dominant else "lat"
    sha = kernel_source_sha(family)
    fmt_tok = re.search(r"fmt=(\S+)", plans[skey(dominant)]) if dominant else None
    traffic = TRAFFIC.get((sha, skey(dominant), fmt_tok.group(1))) if fmt_tok else None
    clocks = sampler.summary(t0, t1)
    if rank != 0:
        return
    cb = None
    if ws == 1 and not args.no_cpu_baseline:
        cb = cpu_baseline(args.workload, M=step.M)
        cb["single_thread"] = cpu_baseline_single_thread(args.workload, M=step.M)
    line = {
        "metric": metric_name(args.workload),
        "value": value,
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": workload_desc(args.workload, step.M), "matrices": len(step.mats),
                   "bytes_alg_per_step": step.bytes_alg, "batch": step.M, "parallelism": f"replicas{ws}",
                   "l2": "inputs larger than L2: each step streams %.3f GB of distinct weights" % (step.bytes_alg / 1e9),
                   "plans": plans},
        "weight_stream_ms_per_token": ms_step,
        "frac_of_peak": gbs_rank / peak,
        "roofline": roofline_fields(step, ms_step, gbs_rank, peak, peak_src, traffic, plans, launches_per_step,
                                    dominant, counts, shape_times),
        "cpu_baseline": cb,
        "e2e": e2e,
        "clocks": clocks,
        "gpu_launches": launches_per_step * args.steps,
        "launches_per_step": launches_per_step,
        "kernel_source_sha": sha,
        "step_shapes": shape_times,
    }
    if per_matrix:
        line["per_matrix"] = per_matrix
    if ws == 1 and not args.no_extras:
        # the other configurations, after the headline step's memory is released
        del g, step
        torch.cuda.empty_cache()
        line["configs"] = extra_configs(device, args.workload, args.extras_tune)
    print(json.dumps(line), flush=True)


def roofline_fields(step, ms_step, gbs, peak, peak_src, traffic, plans, launches_per_step, dominant, counts,
                    shape_times):
    """Roofline of the step's dominant kernel (the shape with the largest share
    of the step: launches x steady-state time per launch). achieved = its
    algorithmic bytes per launch / its average launch duration, timed with
    CUDA events on the launching stream over a PDL-chained graph of its own
    launches on the plan the step uses. With a batch, the tensor-core roofline
    too, and the one whose time is longer is the bound."""
    if dominant is None:  # not timed (other ranks)
        return {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                "traffic": traffic, "peak_source": peak_src, "kernel": "step average"}
    key = skey(dominant)
    st = shape_times[key]
    tot = sum(counts[sh] * shape_times[skey(sh)]["us"] for sh in counts)
    M = step.M
    dm = wl.Mat(key, dominant[1], dominant[2], dominant[0])
    kb = wl.call_bytes(step.fmt, M, dm)
    kfl = wl.call_flops(M, dm)
    achieved = kb / (st["us"] * 1e-6) / 1e9
    r = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
         "traffic": traffic, "peak_source": peak_src,
         "kernel": f"{plans[key]} on the {key} matrices ({counts[dominant]} per step)",
         "frac_of_nominal_hbm": achieved / NOMINAL_HBM_GBS, "nominal_hbm_gbs": NOMINAL_HBM_GBS,
         "bytes_alg_per_launch": kb, "us_per_launch": st["us"],
         "share_of_step": counts[dominant] * st["us"] / tot,
         "note": "per-launch time of the dominant kernel in a PDL-chained graph of %d of its own launches over "
                 "%d distinct weight copies >= 4x L2 taken in turn (same plan as in the step); the step-level "
                 "figure is value / "
                 "frac_of_peak (every launch of the step is one of this library's kernels, %d per step)"
                 % (st["launches"], st["copies"], launches_per_step)}
    if M > 1:
        tc, tc_src = tensor_peak()
        tflops = kfl / (st["us"] * 1e-6) / 1e12
        r["hbm_frac"] = achieved / peak
        r["tensor_frac"] = tflops / tc
        r["tensor_peak"] = tc
        r["tensor_peak_source"] = tc_src
        if kfl / (tc * 1e12) > kb / (peak * 1e9):
            r.update({"bound": "tensor", "achieved": tflops, "peak": tc, "unit": "TFLOP/s", "frac": tflops / tc,
                      "peak_source": tc_src})
    return r


def named_shapes(fmt):
    """The shapes the per-matrix figures are quoted on, besides the step's own:
    tinyinfer's four TinyLlama INT4 matrices, and the 2048x2048 BF16 GEMV."""
    if fmt == wl.FMT_INT4_G64:
        return [(0, m.N, m.K) for m in wl.TINYLLAMA_TABLE_SHAPES]
    if fmt == wl.FMT_INT4_AWQ_G128:
        return [(0, m.N, m.K) for m in wl.SKINNY_SHAPES]
    if fmt == wl.FMT_INT8_PC:
        return []
    return [(0, 2048, 2048)]


def time_per_shape(step, device, reps=5, shapes=None, plans=None, cold_iters=0):
    """Steady-state time per matrix of each shape: a CUDA graph of back-to-back
    launches (programmatic dependent launch, as in the step) over distinct
    copies of the matrix totalling at least 4x the L2, taken in turn for at
    least 40 launches, so every launch reads its weights from HBM and the
    graph's own start weighs little; per-matrix time = graph time / launches.

    With cold_iters > 0, also the cold figure: that many single calls, each
    after a write of twice the L2 that evicts the matrix, each timed with CUDA
    events on the calling stream (launch latency included, nothing overlaps);
    median and interquartile range."""
    import torch

    import memory_bound_weight_gb300 as mbw
    from memory_bound_weight_gb300 import inputs_gpu

    out = {}
    peak, _ = hbm_peak()
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    shapes = sorted(set(step.shapes()) | set(named_shapes(step.fmt))) if shapes is None else list(shapes)
    M = step.M
    for fz, N, K in shapes:
        b = wl.call_bytes(step.fmt, M, wl.Mat("", N, K, fz))
        copies = int(min(512, max(8, -(-4 * l2 // b))))
        x = torch.empty((copies, M, K), dtype=torch.bfloat16, device=device)
        y = torch.empty((copies, M, N), dtype=torch.bfloat16, device=device)
        inputs_gpu.bf16_normal_(x.view(-1), 0, 7, 1.0)
        calls = []
        for i in range(copies):
            xi, yi = (x[i, 0], y[i, 0]) if M == 1 else (x[i], y[i])
            calls.append(device_call(step.fmt, 0, 1000 + i, N, K, xi, yi, device, fz, M, step.repacked))
        if plans is not None and (fz, N, K) in plans:
            mbw.plan_select(step.op | fz, M, N, K, plans[(fz, N, K)])
        else:
            mbw.autotune(step.op | fz, M, N, K)
        for fn, a, o in calls:
            fn(*a, out=o)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(device)
        launches = max(copies, 40)
        with torch.cuda.graph(g, stream=s):
            for i in range(launches):
                fn, a, o = calls[i % copies]
                fn(*a, out=o)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) / launches)
        us = statistics.median(ts) * 1e3
        out[skey((fz, N, K))] = {"us": us, "GB/s": b / (us * 1e-6) / 1e9, "frac": b / (us * 1e-6) / 1e9 / peak,
                                 "TFLOP/s": wl.call_flops(M, wl.Mat("", N, K, fz)) / (us * 1e-6) / 1e12,
                                 "copies": copies, "launches": launches,
                                 "plan": mbw.plan_describe(step.op | fz, M, N, K)}
        if cold_iters > 0:
            out[skey((fz, N, K))].update(time_cold(calls[0], b, peak, l2, device, cold_iters))
        del calls, g
        torch.cuda.empty_cache()
    return out


def time_cold(call, nbytes, peak, l2, device, iters, warmup=3):
    """Cold time of one call: before each timed call, 2x the L2 is written so
    that the call reads its matrix from HBM."""
    import torch

    fn, a, o = call
    flush = torch.empty((2 * l2) // 4 + 1, dtype=torch.int32, device=device)
    ev = []
    for it in range(warmup + iters):
        flush.fill_(it)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        fn(*a, out=o)
        e1.record()
        if it >= warmup:
            ev.append((e0, e1))
    torch.cuda.synchronize()
    ts = sorted(e0.elapsed_time(e1) * 1e3 for e0, e1 in ev)
    q = statistics.quantiles(ts, n=4)
    med = statistics.median(ts)
    del flush
    return {"cold_us": med, "cold_iqr_us": [q[0], q[2]], "cold_frac": nbytes / (med * 1e-6) / 1e9 / peak,
            "cold_iters": iters}


if __name__ == "__main__":
    main()
