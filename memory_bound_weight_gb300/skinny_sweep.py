"""Skinny BF16 GEMM Y = X . W^T over the Qwen2.5-7B MLP shapes at a sweep of
batch sizes, each on its autotuned plan; prints one JSON object.

    python -m memory_bound_weight_gb300.skinny_sweep [--M 1,8,16,32,64,128,256] [--reps 7]

Per shape and batch: a CUDA graph of back-to-back calls over distinct copies
of W totalling at least 4x the L2 (every call reads its weights from HBM),
median of `reps` replays, time per call. The fraction is (W + X bytes) / time
against the measured copy bandwidth. Inputs are the seeded synthetic tensors,
generated on the device.
"""
from __future__ import annotations

import argparse
import json
import statistics

SHAPES = ((18944, 3584), (3584, 18944))
HBM_GBS = 6778.3  # measured copy bandwidth of the GB300s


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--M", default="1,8,16,32,64,128,256")
    p.add_argument("--reps", type=int, default=7)
    a = p.parse_args()

    import torch

    import memory_bound_weight_gb300 as mbw
    from memory_bound_weight_gb300 import inputs_gpu

    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    out = {}
    for N, K in SHAPES:
        for M in (int(v) for v in a.M.split(",")):
            b = N * K * 2 + M * K * 2
            copies = max(4, -(-4 * l2 // b))
            Ws = [inputs_gpu.bf16_weights(0, 2000 + i, N, K) for i in range(copies)]
            X = inputs_gpu.bf16_activations(0, 7, M, K)
            Ys = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(copies)]
            mbw.autotune(mbw.OP_GEMM_SKINNY_BF16, M, N, K)
            for i in range(copies):
                mbw.gemm_skinny_bf16(X, Ws[i], out=Ys[i])
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            s = torch.cuda.Stream()
            with torch.cuda.graph(g, stream=s):
                for i in range(copies):
                    mbw.gemm_skinny_bf16(X, Ws[i], out=Ys[i])
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            ts = []
            for _ in range(a.reps):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record()
                g.replay()
                e1.record()
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1) / copies)
            us = statistics.median(ts) * 1e3
            out[f"{N}x{K} M={M}"] = {"us": round(us, 2), "frac_of_hbm": round(b / (us * 1e-6) / (HBM_GBS * 1e9), 3),
                                     "plan": mbw.plan_describe(mbw.OP_GEMM_SKINNY_BF16, M, N, K)}
            del Ws, Ys, g
            torch.cuda.empty_cache()
    print(json.dumps(out))


if __name__ == "__main__":
    main()
