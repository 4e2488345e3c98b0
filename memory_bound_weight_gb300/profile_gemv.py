"""Run one GEMV shape a few times with a chosen plan (for profilers such as ncu).

    python -m memory_bound_weight_gb300.profile_gemv --op int4_g64 --N 32000 --K 2048 \
        [--M 1] [--plan tuned|default|<index>] [--reps 3] [--list-plans]

Inputs are the seeded synthetic tensors (generated on the device). The last
`--reps` launches are the ones to capture (e.g. ncu `-s <warm-up> -c <n>`).
"""
from __future__ import annotations

import argparse

OPS = {"bf16": 1, "int4_g64": 2, "int4_awq_g128": 3, "skinny_bf16": 4, "int8_pc": 5,
       "int4_awq_g128_repacked": 3 | 0x800}


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--op", default="int4_g64", choices=sorted(OPS))
    p.add_argument("--N", type=int, default=32000)
    p.add_argument("--K", type=int, default=2048)
    p.add_argument("--M", type=int, default=1)
    p.add_argument("--plan", default="tuned")
    p.add_argument("--reps", type=int, default=3)
    p.add_argument("--warmup", type=int, default=2)
    p.add_argument("--list-plans", action="store_true")
    a = p.parse_args()

    import torch

    import memory_bound_weight_gb300 as mbw
    from memory_bound_weight_gb300 import inputs_gpu as ig

    op = OPS[a.op]
    M, N, K = a.M, a.N, a.K
    if a.list_plans:
        for i in range(mbw.plan_candidates(op, M, N, K)):
            mbw.plan_select(op, M, N, K, i)
            print(i, mbw.plan_describe(op, M, N, K))
        return
    if a.plan == "tuned":
        mbw.autotune(op, M, N, K)
    elif a.plan != "default":
        mbw.plan_select(op, M, N, K, int(a.plan))
    print("plan:", mbw.plan_describe(op, M, N, K), flush=True)
    print("plan index:", mbw.plan_index(op, M, N, K), flush=True)

    X = ig.bf16_activations(0, 1, M, K)
    if op in (1, 4):
        W = ig.bf16_weights(0, 0, N, K)
        call = (lambda: mbw.gemv_bf16(W, X[0])) if op == 1 else (lambda: mbw.gemm_skinny_bf16(X, W))
    elif op == 2:
        c = ig.int4_codes(0, 0, N, K)
        s = ig.f16_group_scales(0, 0, N, K // 64)
        call = lambda: mbw.gemv_int4_g64(c, s, X[0])  # noqa: E731
    elif op == 5:
        q = ig.int8_codes(0, 0, N, K)
        s = ig.f32_row_scales(0, 0, N)
        call = lambda: mbw.gemv_int8_pc(q, s, X)  # noqa: E731
    else:
        c = ig.int4_codes(0, 0, N, K)
        s = ig.f16_group_scales(0, 0, N, K // 128)
        z = ig.u4_zero_points(0, 0, N, K // 128)
        rp = bool(op & mbw.REPACKED)
        if rp:
            mbw.repack_int4(c, out=c)  # the load-time reorder, once
        call = lambda: mbw.gemv_int4_awq_g128(c, s, z, X, repacked=rp)  # noqa: E731
    for _ in range(a.warmup + a.reps):
        call()
    torch.cuda.synchronize()
    print("done", flush=True)


if __name__ == "__main__":
    main()
