"""Plan refinement on a whole call sequence (a decode step).

``mbw_autotune`` times each shape on its own, chained with itself. Inside a
decode step every GEMV is chained with different neighbours, and what makes a
small GEMV fast there is that the next launch fits on the SMs beside it and
streams its weights while this one finishes (programmatic dependent launch).
A plan that wins a chain of identical launches can lose that overlap in the
mixed chain. ``tune_sequence`` therefore starts from the per-shape plans and
does coordinate descent over each distinct shape's candidate plans, timing the
caller's whole sequence as a CUDA graph after every change, and keeps a change
only when the sequence gets faster.

The library API used is the plan API of ``include/mbw.h`` (candidates, select,
index); the kernels and their launches are the library's.
"""
from __future__ import annotations

import statistics

from . import _binding as B


def _time_graph(run_once, reps: int, warmup: int) -> float:
    import torch

    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run_once()
    for _ in range(warmup):
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
        ts.append(e0.elapsed_time(e1))
    del g
    return statistics.median(ts)


def tune_sequence(run_once, shapes, passes: int = 2, reps: int = 7, warmup: int = 2, min_gain: float = 0.003,
                  log=None) -> dict:
    """Refine the plans of ``shapes`` (distinct ``(op, M, N, K)`` tuples) for
    the sequence that ``run_once()`` enqueues on the current stream.

    Returns ``{(op, M, N, K): plan_index}`` with the selected plans (also left
    selected in the library's plan cache) and, under ``"_ms"``, the sequence
    time before and after."""
    start = _time_graph(run_once, reps, warmup)
    best = start
    chosen = {sh: B.plan_index(*sh) for sh in shapes}
    for p in range(passes):
        improved = False
        for sh in shapes:
            cur = chosen[sh]
            for i in range(B.plan_candidates(*sh)):
                if i == cur:
                    continue
                B.plan_select(*sh, i)
                t = _time_graph(run_once, reps, warmup)
                if t < best * (1.0 - min_gain):
                    if log:
                        log(f"pass {p} {sh}: {B.plan_describe(*sh)} {best:.4f} -> {t:.4f} ms")
                    best, cur, improved = t, i, True
            B.plan_select(*sh, cur)
            chosen[sh] = cur
        if not improved:
            break
    out = dict(chosen)
    out["_ms"] = (start, best)
    return out
