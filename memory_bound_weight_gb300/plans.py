"""Saved plans: the plan chosen for each call shape (op, M, N, K), written to
a JSON file so that a later process can skip tuning.

A plan is stored as its index among the shape's candidates together with its
one-line description. The file also records the identity the plans were
measured on: the GPU's name, SM count and compute capability, and a hash of
the library's sources. ``load_plans`` restores a file only onto the same
identity, and restores an entry only if the index still describes the same
plan (a changed candidate list makes an index mean something else). Anything
else is skipped, and the shape keeps its current plan.

This is host-side bookkeeping over the plan API of ``include/mbw.h``
(candidates, select, index, describe).
"""
from __future__ import annotations

import hashlib
import json
import os

from . import _binding as B

FORMAT = 1


def library_sources_sha() -> str:
    """Hash of the sources libmbw.so is built from (kernels, ABI, header)."""
    from . import build as mbuild

    h = hashlib.sha256()
    names = sorted(f for f in os.listdir(mbuild.CSRC) if f.endswith((".cu", ".cuh", ".h")))
    for name in names:
        h.update(name.encode())
        with open(os.path.join(mbuild.CSRC, name), "rb") as f:
            h.update(f.read())
    with open(os.path.join(mbuild.INCLUDE, "mbw.h"), "rb") as f:
        h.update(f.read())
    return h.hexdigest()[:16]


def identity() -> dict:
    """What a saved plan depends on besides its shape."""
    import torch

    p = torch.cuda.get_device_properties(torch.cuda.current_device())
    return {"gpu": p.name, "sms": int(p.multi_processor_count), "cc": f"{p.major}.{p.minor}",
            "library": library_sources_sha()}


def save_plans(path: str, shapes) -> int:
    """Write the current plan of every (op, M, N, K) in ``shapes`` to ``path``.
    Returns the number of plans written (shapes without a valid plan are left out)."""
    entries = []
    for op, M, N, K in shapes:
        idx = B.plan_index(op, M, N, K)
        if idx < 0:
            continue
        entries.append({"op": int(op), "M": int(M), "N": int(N), "K": int(K), "index": int(idx),
                        "plan": B.plan_describe(op, M, N, K)})
    doc = {"format": FORMAT, "identity": identity(), "plans": entries}
    tmp = path + ".tmp"
    with open(tmp, "w") as f:
        json.dump(doc, f, indent=1)
    os.replace(tmp, path)
    return len(entries)


def load_plans(path: str) -> tuple[int, list[str]]:
    """Select the saved plans of ``path`` in the library's plan cache.
    Returns (plans restored, reasons for everything skipped)."""
    try:
        with open(path) as f:
            doc = json.load(f)
    except (OSError, ValueError) as e:
        return 0, [f"unreadable plan file: {e}"]
    if not isinstance(doc, dict) or doc.get("format") != FORMAT or not isinstance(doc.get("plans"), list):
        return 0, ["not a plan file of this format"]
    here = identity()
    saved = doc.get("identity")
    if saved != here:
        return 0, [f"identity differs: saved {saved}, here {here}"]
    restored, skipped = 0, []
    for e in doc["plans"]:
        try:
            op, M, N, K, idx, desc = (int(e["op"]), int(e["M"]), int(e["N"]), int(e["K"]), int(e["index"]),
                                      str(e["plan"]))
        except (KeyError, TypeError, ValueError):
            skipped.append(f"malformed entry {e!r}")
            continue
        shape = (op, M, N, K)
        if not 0 <= idx < B.plan_candidates(op, M, N, K):
            skipped.append(f"{shape}: index {idx} out of range")
            continue
        before = B.plan_index(op, M, N, K)
        B.plan_select(op, M, N, K, idx)
        if B.plan_describe(op, M, N, K) != desc:
            if before >= 0:
                B.plan_select(op, M, N, K, before)
            skipped.append(f"{shape}: index {idx} is no longer the saved plan")
            continue
        restored += 1
    return restored, skipped
