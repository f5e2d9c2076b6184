"""Per-(question, kv group) oracle checks of a large prefill batch, run in worker processes.

Questions are independent by construction, and so are the kv groups of one question (a q-head
reads only its own kv head), so the oracle's prefill is evaluated on one question's rows and one
group's q-heads at a time (the oracle's packed = alone invariant is pinned in ``test_oracle.py``):
a [G, L, L] weight array per job instead of [H_q, T, T] for the batch.  Each job carries the GPU's
output rows for its heads and returns error statistics; nothing here touches the GPU or imports
the library.
"""
from __future__ import annotations

import numpy as np

import workloads as W
from oracle import kev_oracle as O


def check_group(job: dict) -> dict:
    """Oracle prefill of one (question, kv group) compared with the GPU's output rows."""
    L = job["L"]
    ref = O.prefill(W.to_float64(job["q"], "bf16"), W.to_float64(job["k"], "bf16"), W.to_float64(job["v"], "bf16"),
                    [(0, L)])
    got = W.to_float64(job["gpu_out"], "bf16")
    d = got - ref
    return {"i": job["i"], "g": job["g"], "finite": bool(np.all(np.isfinite(got))),
            "max": float(np.abs(d).max()) if d.size else 0.0, "d2": float(np.sum(d * d)),
            "r2": float(np.sum(ref * ref))}
