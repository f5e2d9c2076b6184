"""Per-question oracle checks of the stress workload, run in worker processes.

The stress workload (256 questions, prefill then 128 decode steps with early
stop) is checked against the oracle over its whole run.  Questions are
independent by construction (each has its own interval and its own slot), so
the oracle's prefill is evaluated on each question alone (the oracle's
packed = alone invariant is pinned in ``test_oracle.py``) and its decode is
chained step after step on a pool holding that question's slot only.  Each
worker receives the GPU's results for its questions and returns error
statistics; nothing here touches the GPU or imports the library.
"""
from __future__ import annotations

import numpy as np

import workloads as W
from oracle import kev_oracle as O


def _stats(got_bits: np.ndarray, ref: np.ndarray):
    got = W.to_float64(got_bits, "bf16")
    finite = bool(np.all(np.isfinite(got)))
    d = got - ref
    return {"finite": finite, "max": float(np.abs(d).max()) if d.size else 0.0,
            "d2": float(np.sum(d * d)), "r2": float(np.sum(ref * ref))}


def check_question(job: dict) -> dict:
    """Oracle prefill and the chained oracle decode of one question, compared with the GPU's.

    ``job`` holds the question's stored inputs (q/k/v rows, bf16 bits), its decode-step inputs
    for the steps it takes part in, the GPU's prefill output rows, the GPU's decode outputs of
    those steps (eager run and graph replay) and the GPU's final slot rows.
    """
    L, n_dec = job["L"], job["n_dec"]
    q, k, v = job["q"], job["k"], job["v"]
    res = {"i": job["i"]}
    # prefill of the question (the oracle's dense causal x isolation mask over one interval)
    ref = O.prefill(W.to_float64(q, "bf16"), W.to_float64(k, "bf16"), W.to_float64(v, "bf16"), [(0, L)])
    res["prefill"] = _stats(job["gpu_out"], ref)
    # its slot: the slot write, then every decode step it takes part in, appended in place
    h_kv, d = k.shape[1], k.shape[2]
    cap = L + n_dec
    pk = np.zeros((1, h_kv, cap, d), np.uint16)
    pv = np.zeros((1, h_kv, cap, d), np.uint16)
    pk, pv = O.slot_write(pk, pv, k, v, [(0, L)], [0])
    steps = []
    for t in range(n_dec):
        o, pk, pv = O.decode(job["qn"][t][None], job["kn"][t][None], job["vn"][t][None], pk, pv,
                             np.array([0]), np.array([L + t]), np.array([1], np.uint8), "bf16", inplace=True)
        steps.append({"eager": _stats(job["gpu_eager"][t], o[0]), "graph": _stats(job["gpu_graph"][t], o[0])})
    res["steps"] = steps
    res["pool_k_exact"] = bool(np.array_equal(pk[0], job["gpu_pool_k"]))
    res["pool_v_exact"] = bool(np.array_equal(pv[0], job["gpu_pool_v"]))
    return res
