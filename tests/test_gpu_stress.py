"""GPU parity of the stress workload over its whole run.

256 questions with heavy-tailed lengths (T = 19,483) are prefilled into their slots, then
decoded for 128 steps with the seeded early-stop schedule: a question leaves after an EOS
draw or after its max_new_tokens steps (Kev pipeline article, gsyq.cn, §2.3: a finished
question takes no further part in attention).  The decode loop runs twice from the same
post-prefill state: eagerly (kev_decode_attn, then kev_decode_advance), and as one captured CUDA
graph replay of kev_decode_step (the advance folded into the step; the form the benchmark times),
with lens advanced on the device between steps.

Checked against the oracle: every row of every question's prefill output; every live
question's output at every step of both runs; the final slot contents bit for bit; rows of
dropped questions untouched at every step; the two runs bit for bit equal to each other.
The oracle is evaluated per question in spawned worker processes (``stress_oracle``).
"""
import multiprocessing as mp
import os

import numpy as np
import pytest
import torch

import packed_question_isolated_gb300 as kev
import stress_oracle
import workloads as W
from kev_harness import TOL_BF16_MAX, TOL_BF16_REL_L2, dev, host

pytestmark = pytest.mark.gpu

SENT_K, SENT_V = -7.0, -9.0


def _oracle_results(jobs):
    # spawned (not forked) workers: this process already holds a CUDA context
    ctx = mp.get_context("spawn")
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in saved:
        os.environ[k] = "1"
    try:
        with ctx.Pool(max(1, min(32, os.cpu_count() or 1))) as pool:
            # longest questions first, so the slowest jobs start early
            order = sorted(range(len(jobs)), key=lambda j: -(jobs[j]["L"] * (1 + jobs[j]["n_dec"])))
            res = pool.map(stress_oracle.check_question, [jobs[j] for j in order], chunksize=1)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    return sorted(res, key=lambda r: r["i"])


def test_stress_whole_run_eager_and_graph():
    s = W.stress()
    w = s.prefill
    N, steps = w.n_questions, s.n_steps
    shape = kev.make_shape(w.h_q, w.h_kv, w.d, "bf16")
    q, k, v = dev(w.q), dev(w.k), dev(w.v)
    iv = torch.from_numpy(np.ascontiguousarray(w.intervals)).cuda()
    sl = torch.from_numpy(np.ascontiguousarray(w.slot_ids)).cuda()
    pk = torch.full((w.n_slots, w.h_kv, w.cap, w.d), SENT_K, dtype=torch.bfloat16, device="cuda")
    pv = torch.full_like(pk, SENT_V)
    out = torch.full((w.total_tokens, w.h_q, w.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    pws_bytes = kev.kev_prefill_workspace_size(N, w.total_tokens, shape)
    pws = torch.empty(pws_bytes, dtype=torch.uint8, device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    kev.kev_prefill_attn(q, k, v, w.total_tokens, iv, N, sl, pk, pv, w.n_slots, w.cap, out, shape, pws, pws_bytes, st)
    assert kev.kev_read_status(st) == 0
    out_h = host(out)
    pk_pre, pv_pre = pk.clone(), pv.clone()

    act_h = np.stack([s.active_at(t) for t in range(steps)])
    ins = [s.step_inputs(t) for t in range(steps)]
    qn_h = np.stack([x[0] for x in ins])
    kn_h = np.stack([x[1] for x in ins])
    vn_h = np.stack([x[2] for x in ins])
    del ins
    qn, kn, vn = dev(qn_h), dev(kn_h), dev(vn_h)
    act = torch.from_numpy(act_h).cuda()
    lens0 = torch.from_numpy(s.lens_at(0)).cuda()
    lens = lens0.clone()
    dws_bytes = kev.kev_decode_workspace_size(N, w.cap, shape)
    dws = torch.zeros(dws_bytes, dtype=torch.uint8, device="cuda")
    dst = torch.full((1,), -1, dtype=torch.int32, device="cuda")

    def loop(outs):  # decode, then the lens advance, as two calls
        for t in range(steps):
            kev.kev_decode_attn(qn[t], kn[t], vn[t], pk, pv, w.n_slots, w.cap, sl, lens, act[t], N, outs[t], shape,
                                dws, dws_bytes, dst)
            kev.kev_decode_advance(lens, act[t], N)

    def loop_fused(outs):  # kev_decode_step: the advance folded into the merge kernel
        for t in range(steps):
            kev.kev_decode_step(qn[t], kn[t], vn[t], pk, pv, w.n_slots, w.cap, sl, lens, act[t], N, outs[t], shape,
                                dws, dws_bytes, dst)

    # eager run
    outs_e = torch.full((steps, N, w.h_q, w.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    loop(outs_e)
    torch.cuda.synchronize()
    assert kev.kev_read_status(dst) == 0
    assert np.array_equal(host(lens), s.lens_at(steps))
    eager = host(outs_e)
    final = s.lens_at(steps)
    rows_e = [(host(pk[w.slot_ids[i], :, :final[i]]), host(pv[w.slot_ids[i], :, :final[i]])) for i in range(N)]
    # positions past each question's last appended row keep their sentinels
    for i in range(N):
        tail = slice(int(final[i]), min(w.cap, int(final[i]) + 128))
        assert torch.all(pk[w.slot_ids[i], :, tail] == SENT_K) and torch.all(pv[w.slot_ids[i], :, tail] == SENT_V)
    del outs_e

    # graph replay of the fused steps, from the same post-prefill state
    outs_g = torch.full((steps, N, w.h_q, w.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        loop_fused(outs_g)
    pk.copy_(pk_pre)
    pv.copy_(pv_pre)
    lens.copy_(lens0)
    dst.fill_(-1)
    outs_g.fill_(float("nan"))
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert kev.kev_read_status(dst) == 0
    assert np.array_equal(host(lens), final)
    graph = host(outs_g)
    del outs_g
    for i in range(N):
        gk, gv = host(pk[w.slot_ids[i], :, :final[i]]), host(pv[w.slot_ids[i], :, :final[i]])
        assert np.array_equal(gk, rows_e[i][0]) and np.array_equal(gv, rows_e[i][1]), f"graph pools, question {i}"

    # dropped questions' rows untouched at every step; live rows finite; both runs bit-identical
    live = act_h.astype(bool)
    for t in range(steps):
        assert np.all(np.isnan(W.to_float64(eager[t][~live[t]], "bf16"))), f"eager step {t}: dropped row written"
        assert np.all(np.isnan(W.to_float64(graph[t][~live[t]], "bf16"))), f"graph step {t}: dropped row written"
    assert np.array_equal(eager[live], graph[live]), "graph replay differs from the eager run"
    assert int(live.any(axis=1).sum()) == 116  # steps with at least one live question (seeded schedule)

    jobs = []
    for i in range(N):
        s0, e0 = (int(x) for x in w.intervals[i])
        nd = int(s.n_decoded[i])
        jobs.append({"i": i, "L": e0 - s0, "n_dec": nd, "q": w.q[s0:e0], "k": w.k[s0:e0], "v": w.v[s0:e0],
                     "gpu_out": out_h[s0:e0], "qn": qn_h[:nd, i], "kn": kn_h[:nd, i], "vn": vn_h[:nd, i],
                     "gpu_eager": eager[:nd, i], "gpu_graph": graph[:nd, i],
                     "gpu_pool_k": rows_e[i][0], "gpu_pool_v": rows_e[i][1]})
        assert np.all(live[:nd, i]) and not np.any(live[nd:, i])
    res = _oracle_results(jobs)

    for r in res:
        p = r["prefill"]
        rel = (p["d2"] / p["r2"]) ** 0.5
        assert p["finite"] and p["max"] <= TOL_BF16_MAX and rel <= TOL_BF16_REL_L2, f"prefill question {r['i']}: {p}"
        assert r["pool_k_exact"] and r["pool_v_exact"], f"slot rows of question {r['i']} differ"
    for run in ("eager", "graph"):
        for t in range(steps):
            sts = [r["steps"][t][run] for r in res if t < len(r["steps"])]
            if not sts:
                continue
            mx = max(x["max"] for x in sts)
            rel = (sum(x["d2"] for x in sts) / sum(x["r2"] for x in sts)) ** 0.5
            assert all(x["finite"] for x in sts), f"{run} step {t}: non-finite output"
            assert mx <= TOL_BF16_MAX and rel <= TOL_BF16_REL_L2, f"{run} step {t}: max|d| {mx:.3e}, rel L2 {rel:.3e}"
