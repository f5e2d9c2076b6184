"""GPU parity of prefill (segments, attention, slot write) against the CPU oracle."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import kev_oracle as O

from kev_harness import PrefillRun, compare, f64, host

pytestmark = pytest.mark.gpu


def _oracle_out(w):
    return O.prefill(W.to_float64(w.q, w.dtype), W.to_float64(w.k, w.dtype), W.to_float64(w.v, w.dtype),
                     w.intervals, scale=w.scale or None)


def _check_pools(run, w):
    pk0, pv0 = host(run.pool_k0), host(run.pool_v0)
    ek, ev = O.slot_write(pk0, pv0, w.k, w.v, w.intervals, w.slot_ids)
    assert np.array_equal(host(run.pool_k), ek), "pool_k differs from the oracle's bit copy"
    assert np.array_equal(host(run.pool_v), ev), "pool_v differs from the oracle's bit copy"


def test_tiny_fp32_config_full_parity():
    w = W.tiny_fp32()
    run = PrefillRun(w)
    run.run()
    assert run.device_status() == 0
    compare(f64(run.out, w.dtype), _oracle_out(w), w.dtype, "tiny fp32 prefill")
    _check_pools(run, w)


CASES = [
    # lengths, h_q, h_kv, d, dtype, gaps, tail
    ([300, 129, 1, 0, 517], 8, 2, 128, "bf16", [0, 3, 0, 5, 1], 7),
    ([128, 256, 127, 383], 4, 4, 128, "bf16", None, 0),
    ([200, 77, 640], 7, 1, 128, "bf16", [2, 0, 1], 3),
    ([65, 190, 3, 129], 8, 2, 64, "bf16", [1, 1, 1, 1], 1),
    ([40, 7, 130], 4, 2, 64, "fp32", [0, 2, 1], 2),
    ([256, 5], 2, 1, 128, "fp32", None, 0),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_random_cases_full_parity(case):
    lengths, h_q, h_kv, d, dtype, gaps, tail = CASES[case]
    w = W.random_case(300 + case, lengths, h_q, h_kv, d, dtype, gaps=gaps, tail=tail, permute_slots=True,
                      n_slots=len(lengths) + 2)
    run = PrefillRun(w)
    run.run()
    assert run.device_status() == 0
    ref = _oracle_out(w)
    got = f64(run.out, w.dtype)[:w.total_tokens]
    compare(got, ref, dtype, f"case {case}")
    seg = O.segment_ids(w.intervals, w.total_tokens)
    assert (got[seg < 0] == 0).all(), "rows of tokens in no question must be 0"
    _check_pools(run, w)


@pytest.mark.parametrize("d", [16, 48, 96, 256])
def test_fp32_head_dims_multiple_of_16(d):
    """fp32 (CUDA cores) at head dims other than 64 and 128: any multiple of 16 up to 256."""
    w = W.random_case(400 + d, [70, 1, 0, 161, 33], 6, 2, d, "fp32", gaps=[0, 2, 1, 0, 3], tail=2,
                      permute_slots=True, n_slots=7)
    run = PrefillRun(w)
    run.run()
    assert run.device_status() == 0
    got = f64(run.out, w.dtype)[:w.total_tokens]
    compare(got, _oracle_out(w), "fp32", f"fp32 d={d}")
    seg = O.segment_ids(w.intervals, w.total_tokens)
    assert (got[seg < 0] == 0).all()
    _check_pools(run, w)


def test_unsorted_interval_order_and_no_slot_write():
    w = W.random_case(77, [90, 300, 12, 150], 8, 2, 128, "bf16", gaps=[3, 0, 2, 0], order=[2, 0, 3, 1])
    run = PrefillRun(w, slots=False)
    run.run()
    assert run.device_status() == 0
    compare(f64(run.out, w.dtype), _oracle_out(w), w.dtype, "unsorted")


def test_qwen25_7b_config_every_question_against_oracle():
    w = W.qwen25_7b_prefill()
    run = PrefillRun(w)
    run.run()
    assert run.device_status() == 0
    got = f64(run.out, w.dtype)
    q, k, v = (W.to_float64(x, w.dtype) for x in (w.q, w.k, w.v))
    for (s, e) in w.intervals:
        # invariant (b) of the oracle: the packed rows of a question equal the question alone
        ref = O.prefill(q[s:e], k[s:e], v[s:e], [(0, e - s)])
        compare(got[s:e], ref, w.dtype, f"question [{s},{e})")
    _check_pools(run, w)


def test_qwen3_8b_config_sampled_rows_and_pools():
    w = W.qwen3_8b_prefill()
    run = PrefillRun(w)
    run.run()
    assert run.device_status() == 0
    got = f64(run.out, w.dtype)
    q, k, v = (W.to_float64(x, w.dtype) for x in (w.q, w.k, w.v))
    rng = np.random.default_rng(0)
    rows = set(rng.choice(w.total_tokens, 40, replace=False).tolist())
    for s, e in w.intervals:           # first, last and a tile-boundary row of each question
        rows.update({int(s), int(e - 1), int(min(e - 1, s + 128))})
    rows = sorted(rows)
    ref = O.prefill_rows(q, k, v, w.intervals, rows)
    compare(got[rows], ref, w.dtype, "sampled rows")
    # whole short questions
    for s, e in w.intervals:
        if e - s <= 300:
            ref = O.prefill(q[s:e], k[s:e], v[s:e], [(0, e - s)])
            compare(got[s:e], ref, w.dtype, f"question [{s},{e})")
    _check_pools(run, w)


def test_qwen3_8b_config_every_row_against_oracle():
    """Every output row of the Qwen3-8B-shaped batch (T = 24,100, questions up to 4096 tokens)
    against the oracle, one (question, kv group) per job in spawned worker processes."""
    import multiprocessing as mp
    import os
    import prefill_oracle
    from kev_harness import TOL_BF16_MAX, TOL_BF16_REL_L2
    w = W.qwen3_8b_prefill()
    run = PrefillRun(w)
    run.run()
    assert run.device_status() == 0
    out = host(run.out)
    G = w.h_q // w.h_kv
    jobs = []
    for i, (s, e) in enumerate(w.intervals):
        s, e = int(s), int(e)
        for g in range(w.h_kv):
            jobs.append({"i": i, "g": g, "L": e - s, "q": w.q[s:e, g * G:(g + 1) * G], "k": w.k[s:e, g:g + 1],
                         "v": w.v[s:e, g:g + 1], "gpu_out": out[s:e, g * G:(g + 1) * G]})
    jobs.sort(key=lambda j: -j["L"])  # the longest start first
    ctx = mp.get_context("spawn")  # this process already holds a CUDA context
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in saved:
        os.environ[k] = "1"
    try:
        with ctx.Pool(max(1, min(32, os.cpu_count() or 1))) as pool:
            res = pool.map(prefill_oracle.check_group, jobs, chunksize=1)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    per_q = {}
    for r in res:
        assert r["finite"], f"question {r['i']} group {r['g']}: non-finite output"
        a = per_q.setdefault(r["i"], [0.0, 0.0, 0.0])
        a[0], a[1], a[2] = max(a[0], r["max"]), a[1] + r["d2"], a[2] + r["r2"]
    assert len(per_q) == w.n_questions
    for i, (mx, d2, r2) in per_q.items():
        rel = (d2 / r2) ** 0.5 if r2 > 0 else 0.0
        assert mx <= TOL_BF16_MAX and rel <= TOL_BF16_REL_L2, f"question {i}: max|d| {mx:.3e}, rel L2 {rel:.3e}"


def test_deterministic_and_isolated_bitwise():
    """Same call twice gives identical bits; a question's rows do not depend on its neighbours
    or on where it sits in the packed sequence (segment-local tiling)."""
    w = W.random_case(88, [150, 260, 33, 129], 8, 2, 128, "bf16", gaps=[0, 1, 0, 2])
    a = PrefillRun(w, slots=False)
    a.run()
    first = host(a.out).copy()
    a.run()
    assert np.array_equal(first, host(a.out))
    for i, (s, e) in enumerate(w.intervals):
        alone = W.Workload(name="alone", seed=0, dtype=w.dtype, h_q=w.h_q, h_kv=w.h_kv, d=w.d,
                           lengths=np.array([e - s], np.int32), intervals=np.array([[5, 5 + e - s]], np.int32),
                           total_tokens=int(e - s + 9), q=np.concatenate([w.q[:5], w.q[s:e], w.q[:4]]),
                           k=np.concatenate([w.k[:5], w.k[s:e], w.k[:4]]),
                           v=np.concatenate([w.v[:5], w.v[s:e], w.v[:4]]),
                           slot_ids=np.array([0], np.int32), n_slots=1, cap=int(e - s))
        b = PrefillRun(alone, slots=False)
        b.run()
        assert np.array_equal(host(b.out)[5:5 + e - s], first[s:e]), f"question {i} not bitwise isolated"


@pytest.mark.parametrize("h_q,h_kv", [(4, 2), (7, 1), (14, 2)])
def test_work_list_covers_exactly_the_allowed_tiles(h_q, h_kv):
    import packed_question_isolated_gb300 as kev
    w = W.random_case(99, [300, 1, 0, 129, 128, 257, 640], h_q, h_kv, 64, "bf16", gaps=[0, 2, 1, 0, 3, 1, 0],
                      tail=5)
    run = PrefillRun(w)
    run.run()
    items, n = kev.kev_read_work_list(run.ws, run.ws_bytes, 100000)
    assert n == len(items)
    T = w.total_tokens
    allowed = O.allowed_mask(w.intervals, T)
    covered = np.zeros((w.h_q, T, T), dtype=np.int32)
    costs = []
    G = w.h_q // w.h_kv
    n_two = 0
    for (qi, r0, rows, hw) in items:
        h0, nh, two = hw & 0xffff, (hw >> 16) & 0x3fff, (hw >> 30) & 1
        s, e = w.intervals[qi]
        if two:
            # one q-head, query tiles starting at r0 (whole) and r0 + 128 (`rows` rows)
            n_two += 1
            assert nh == 1 and G % 2 == 1 and h0 % G == G - 1, "only the odd head left over in a group"
            assert (r0 - s) % 256 == 0 and r0 + 128 + rows <= e and 0 < rows <= 128
            tiles = [(r0, 128), (r0 + 128, rows)]
            heads = [h0]
        else:
            assert 1 <= nh <= 2 and h0 // G == (h0 + nh - 1) // G, "an item's heads share one kv head"
            assert s <= r0 and r0 + rows <= e and 0 < rows <= 128 and (r0 - s) % 128 == 0
            tiles = [(r0, rows)]
            heads = list(range(h0, h0 + nh))
        for (t0, tr) in tiles:
            # key range of the tile: [s, t0 + tr)
            assert allowed[t0:t0 + tr, s:t0 + tr].any(), "an item with no allowed entry was scheduled"
            for h in heads:
                covered[h, t0:t0 + tr, s:t0 + tr] += 1
        last = tiles[-1][0]
        costs.append((last - s) // 128 + 1)
    for h in range(w.h_q):
        assert (covered[h][allowed] == 1).all(), "allowed entry not covered exactly once"
        assert (covered[h] <= 1).all()
    assert costs == sorted(costs, reverse=True), "items are not ordered longest first"
    if G % 2 == 1 and G > 1:
        assert n_two > 0


@pytest.mark.parametrize("h_q,h_kv", [(4, 1), (7, 1), (14, 2), (2, 2), (3, 1), (16, 1)])
def test_work_units_cover_exactly_the_allowed_tiles(h_q, h_kv):
    """bf16 with d = 128: the CTA-pair kernel's units cover every allowed (head, query, key) entry
    exactly once; a unit's halves share its kv head; tiles A and B differ by at most one key tile
    (two for G = 1); units come longest first; and the output matches the oracle."""
    import packed_question_isolated_gb300 as kev
    w = W.random_case(98, [300, 1, 0, 129, 128, 257, 640, 1100], h_q, h_kv, 128, "bf16",
                      gaps=[0, 2, 1, 0, 3, 1, 0, 4], tail=5)
    run = PrefillRun(w)
    run.run()
    assert run.device_status() == 0
    units, n = kev.kev_read_work_units(run.ws, run.ws_bytes, 100000)
    assert n == len(units)
    T = w.total_tokens
    G = w.h_q // w.h_kv
    allowed = O.allowed_mask(w.intervals, T)
    covered = np.zeros((w.h_q, T, T), dtype=np.int32)
    costs = []
    for (qi, g, nkv_a, nkv_b, a0, a1, b0, b1) in units:
        s, e = w.intervals[qi]
        assert 0 <= g < w.h_kv
        for nkv_t, halves in ((nkv_a, (a0, a1)), (nkv_b, (b0, b1))):
            on = [x for x in halves if x >= 0]
            assert nkv_t == (max((x >> 8) + 1 for x in on) if on else 0)
            for x in on:
                m, hl = x >> 8, x & 0xff
                assert hl < G
                t0 = s + 128 * m
                tr = min(128, e - t0)
                assert tr > 0
                covered[g * G + hl, t0:t0 + tr, s:t0 + tr] += 1
        assert nkv_a > 0 and (nkv_b == 0 or 0 <= nkv_b - nkv_a <= (2 if G == 1 else 1))
        costs.append(max(nkv_a, nkv_b))
    for h in range(w.h_q):
        assert (covered[h][allowed] == 1).all(), "allowed entry not covered exactly once"
        assert (covered[h] <= 1).all()
    assert costs == sorted(costs, reverse=True), "units are not ordered longest first"
    with pytest.raises(kev.KevError):
        kev.kev_read_work_list(run.ws, run.ws_bytes, 10)
    compare(f64(run.out, w.dtype), _oracle_out(w), w.dtype, "unit-form prefill")
    _check_pools(run, w)


def test_scores_growing_past_the_reference_max():
    """Keys aligned with the queries and growing along the sequence: later key tiles exceed the
    first tile of an item by far more than 2^64 in exp2 (the exact rescaling path)."""
    rng = np.random.default_rng(23)
    h_q, h_kv, d, L = 4, 2, 128, 900
    w = W.random_case(23, [L, 130], h_q, h_kv, d, "bf16", gaps=[1, 0], tail=2)
    u = np.where(rng.random(d) < 0.5, -1.0, 1.0).astype(np.float32)
    step = 0.25 / (d / np.sqrt(d) * np.log2(np.e))  # ~32 log2 units per 128 keys
    pos = np.zeros(w.total_tokens, np.float32)
    for s0, e0 in w.intervals:
        pos[s0:e0] = np.arange(e0 - s0, dtype=np.float32)
    k = u[None, None, :] * (pos * step)[:, None, None] + rng.standard_normal(
        (w.total_tokens, h_kv, d), dtype=np.float32) * 0.05
    w.k = W.f32_to_bf16_bits(k)
    w.q = W.f32_to_bf16_bits(np.broadcast_to(u, (w.total_tokens, h_q, d)).copy())
    run = PrefillRun(w)
    run.run()
    assert run.device_status() == 0
    compare(f64(run.out, w.dtype), _oracle_out(w), w.dtype, "growing scores")


def test_empty_batch_and_all_empty_questions():
    w = W.random_case(5, [0, 0], 4, 2, 64, "bf16", gaps=[3, 2], tail=1)
    run = PrefillRun(w)
    run.run()
    assert run.device_status() == 0
    assert (f64(run.out, w.dtype)[:w.total_tokens] == 0).all()
    _check_pools(run, w)
