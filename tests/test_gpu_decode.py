"""GPU parity of the decode step (append, split-K over slots, early stop) against the oracle."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import kev_oracle as O

from kev_harness import DecodeRun, PrefillRun, compare, f64, host

pytestmark = pytest.mark.gpu


def _check_decode(run, pool_k0, pool_v0, slot_ids, lens, active, q_new, k_new, v_new, dtype, scale=None):
    o_ref, ek, ev = O.decode(q_new, k_new, v_new, pool_k0, pool_v0, slot_ids, lens, active, dtype, scale=scale)
    got = f64(run.out, dtype)
    live = np.asarray(active).astype(bool)
    if live.any():
        compare(got[live], o_ref[live], dtype, "decode o_new")
    assert np.isnan(got[~live]).all(), "rows of dropped questions must be left untouched"
    assert np.array_equal(host(run.pool_k), ek), "pool_k after append differs"
    assert np.array_equal(host(run.pool_v), ev), "pool_v after append differs"


def test_tiny_fp32_prefill_then_one_decode_step():
    w = W.tiny_fp32()
    pre = PrefillRun(w)
    pre.run()
    assert pre.device_status() == 0
    pk0, pv0 = host(pre.pool_k).copy(), host(pre.pool_v).copy()
    lens = w.lengths.copy()
    active = np.ones(w.n_questions, np.uint8)
    run = DecodeRun(w.dtype, w.h_q, w.h_kv, w.d, pre.pool_k, pre.pool_v, w.slot_ids, lens, active,
                    w.q_new, w.k_new, w.v_new, w.cap, w.n_slots)
    run.run()
    assert run.device_status() == 0
    _check_decode(run, pk0, pv0, w.slot_ids, lens, active, w.q_new, w.k_new, w.v_new, w.dtype)


def test_decode_equals_last_row_of_packed_prefill():
    """Invariant (c) on the GPU: decode after prefill == prefill over the extended question."""
    w = W.random_case(17, [200, 31, 300], 8, 2, 128, "bf16", cap=512)
    pre = PrefillRun(w)
    pre.run()
    active = np.ones(3, np.uint8)
    run = DecodeRun(w.dtype, w.h_q, w.h_kv, w.d, pre.pool_k, pre.pool_v, w.slot_ids, w.lengths, active,
                    w.q_new, w.k_new, w.v_new, w.cap, w.n_slots)
    run.run()
    assert run.device_status() == 0
    got = f64(run.out, w.dtype)
    for i, (s, e) in enumerate(w.intervals):
        qe = np.concatenate([w.q[s:e], w.q_new[i:i + 1]])
        ke = np.concatenate([w.k[s:e], w.k_new[i:i + 1]])
        ve = np.concatenate([w.v[s:e], w.v_new[i:i + 1]])
        full = O.prefill(W.to_float64(qe, "bf16"), W.to_float64(ke, "bf16"), W.to_float64(ve, "bf16"),
                         [(0, e - s + 1)])
        compare(got[i], full[-1], "bf16", f"question {i}")


@pytest.mark.parametrize("G", [1, 4, 7, 8, 16])
def test_random_decode_group_sizes(G):
    rng = np.random.default_rng(G)
    h_kv, d, cap, n, n_slots = 2, 128, 700, 9, 12
    pool_k = W.f32_to_bf16_bits(rng.standard_normal((n_slots, h_kv, cap, d), dtype=np.float32))
    pool_v = W.f32_to_bf16_bits(rng.standard_normal((n_slots, h_kv, cap, d), dtype=np.float32))
    slot_ids = rng.permutation(n_slots)[:n].astype(np.int32)
    lens = np.array([0, 1, 255, 256, 257, 511, 512, cap - 1, 37], np.int32)
    active = np.array([1, 1, 1, 1, 0, 1, 1, 1, 1], np.uint8)
    q_new = W.f32_to_bf16_bits(rng.standard_normal((n, h_kv * G, d), dtype=np.float32))
    k_new = W.f32_to_bf16_bits(rng.standard_normal((n, h_kv, d), dtype=np.float32))
    v_new = W.f32_to_bf16_bits(rng.standard_normal((n, h_kv, d), dtype=np.float32))
    run = DecodeRun("bf16", h_kv * G, h_kv, d, pool_k, pool_v, slot_ids, lens, active, q_new, k_new, v_new,
                    cap, n_slots)
    run.run()
    assert run.device_status() == 0
    _check_decode(run, pool_k, pool_v, slot_ids, lens, active, q_new, k_new, v_new, "bf16")
    # the workspace counters are left at zero: a second identical call gives the same bits
    first = host(run.out).copy()
    run.pool_k.copy_(torch.from_numpy(pool_k).view(torch.bfloat16))
    run.pool_v.copy_(torch.from_numpy(pool_v).view(torch.bfloat16))
    run.run()
    assert np.array_equal(first, host(run.out))


@pytest.mark.parametrize("d", [16, 96, 256])
def test_fp32_decode_head_dims_multiple_of_16(d):
    """fp32 decode at head dims other than 64 and 128 (the one-warp-per-head kernel): appended
    rows bit-exact, dropped questions untouched, outputs within the fp32 tolerance."""
    rng = np.random.default_rng(500 + d)
    h_kv, G, cap, n, n_slots = 2, 3, 300, 7, 9
    pool_k = rng.standard_normal((n_slots, h_kv, cap, d), dtype=np.float32)
    pool_v = rng.standard_normal((n_slots, h_kv, cap, d), dtype=np.float32)
    slot_ids = rng.permutation(n_slots)[:n].astype(np.int32)
    lens = np.array([0, 1, 31, 32, 33, 299, 150], np.int32)
    active = np.array([1, 1, 1, 0, 1, 1, 1], np.uint8)
    q_new = rng.standard_normal((n, h_kv * G, d), dtype=np.float32)
    k_new = rng.standard_normal((n, h_kv, d), dtype=np.float32)
    v_new = rng.standard_normal((n, h_kv, d), dtype=np.float32)
    run = DecodeRun("fp32", h_kv * G, h_kv, d, pool_k, pool_v, slot_ids, lens, active, q_new, k_new, v_new,
                    cap, n_slots)
    run.run()
    assert run.device_status() == 0
    _check_decode(run, pool_k, pool_v, slot_ids, lens, active, q_new, k_new, v_new, "fp32")


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("fp32", 64), ("fp32", 96)])
def test_decode_step_equals_decode_then_advance(dtype, d):
    """kev_decode_step = kev_decode_attn, then lens[i] += 1 for live i (tensor-core path: in the
    merge kernel); an invalid step writes nothing and leaves lens as it was."""
    import packed_question_isolated_gb300 as kev
    rng = np.random.default_rng(600 + d)
    h_kv, G, cap, n, n_slots = 2, 4, 900, 8, 10
    f = W.f32_to_bf16_bits if dtype == "bf16" else (lambda x: x)
    pool_k = f(rng.standard_normal((n_slots, h_kv, cap, d), dtype=np.float32))
    pool_v = f(rng.standard_normal((n_slots, h_kv, cap, d), dtype=np.float32))
    slot_ids = rng.permutation(n_slots)[:n].astype(np.int32)
    lens = np.array([0, 127, 128, 500, 899, 3, 640, 255], np.int32)
    active = np.array([1, 1, 0, 1, 1, 1, 0, 1], np.uint8)
    q_new = f(rng.standard_normal((n, h_kv * G, d), dtype=np.float32))
    k_new = f(rng.standard_normal((n, h_kv, d), dtype=np.float32))
    v_new = f(rng.standard_normal((n, h_kv, d), dtype=np.float32))
    ref = DecodeRun(dtype, h_kv * G, h_kv, d, pool_k, pool_v, slot_ids, lens, active, q_new, k_new, v_new, cap,
                    n_slots)
    assert ref.run() == 0 and ref.device_status() == 0
    run = DecodeRun(dtype, h_kv * G, h_kv, d, pool_k, pool_v, slot_ids, lens, active, q_new, k_new, v_new, cap,
                    n_slots)
    st = kev.kev_decode_step(run.q_new, run.k_new, run.v_new, run.pool_k, run.pool_v, run.n_slots, run.cap,
                             run.slot_ids, run.lens, run.active, run.n, run.out, run.shape, run.ws, run.ws_bytes,
                             run.status)
    assert st == 0 and run.device_status() == 0
    assert np.array_equal(host(run.lens), lens + active.astype(np.int32))
    live = active.astype(bool)
    assert np.array_equal(host(run.out)[live], host(ref.out)[live])  # the same kernels, the same bits
    _check_decode(run, pool_k, pool_v, slot_ids, lens, active, q_new, k_new, v_new, dtype)
    # an invalid step (two live questions on one slot): nothing written, lens kept
    bad_slots = slot_ids.copy()
    bad_slots[1] = bad_slots[0]
    bad = DecodeRun(dtype, h_kv * G, h_kv, d, pool_k, pool_v, bad_slots, lens, active, q_new, k_new, v_new, cap,
                    n_slots)
    kev.kev_decode_step(bad.q_new, bad.k_new, bad.v_new, bad.pool_k, bad.pool_v, bad.n_slots, bad.cap,
                        bad.slot_ids, bad.lens, bad.active, bad.n, bad.out, bad.shape, bad.ws, bad.ws_bytes,
                        bad.status)
    assert bad.device_status() == kev.binding.KEV_ERR_SLOT
    assert np.array_equal(host(bad.lens), lens)
    assert np.isnan(f64(bad.out, dtype)).all()
    assert np.array_equal(host(bad.pool_k), pool_k)


def _ramp_pools(rng, n_slots, h_kv, cap, d, growth):
    """K rows aligned with a fixed +-1 direction u and growing with position: q = u scores
    position j at growth * j (log2 units, after the 1/sqrt(d) scale), so later chunks exceed
    the first chunk of a piece by far more than 2^64 in exp2."""
    u = np.where(rng.random(d) < 0.5, -1.0, 1.0).astype(np.float32)
    step = growth / (d / np.sqrt(d) * np.log2(np.e))  # per-position growth of k along u
    ramp = (np.arange(cap, dtype=np.float32) * step)[None, None, :, None]
    noise = rng.standard_normal((n_slots, h_kv, cap, d), dtype=np.float32) * 0.05
    pool_k = W.f32_to_bf16_bits(u[None, None, None, :] * ramp + noise)
    pool_v = W.f32_to_bf16_bits(rng.standard_normal((n_slots, h_kv, cap, d), dtype=np.float32))
    return u, pool_k, pool_v


def test_decode_scores_growing_past_the_reference_max():
    rng = np.random.default_rng(21)
    h_kv, G, d, cap, n = 4, 4, 128, 4096, 8
    u, pool_k, pool_v = _ramp_pools(rng, n, h_kv, cap, d, growth=0.25)  # ~32 log2 units per chunk
    slot_ids = rng.permutation(n).astype(np.int32)
    lens = rng.integers(3000, cap - 1, n).astype(np.int32)
    active = np.ones(n, np.uint8)
    q_new = W.f32_to_bf16_bits(np.broadcast_to(u, (n, h_kv * G, d)).copy())
    k_new = W.f32_to_bf16_bits(rng.standard_normal((n, h_kv, d), dtype=np.float32))
    v_new = W.f32_to_bf16_bits(rng.standard_normal((n, h_kv, d), dtype=np.float32))
    run = DecodeRun("bf16", h_kv * G, h_kv, d, pool_k, pool_v, slot_ids, lens, active, q_new, k_new, v_new,
                    cap, n)
    run.run()
    assert run.device_status() == 0
    _check_decode(run, pool_k, pool_v, slot_ids, lens, active, q_new, k_new, v_new, "bf16")


@pytest.mark.parametrize("h_kv,G", [(1, 4), (1, 16)])
def test_long_context_pieces_merged_across_many_ctas(h_kv, G):
    """Few (question, kv head) pairs, each far longer than one CTA's share of the chunks: every
    pair is split over dozens of CTAs and merged in more than one round."""
    rng = np.random.default_rng(31 + G)
    d, cap, n = 128, 40000, 2
    pool_k = W.f32_to_bf16_bits(rng.standard_normal((n, h_kv, cap, d), dtype=np.float32))
    pool_v = W.f32_to_bf16_bits(rng.standard_normal((n, h_kv, cap, d), dtype=np.float32))
    slot_ids = np.array([1, 0], np.int32)
    lens = np.array([cap - 1, 23456], np.int32)
    active = np.ones(n, np.uint8)
    q_new = W.f32_to_bf16_bits(rng.standard_normal((n, h_kv * G, d), dtype=np.float32))
    k_new = W.f32_to_bf16_bits(rng.standard_normal((n, h_kv, d), dtype=np.float32))
    v_new = W.f32_to_bf16_bits(rng.standard_normal((n, h_kv, d), dtype=np.float32))
    run = DecodeRun("bf16", h_kv * G, h_kv, d, pool_k, pool_v, slot_ids, lens, active, q_new, k_new, v_new,
                    cap, n)
    run.run()
    assert run.device_status() == 0
    _check_decode(run, pool_k, pool_v, slot_ids, lens, active, q_new, k_new, v_new, "bf16")


def test_qwen3_8b_decode_config():
    w = W.qwen3_8b_decode()
    run = DecodeRun(w.dtype, w.h_q, w.h_kv, w.d, w.pool_k, w.pool_v, w.slot_ids, w.lens, w.active,
                    w.q_new, w.k_new, w.v_new, w.cap, w.n_slots)
    run.run()
    assert run.device_status() == 0
    _check_decode(run, w.pool_k, w.pool_v, w.slot_ids, w.lens, w.active, w.q_new, w.k_new, w.v_new, w.dtype)


def test_all_questions_dropped_is_a_no_op():
    rng = np.random.default_rng(3)
    pool = W.f32_to_bf16_bits(rng.standard_normal((4, 2, 64, 64), dtype=np.float32))
    q = W.f32_to_bf16_bits(rng.standard_normal((4, 4, 64), dtype=np.float32))
    kv = W.f32_to_bf16_bits(rng.standard_normal((4, 2, 64), dtype=np.float32))
    # dropped questions are not validated: duplicate and out-of-range slots, lens past cap
    run = DecodeRun("bf16", 4, 2, 64, pool, pool.copy(), [0, 0, 9, -1], [5, 64, 70, 3], np.zeros(4, np.uint8),
                    q, kv, kv, 64, 4)
    run.run()
    assert run.device_status() == 0
    assert np.isnan(f64(run.out, "bf16")).all()
    assert np.array_equal(host(run.pool_k), pool)


def test_stress_config_prefill_and_first_decode_steps():
    s = W.stress()
    w = s.prefill
    pre = PrefillRun(w)
    pre.run()
    assert pre.device_status() == 0
    got = f64(pre.out, w.dtype)
    q, k, v = (W.to_float64(x, w.dtype) for x in (w.q, w.k, w.v))
    for qi in range(0, w.n_questions, 17):
        s0, e0 = w.intervals[qi]
        ref = O.prefill(q[s0:e0], k[s0:e0], v[s0:e0], [(0, e0 - s0)])
        compare(got[s0:e0], ref, w.dtype, f"stress question {qi}")
    pool_k, pool_v = host(pre.pool_k), host(pre.pool_v)
    ek, ev = O.slot_write(host(pre.pool_k0), host(pre.pool_v0), w.k, w.v, w.intervals, w.slot_ids)
    assert np.array_equal(pool_k, ek) and np.array_equal(pool_v, ev)
    # three decode steps with the seeded early-stop schedule; lens advanced on the device
    lens_dev = torch.from_numpy(s.lens_at(0)).cuda()
    import packed_question_isolated_gb300 as kev
    for step in range(3):
        qn, kn, vn = s.step_inputs(step)
        active = s.active_at(step)
        lens = host(lens_dev).copy()
        assert np.array_equal(lens, s.lens_at(step))
        run = DecodeRun(w.dtype, w.h_q, w.h_kv, w.d, pre.pool_k, pre.pool_v, w.slot_ids, lens, active,
                        qn, kn, vn, w.cap, w.n_slots)
        run.run()
        assert run.device_status() == 0
        o_ref, pool_k, pool_v = O.decode(qn, kn, vn, pool_k, pool_v, w.slot_ids, lens, active, w.dtype,
                                         inplace=True)
        live = active.astype(bool)
        compare(f64(run.out, w.dtype)[live], o_ref[live], w.dtype, f"step {step}")
        kev.kev_decode_advance(lens_dev, run.active, w.n_questions)
    assert np.array_equal(host(pre.pool_k), pool_k)
