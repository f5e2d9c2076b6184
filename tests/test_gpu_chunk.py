"""GPU parity of chunked prefill into slots against the CPU oracle: chunks after cached
prefixes of several tiles, chunks in sequence against one prefill (bit for bit), and the
prefix / capacity errors that must write nothing."""
import numpy as np
import pytest
import torch

import packed_question_isolated_gb300 as kev
import workloads as W
from oracle import kev_oracle as O

from kev_harness import PrefillRun, compare, dev, f64, host, shape_of

pytestmark = pytest.mark.gpu


def _itensor(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def _expected_pools(pk0, pv0, w, prefix, cap):
    """The oracle's slot contents after the chunk, plus the documented zeroing of the slot rows
    from the chunk's end up to the next multiple of 128."""
    _, ek, ev = O.prefill_chunk(w.q, w.k, w.v, w.intervals, prefix, w.slot_ids, pk0, pv0, w.dtype)
    for (s, e), P, slot in zip(w.intervals, prefix, w.slot_ids):
        L = int(e - s)
        if L == 0:
            continue
        p0 = int(P) + L
        p1 = min(cap, (p0 + 127) // 128 * 128)
        ek[slot, :, p0:p1] = 0
        ev[slot, :, p0:p1] = 0
    return ek, ev


def _run_chunk(w, prefix, cap, pk, pv, out, ws, ws_bytes, status, slots=None):
    return kev.kev_prefill_chunk(dev(w.q), dev(w.k), dev(w.v), w.total_tokens, _itensor(w.intervals),
                                 len(w.intervals), _itensor(prefix), _itensor(w.slot_ids if slots is None else slots),
                                 pk, pv, w.n_slots, cap, out, shape_of(w), ws, ws_bytes, status, check=False)


CASES = [
    # chunk lengths, prefixes, h_q, h_kv, d
    ([300, 129, 1, 0, 517], [256, 0, 128, 384, 640], 8, 2, 128),
    ([200, 77, 640], [128, 1024, 0], 7, 1, 128),
    ([65, 190, 3, 129], [0, 128, 256, 384], 4, 4, 64),
    ([257, 128], [512, 128], 28, 4, 128),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_prefill_chunk_against_oracle(case):
    lengths, prefix, h_q, h_kv, d = CASES[case]
    cap = 1792
    w = W.random_case(700 + case, lengths, h_q, h_kv, d, "bf16", gaps=[1] * len(lengths), tail=2,
                      permute_slots=True, n_slots=len(lengths) + 1, cap=cap)
    rng = np.random.default_rng(701 + case)
    # the cached prefixes (and everything else in the pool): random bf16 values
    pool_shape = (w.n_slots, h_kv, cap, d)
    pk0 = W.f32_to_bf16_bits(rng.standard_normal(pool_shape, dtype=np.float32))
    pv0 = W.f32_to_bf16_bits(rng.standard_normal(pool_shape, dtype=np.float32))
    run = PrefillRun(w, slots=False)
    pk, pv = dev(pk0), dev(pv0)
    st = _run_chunk(w, prefix, cap, pk, pv, run.out, run.ws, run.ws_bytes, run.status)
    assert st == 0 and run.device_status() == 0
    ref, _, _ = O.prefill_chunk(w.q, w.k, w.v, w.intervals, prefix, w.slot_ids, pk0, pv0, "bf16")
    T = w.total_tokens
    got = f64(run.out, "bf16")[:T]
    compare(got, ref, "bf16", f"chunk case {case}")
    assert (got[O.segment_ids(w.intervals, T) < 0] == 0).all()
    ek, ev = _expected_pools(pk0, pv0, w, prefix, cap)
    np.testing.assert_array_equal(host(pk), ek)
    np.testing.assert_array_equal(host(pv), ev)


@pytest.mark.parametrize("h_q,h_kv", [(8, 2), (7, 1)])
def test_chunks_in_sequence_equal_one_prefill_bitwise(h_q, h_kv):
    """Questions prefilled in one call, and the same questions as two chunks (the first ending on
    a tile boundary): the second chunk's rows reduce the same key tiles in the same order, so they
    equal the one-shot rows bit for bit, and so do the slots."""
    lengths, cut = [700, 300, 129], [384, 128, 128]
    cap = 768
    w = W.random_case(720 + h_q, lengths, h_q, h_kv, 128, "bf16", gaps=[0, 1, 2], tail=1, n_slots=3, cap=cap)
    one = PrefillRun(w)
    one.run()
    assert one.device_status() == 0
    # two chunks: [s, s + cut) with prefix 0, then [s + cut, e) with prefix cut
    iv = np.asarray(w.intervals)
    pk = torch.zeros((3, h_kv, cap, 128), dtype=torch.bfloat16, device="cuda")
    pv = torch.zeros_like(pk)
    outs = []
    for part in range(2):
        ivp = np.stack([iv[:, 0], iv[:, 0] + cut], 1) if part == 0 else np.stack([iv[:, 0] + cut, iv[:, 1]], 1)
        wp = W.random_case(720 + h_q, lengths, h_q, h_kv, 128, "bf16", gaps=[0, 1, 2], tail=1, n_slots=3, cap=cap)
        wp.intervals = ivp.astype(np.int32)
        out = torch.full((w.total_tokens, h_q, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        nb = kev.kev_prefill_workspace_size(3, w.total_tokens, shape_of(w))
        ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        prefix = [0, 0, 0] if part == 0 else cut
        assert _run_chunk(wp, prefix, cap, pk, pv, out, ws, nb, st) == 0
        assert kev.kev_read_status(st) == 0
        outs.append((ivp, host(out)))
    ref = host(one.out)
    for ivp, o in outs:
        for s, e in ivp:
            np.testing.assert_array_equal(o[s:e], ref[s:e])
    hk, hv, rk, rv = host(pk), host(pv), host(one.pool_k), host(one.pool_v)
    for i, L in enumerate(lengths):
        np.testing.assert_array_equal(hk[w.slot_ids[i], :, :L], rk[w.slot_ids[i], :, :L])
        np.testing.assert_array_equal(hv[w.slot_ids[i], :, :L], rv[w.slot_ids[i], :, :L])


def test_qwen25_7b_batch_as_second_chunks_sampled_rows():
    """The Qwen2.5-7B-shaped batch (8 questions, H_q 28, H_kv 4) prefilled as two chunks per question
    (the first ending on the last tile boundary at or below half the question): sampled rows of
    the second chunks against the one-shot oracle rows."""
    w = W.qwen25_7b_prefill()
    cap = (w.cap + 127) // 128 * 128
    iv = np.asarray(w.intervals)
    L = iv[:, 1] - iv[:, 0]
    cut = (L // 2) // 128 * 128
    pk = torch.zeros((w.n_slots, w.h_kv, cap, w.d), dtype=torch.bfloat16, device="cuda")
    pv = torch.zeros_like(pk)
    nb = kev.kev_prefill_workspace_size(w.n_questions, w.total_tokens, shape_of(w))
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((w.total_tokens, w.h_q, w.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    q, k, v = dev(w.q), dev(w.k), dev(w.v)
    for part in range(2):
        ivp = np.stack([iv[:, 0], iv[:, 0] + cut], 1) if part == 0 else np.stack([iv[:, 0] + cut, iv[:, 1]], 1)
        prefix = np.zeros(len(L), np.int32) if part == 0 else cut
        assert kev.kev_prefill_chunk(q, k, v, w.total_tokens, _itensor(ivp), w.n_questions, _itensor(prefix),
                                     _itensor(w.slot_ids), pk, pv, w.n_slots, cap, out, shape_of(w), ws, nb, st) == 0
        assert kev.kev_read_status(st) == 0
    rng = np.random.default_rng(12)
    rows = set()
    for (s, e), c in zip(iv, cut):
        rows.update([s + c, min(s + c + 127, e - 1), e - 1, int(rng.integers(s + c, e))])
    rows = sorted(rows)
    ref = O.prefill_rows(W.to_float64(w.q, "bf16"), W.to_float64(w.k, "bf16"), W.to_float64(w.v, "bf16"),
                         w.intervals, rows)
    compare(f64(out, "bf16")[rows], ref, "bf16", "qwen25 second chunks")


def test_prefix_and_capacity_errors_write_nothing():
    lengths, cap = [200, 100], 512
    w = W.random_case(730, lengths, 4, 2, 128, "bf16", gaps=[1, 1], tail=1, n_slots=2, cap=cap)
    for prefix, want in (([100, 0], kev.binding.KEV_ERR_PREFIX), ([384, 0], kev.binding.KEV_ERR_SLOT_OVERFLOW)):
        assert O.validate_chunk(w.intervals, w.total_tokens, prefix, w.slot_ids, 2, cap) == \
            (O.PREFIX if want == kev.binding.KEV_ERR_PREFIX else O.SLOT_OVERFLOW)
        run = PrefillRun(w, slots=False)
        pk = torch.full((2, 2, cap, 128), -7.0, dtype=torch.bfloat16, device="cuda")
        pv = torch.full((2, 2, cap, 128), -9.0, dtype=torch.bfloat16, device="cuda")
        assert _run_chunk(w, prefix, cap, pk, pv, run.out, run.ws, run.ws_bytes, run.status) == 0
        assert run.device_status() == want
        assert torch.isnan(run.out.float()).all()
        assert (pk.float() == -7.0).all() and (pv.float() == -9.0).all()
