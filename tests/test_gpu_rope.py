"""GPU parity of the rotary position encoding path (positions counted per question) against
the CPU oracle: the cos/sin table, the prefill-side rotation with its fused slot write, full
prefill and decode with RoPE, and the position-overflow error.

Tolerance of a rotated value: the kernel computes (a cos - b sin, b cos + a sin) in fp32 from
the table's float cos/sin (each within 2^-25 of the exact value) and rounds once to the storage
type.  Every element is within one unit in the last place of the storage type (plus 4e-7 of the
pair's magnitude for cancellation in the fp32 arithmetic).  For bf16 the fp32 arithmetic error is
~2^16 times smaller than the storage ulp, so the result is the oracle's correctly rounded value
except within ~1e-7 of a rounding boundary: at most one in a thousand elements may differ.  For
fp32 storage the arithmetic error is itself of the order of an ulp, so only the bound applies."""
import numpy as np
import pytest
import torch

import packed_question_isolated_gb300 as kev
import workloads as W
from oracle import kev_oracle as O

from kev_harness import PrefillRun, compare, dev, f64, host, shape_of, tdtype

pytestmark = pytest.mark.gpu

THETA = 1e6


def _table(max_pos, d, theta=THETA):
    t = torch.empty(kev.kev_rope_table_size(max_pos, d) // 4, dtype=torch.float32, device="cuda")
    kev.kev_rope_table(t, max_pos, d, theta)
    return t


def _assert_rotated(got_stored, x64, positions, dtype, theta, what):
    want64 = O.rope_rotate(x64, positions, theta)
    want = O.round_to_stored(want64, dtype)
    g = W.to_float64(got_stored, dtype)
    wv = W.to_float64(want, dtype)
    half = x64.shape[-1] // 2
    mag = np.abs(x64[..., :half]) + np.abs(x64[..., half:])
    mag = np.concatenate([mag, mag], axis=-1)
    if dtype == "bf16":
        ulp = np.ldexp(1.0, (np.floor(np.log2(np.maximum(np.abs(wv), 1e-30))) - 7).astype(int))
    else:
        ulp = np.spacing(np.abs(wv).astype(np.float32)).astype(np.float64)
    err = np.abs(g - want64)
    assert (err <= ulp + 4e-7 * mag).all(), f"{what}: {int((err > ulp + 4e-7 * mag).sum())} elements off by more than 1 ulp"
    if dtype == "bf16":
        frac = float((g != wv).mean()) if g.size else 0.0
        assert frac <= 1e-3, f"{what}: {frac:.2e} of the elements differ from the correctly rounded value"


def test_table_is_the_rounded_cos_sin():
    max_pos, d = 4224, 128
    t = host(_table(max_pos, d)).astype(np.float64).reshape(max_pos, d // 2, 2)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * O.rope_freqs(d, THETA)[None, :]
    assert np.abs(t[..., 0] - np.cos(ang)).max() <= 2.0 ** -24
    assert np.abs(t[..., 1] - np.sin(ang)).max() <= 2.0 ** -24
    np.testing.assert_array_equal(t[0, :, 0], 1.0)
    np.testing.assert_array_equal(t[0, :, 1], 0.0)


CASES = [
    # lengths, h_q, h_kv, d, dtype, gaps, tail, order
    ([300, 129, 1, 0, 517], 8, 2, 128, "bf16", [0, 3, 0, 5, 1], 7, None),
    ([200, 77, 640], 7, 1, 128, "bf16", [2, 0, 1], 3, [2, 0, 1]),
    ([65, 190, 3, 129], 8, 2, 64, "bf16", [1, 1, 1, 1], 1, None),
    ([40, 7, 130], 4, 2, 64, "fp32", [0, 2, 1], 2, None),
    ([256, 5], 2, 1, 128, "fp32", None, 0, None),
]


def _case(i):
    lengths, h_q, h_kv, d, dtype, gaps, tail, order = CASES[i]
    return W.random_case(500 + i, lengths, h_q, h_kv, d, dtype, gaps=gaps, tail=tail, permute_slots=True,
                         n_slots=len(lengths) + 2, order=order)


@pytest.mark.parametrize("case", range(len(CASES)))
def test_rope_prefill_rotates_in_place_and_writes_rotated_slots(case):
    w = _case(case)
    run = PrefillRun(w)
    table = _table(w.cap, w.d)
    kev.kev_build_segments(run.intervals, run.n_questions, w.total_tokens, run.slot_ids, w.n_slots, w.cap,
                           shape_of(w), run.ws, run.ws_bytes, run.status)
    kev.kev_rope_prefill(run.q, run.k, run.v, w.total_tokens, run.intervals, run.n_questions, run.slot_ids,
                         run.pool_k, run.pool_v, w.n_slots, w.cap, shape_of(w), table, w.cap, run.ws, run.ws_bytes,
                         run.status)
    assert run.device_status() == 0
    T = w.total_tokens
    pos = O.prefill_positions(w.intervals, T)
    q_got, k_got = host(run.q)[:T], host(run.k)[:T]
    _assert_rotated(q_got, W.to_float64(w.q, w.dtype)[:T], pos, w.dtype, THETA, f"case {case} q")
    _assert_rotated(k_got, W.to_float64(w.k, w.dtype)[:T], pos, w.dtype, THETA, f"case {case} k")
    gap = pos < 0
    np.testing.assert_array_equal(q_got[gap], np.asarray(w.q)[:T][gap])   # tokens in no question: untouched
    np.testing.assert_array_equal(k_got[gap], np.asarray(w.k)[:T][gap])
    np.testing.assert_array_equal(host(run.v), np.asarray(w.v))
    # the slots hold exactly the rotated K rows (the same bits as k in place) and the V rows
    ek, ev = O.slot_write(host(run.pool_k0), host(run.pool_v0), k_got, w.v, w.intervals, w.slot_ids)
    np.testing.assert_array_equal(host(run.pool_k), ek)
    np.testing.assert_array_equal(host(run.pool_v), ev)


@pytest.mark.parametrize("case", range(len(CASES)))
def test_prefill_attn_rope_full_parity(case):
    w = _case(case)
    run = PrefillRun(w)
    table = _table(w.cap, w.d)
    kev.kev_prefill_attn_rope(run.q, run.k, run.v, w.total_tokens, run.intervals, run.n_questions, run.slot_ids,
                              run.pool_k, run.pool_v, w.n_slots, w.cap, run.out, shape_of(w), table, w.cap,
                              run.ws, run.ws_bytes, run.status)
    assert run.device_status() == 0
    T = w.total_tokens
    ref, _, _ = O.prefill_rope(W.to_float64(w.q, w.dtype), W.to_float64(w.k, w.dtype), W.to_float64(w.v, w.dtype),
                               w.intervals, THETA, scale=w.scale or None)
    got = f64(run.out, w.dtype)[:T]
    compare(got, ref, w.dtype, f"rope case {case}")
    assert (got[O.segment_ids(w.intervals, T) < 0] == 0).all()
    pos = O.prefill_positions(w.intervals, T)
    k_rot = O.round_to_stored(O.rope_rotate(W.to_float64(w.k, w.dtype)[:T], pos, THETA), w.dtype)
    ek, _ = O.slot_write(host(run.pool_k0), host(run.pool_v0), k_rot, w.v, w.intervals, w.slot_ids)
    got_pk, want_pk = W.to_float64(host(run.pool_k), w.dtype), W.to_float64(ek, w.dtype)
    # whole pool within one ulp of the oracle's rounded rotation (untouched positions bit-exact)
    if w.dtype == "bf16":
        assert (got_pk == want_pk).mean() >= 1 - 1e-3
        np.testing.assert_allclose(got_pk, want_pk, rtol=2 ** -7, atol=1e-6)
    else:
        np.testing.assert_allclose(got_pk, want_pk, rtol=2 ** -22, atol=1e-6)


def test_qwen25_7b_config_with_rope_sampled_rows():
    """The Qwen2.5-7B-shaped batch (T = 7921, H_q 28, H_kv 4, d 128) with RoPE, theta = 1e6: sampled
    rows (first, last and boundary rows of every question, plus random ones) on all heads."""
    w = W.qwen25_7b_prefill()
    run = PrefillRun(w)
    table = _table(w.cap, w.d)
    kev.kev_prefill_attn_rope(run.q, run.k, run.v, w.total_tokens, run.intervals, run.n_questions, run.slot_ids,
                              run.pool_k, run.pool_v, w.n_slots, w.cap, run.out, shape_of(w), table, w.cap,
                              run.ws, run.ws_bytes, run.status)
    assert run.device_status() == 0
    T = w.total_tokens
    pos = O.prefill_positions(w.intervals, T)
    q_rot = O.rope_rotate(W.to_float64(w.q, w.dtype), pos, THETA)
    k_rot = O.rope_rotate(W.to_float64(w.k, w.dtype), pos, THETA)
    rng = np.random.default_rng(11)
    rows = set(rng.integers(0, T, 40).tolist())
    for s, e in w.intervals:
        rows.update([s, min(s + 127, e - 1), min(s + 128, e - 1), e - 1])
    rows = sorted(rows)
    ref = O.prefill_rows(q_rot, k_rot, W.to_float64(w.v, w.dtype), w.intervals, rows)
    got = f64(run.out, w.dtype)[rows]
    compare(got, ref, w.dtype, "qwen25 rope rows")


def test_decode_attn_rope_against_oracle():
    """A prefill with RoPE fills the slots; one decode step with RoPE at position lens_i (the cache
    length), with dropped questions, against the oracle's own pool and rotation."""
    lengths, h_q, h_kv, d = [300, 129, 7, 517], 8, 2, 128
    w = W.random_case(77, lengths, h_q, h_kv, d, "bf16", gaps=[0, 2, 0, 1], tail=1, permute_slots=True,
                      n_slots=6)
    run = PrefillRun(w, sentinel_pool=False)
    run.pool_k.zero_()
    run.pool_v.zero_()
    pk0, pv0 = host(run.pool_k), host(run.pool_v)
    table = _table(w.cap, w.d)
    kev.kev_prefill_attn_rope(run.q, run.k, run.v, w.total_tokens, run.intervals, run.n_questions, run.slot_ids,
                              run.pool_k, run.pool_v, w.n_slots, w.cap, run.out, shape_of(w), table, w.cap,
                              run.ws, run.ws_bytes, run.status)
    assert run.device_status() == 0
    rng = np.random.default_rng(78)
    N = len(lengths)
    q_new = W.f32_to_bf16_bits(rng.standard_normal((N, h_q, d), dtype=np.float32) / np.sqrt(d))
    k_new = W.f32_to_bf16_bits(rng.standard_normal((N, h_kv, d), dtype=np.float32) / np.sqrt(d))
    v_new = W.f32_to_bf16_bits(rng.standard_normal((N, h_kv, d), dtype=np.float32))
    lens = np.array(lengths, np.int32)
    active = np.array([1, 0, 1, 1], np.uint8)
    dq, dk, dv = dev(q_new), dev(k_new), dev(v_new)
    out = torch.full((N, h_q, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    shape = kev.make_shape(h_q, h_kv, d, "bf16")
    nb = kev.kev_decode_workspace_size(N, w.cap, shape)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    sl, dl, da = (torch.from_numpy(x).cuda() for x in (np.asarray(w.slot_ids, np.int32), lens, active))
    kev.kev_decode_attn_rope(dq, dk, dv, run.pool_k, run.pool_v, w.n_slots, w.cap, sl, dl, da, N, out, shape,
                             table, w.cap, ws, nb, st)
    assert kev.kev_read_status(st) == 0
    # the oracle's own pool: K rotated at per-question positions, rounded to bf16, written to the slots
    T = w.total_tokens
    pos = O.prefill_positions(w.intervals, T)
    k_rot = O.round_to_stored(O.rope_rotate(W.to_float64(w.k, "bf16"), pos, THETA), "bf16")
    ek, ev = O.slot_write(pk0, pv0, k_rot, w.v, w.intervals, w.slot_ids)
    qn = O.rope_rotate(W.to_float64(q_new, "bf16"), lens, THETA)
    kn = W.to_float64(O.round_to_stored(O.rope_rotate(W.to_float64(k_new, "bf16"), lens, THETA), "bf16"), "bf16")
    o_ref, pk_ref, _ = O.decode(qn, kn, W.to_float64(v_new, "bf16"), W.to_float64(ek, "bf16"),
                                W.to_float64(ev, "bf16"), w.slot_ids, lens, active, "fp64")
    got = f64(out, "bf16")
    live = active.astype(bool)
    compare(got[live], o_ref[live], "bf16", "decode with rope")
    assert np.isnan(got[~live]).all()  # dropped questions: out rows untouched
    # the appended row is the rotated new K, within one ulp; dropped questions' q_new / k_new untouched
    for i in np.nonzero(live)[0]:
        row = f64(run.pool_k, "bf16")[w.slot_ids[i], :, lens[i]]
        np.testing.assert_allclose(row, kn[i], rtol=2 ** -7, atol=1e-6)
    np.testing.assert_array_equal(host(dq)[~live], q_new[~live])
    np.testing.assert_array_equal(host(dk)[~live], k_new[~live])


def test_position_past_the_table_writes_nothing():
    w = _case(0)
    run = PrefillRun(w)
    max_pos = int(max(e - s for s, e in w.intervals)) - 1  # one question longer than the table
    table = _table(max_pos, w.d)
    st = kev.kev_prefill_attn_rope(run.q, run.k, run.v, w.total_tokens, run.intervals, run.n_questions,
                                   run.slot_ids, run.pool_k, run.pool_v, w.n_slots, w.cap, run.out, shape_of(w),
                                   table, max_pos, run.ws, run.ws_bytes, run.status)
    assert st == 0 and run.device_status() == kev.binding.KEV_ERR_POSITION
    np.testing.assert_array_equal(host(run.q), np.asarray(w.q))
    np.testing.assert_array_equal(host(run.k), np.asarray(w.k))
    assert torch.isnan(run.out.float()).all()
    np.testing.assert_array_equal(host(run.pool_k), host(run.pool_k0))
    np.testing.assert_array_equal(host(run.pool_v), host(run.pool_v0))
    # decode side: a live lens at max_pos
    rng = np.random.default_rng(3)
    q_new = W.f32_to_bf16_bits(rng.standard_normal((3, 4, 64), dtype=np.float32))
    k_new = W.f32_to_bf16_bits(rng.standard_normal((3, 2, 64), dtype=np.float32))
    dq, dk = dev(q_new), dev(k_new)
    lens = torch.tensor([5, 16, 2], dtype=torch.int32, device="cuda")
    active = torch.tensor([1, 1, 0], dtype=torch.uint8, device="cuda")
    st_d = torch.zeros(1, dtype=torch.int32, device="cuda")
    kev.kev_rope_decode(dq, dk, lens, active, 3, kev.make_shape(4, 2, 64, "bf16"), _table(16, 64), 16, st_d)
    assert kev.kev_read_status(st_d) == kev.binding.KEV_ERR_POSITION
    np.testing.assert_array_equal(host(dq), q_new)
    np.testing.assert_array_equal(host(dk), k_new)
