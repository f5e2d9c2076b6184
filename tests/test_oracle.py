"""Pins of the CPU oracle against what the pages and mathematics fix.

Each test ties the oracle to something other than itself: the pages' worked
examples (fixtures under tests/golden/, each with its citation), closed
forms, the invariants (a)-(d), a library routine (torch's scaled dot-product
attention in float64) and a separate pure-Python brute force.  The
``test_planted_*`` tests plant plausible mistakes into a copy of the oracle
and check that at least one pin catches each of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import workloads as W
from oracle import brute
from oracle import kev_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            if "->" in line:
                k, v = line.split("->")
                vals[k.strip()] = float(v)
            elif "=" in line:
                k, v = line.split("=", 1)
                vals[k.strip()] = [float(x) for x in v.split()]
    return vals


def _f64(w, name):
    return W.to_float64(getattr(w, name), w.dtype)


# ---------------------------------------------------------------------------
# worked examples printed on the pages
# ---------------------------------------------------------------------------

def test_worked_example_online_softmax():
    g = _golden("online_softmax_worked_example.txt")
    k = np.array(g["k"]).reshape(4, 1, 1)
    v = np.array(g["v"]).reshape(4, 1, 1)
    q = np.full((4, 1, 1), g["q"][0])
    out = O.prefill(q, k, v, [(0, 4)], scale=g["scale"][0])
    # the last token sees all four keys: the page's single query row
    assert round(float(out[3, 0, 0]), int(g["decimals"][0])) == pytest.approx(g["output"][0], abs=0)
    o_online, alphas = O.online_softmax_row(q[3, 0], k[:, 0], v[:, 0], g["scale"][0], int(g["block"][0]))
    assert round(float(o_online[0]), 6) == g["output"][0]
    assert abs(o_online[0] - out[3, 0, 0]) < 1e-12
    assert round(100 * alphas[1], 1) == g["second_block_rescale_percent"][0]
    bf = brute.prefill(q.tolist(), k.tolist(), v.tolist(), [(0, 4)], 1.0)
    assert abs(bf[3][0][0] - out[3, 0, 0]) < 1e-12


def test_worked_example_arithmetic_intensity():
    from packed_question_isolated_gb300.roofline import projection_intensity
    g = _golden("arithmetic_intensity.txt")
    d, b = int(g["d"][0]), int(g["bytes_per_value"][0])
    assert round(projection_intensity(1, d, b), 2) == g["n=1"]
    assert round(projection_intensity(1024, d, b), 2) == g["n=1024"]


def test_kv_cache_demo_shapes_and_last_row():
    g = _golden("kv_cache_demo.txt")
    T, dh = int(g["T"][0]), int(g["d_h"][0])
    rng = np.random.default_rng(7)
    x = rng.standard_normal((T + 1, 1, dh))
    k = rng.standard_normal((T + 1, 1, dh))
    v = rng.standard_normal((T + 1, 1, dh))
    full, P = O.prefill(x, k, v, [(0, T + 1)], return_probs=True)
    assert float(np.abs(np.triu(P[0], 1)).max()) == g["future_weight_max"][0]
    pool_k = np.zeros((1, 1, T + 1, dh))
    pool_v = np.zeros((1, 1, T + 1, dh))
    pool_k[0, 0, :T] = k[:T, 0]
    pool_v[0, 0, :T] = v[:T, 0]
    o, pk, _ = O.decode(x[T:T + 1].astype(np.float32), k[T:T + 1].astype(np.float32),
                        v[T:T + 1].astype(np.float32), pool_k.astype(np.float32),
                        pool_v.astype(np.float32), [0], [T], [1], "fp32")
    assert pk[0, 0, :T + 1].shape == tuple(int(x) for x in g["k_cache_after_step"])
    assert o[0].shape == tuple(int(x) for x in g["z_cached"])
    # same values rounded to fp32 on both sides
    x32 = x.astype(np.float32).astype(np.float64)
    k32 = k.astype(np.float32).astype(np.float64)
    v32 = v.astype(np.float32).astype(np.float64)
    full32 = O.prefill(x32, k32, v32, [(0, T + 1)])
    assert np.max(np.abs(o[0] - full32[T])) < 1e-12


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------

def test_closed_form_zero_keys_give_prefix_mean():
    rng = np.random.default_rng(11)
    lengths = [5, 9, 1, 7]
    iv = W.pack_intervals(lengths, gaps=[0, 2, 1, 3])
    T = int(iv[:, 1].max()) + 2
    q = rng.standard_normal((T, 4, 8))
    k = np.zeros((T, 2, 8))
    v = rng.standard_normal((T, 2, 8))
    out = O.prefill(q, k, v, iv)
    for s, e in iv:
        for t in range(s, e):
            for h in range(4):
                expect = v[s:t + 1, h // 2].mean(axis=0)
                assert np.max(np.abs(out[t, h] - expect)) < 1e-12


def test_closed_form_single_token_question_copies_v():
    rng = np.random.default_rng(12)
    iv = np.array([[0, 3], [3, 4], [4, 9]])
    q = rng.standard_normal((9, 2, 16))
    k = rng.standard_normal((9, 1, 16))
    v = rng.standard_normal((9, 1, 16))
    out = O.prefill(q, k, v, iv)
    assert np.array_equal(out[3, 0], v[3, 0]) and np.array_equal(out[3, 1], v[3, 0])
    assert np.array_equal(out[0, 0], v[0, 0])


def test_closed_form_dominant_key_selects_its_value():
    rng = np.random.default_rng(13)
    T, d = 12, 4
    q = np.zeros((T, 1, d))
    q[:, 0, 0] = 1.0
    k = rng.standard_normal((T, 1, d)) * 0.01
    k[5, 0, 0] = 80.0  # score 40 above the rest at scale 1/2
    v = rng.standard_normal((T, 1, d))
    out = O.prefill(q, k, v, [(0, T)])
    for t in range(5, T):
        assert np.max(np.abs(out[t, 0] - v[5, 0])) < 1e-12
    # before the key is visible it has no effect
    assert np.max(np.abs(out[4, 0] - v[5, 0])) > 1e-3


# ---------------------------------------------------------------------------
# invariants (a)-(d)
# ---------------------------------------------------------------------------

def test_invariant_a_future_and_cross_question_weights_are_exactly_zero():
    w = W.random_case(21, [6, 1, 9, 4], 4, 2, 8, "fp32", gaps=[1, 0, 2, 3], tail=2)
    _, P = O.prefill(_f64(w, "q"), _f64(w, "k"), _f64(w, "v"), w.intervals, return_probs=True)
    seg = O.segment_ids(w.intervals, w.total_tokens)
    T = w.total_tokens
    for t in range(T):
        for u in range(T):
            if u > t or seg[t] < 0 or seg[u] != seg[t]:
                assert (P[:, t, u] == 0.0).all()
    for t in range(T):
        row = P[:, t, :].sum(-1)
        if seg[t] >= 0:
            assert np.max(np.abs(row - 1.0)) < 1e-12
        else:
            assert (row == 0.0).all()


@pytest.mark.parametrize("seed", [31, 32])
def test_invariant_b_packed_equals_alone(seed):
    w = W.random_case(seed, [17, 3, 29, 1, 12], 6, 2, 16, "fp32", gaps=[0, 4, 1, 2, 0], tail=3,
                      order=[2, 0, 4, 1, 3])
    q, k, v = _f64(w, "q"), _f64(w, "k"), _f64(w, "v")
    packed = O.prefill(q, k, v, w.intervals)
    for s, e in w.intervals:
        alone = O.prefill(q[s:e], k[s:e], v[s:e], [(0, e - s)])
        assert np.max(np.abs(packed[s:e] - alone)) <= 1e-12
    # rows of tokens that belong to no question are zero
    seg = O.segment_ids(w.intervals, w.total_tokens)
    assert (packed[seg < 0] == 0).all()


def test_invariant_c_decode_equals_last_row_of_recompute():
    w = W.random_case(41, [5, 11, 8], 4, 2, 8, "fp32")
    q, k, v = _f64(w, "q"), _f64(w, "k"), _f64(w, "v")
    cap = 16
    pool_k = np.zeros((3, 2, cap, 8), np.float32)
    pool_v = np.zeros((3, 2, cap, 8), np.float32)
    pool_k, pool_v = O.slot_write(pool_k, pool_v, w.k, w.v, w.intervals, w.slot_ids)
    lens = w.lengths.copy()
    active = np.array([1, 0, 1], np.uint8)
    o, pk, pv = O.decode(w.q_new, w.k_new, w.v_new, pool_k, pool_v, w.slot_ids, lens, active, "fp32")
    assert np.isnan(o[1]).all()
    for i, (s, e) in enumerate(w.intervals):
        if not active[i]:
            continue
        qe = np.concatenate([q[s:e], _f64(w, "q_new")[i:i + 1]])
        ke = np.concatenate([k[s:e], _f64(w, "k_new")[i:i + 1]])
        ve = np.concatenate([v[s:e], _f64(w, "v_new")[i:i + 1]])
        full = O.prefill(qe, ke, ve, [(0, e - s + 1)])
        assert np.max(np.abs(o[i] - full[-1])) <= 1e-12
        assert np.array_equal(pk[w.slot_ids[i], :, e - s], w.k_new[i])
    # the dropped question's slot is untouched
    assert np.array_equal(pk[w.slot_ids[1]], pool_k[w.slot_ids[1]])


def _nested(a):
    return a.tolist()


def test_invariant_d_brute_force_tiny_fp32_config():
    w = W.tiny_fp32()
    q, k, v = _f64(w, "q"), _f64(w, "k"), _f64(w, "v")
    out = O.prefill(q, k, v, w.intervals)
    bf = np.array(brute.prefill(_nested(q), _nested(k), _nested(v), w.intervals.tolist(),
                                1.0 / math.sqrt(w.d)))
    assert np.max(np.abs(out - bf)) <= 1e-12


@pytest.mark.parametrize("seed", range(6))
def test_invariant_d_brute_force_random_tiny(seed):
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(1, 5))
    lengths = rng.integers(0, 9, size=n)
    h_kv = int(rng.integers(1, 3))
    G = int(rng.integers(1, 4))
    w = W.random_case(200 + seed, lengths, h_kv * G, h_kv, 4, "fp32",
                      gaps=rng.integers(0, 3, size=n), tail=int(rng.integers(0, 3)))
    if w.total_tokens == 0:
        return
    q, k, v = _f64(w, "q"), _f64(w, "k"), _f64(w, "v")
    out = O.prefill(q, k, v, w.intervals)
    bf = np.array(brute.prefill(_nested(q), _nested(k), _nested(v), w.intervals.tolist(), 0.5))
    assert np.max(np.abs(out - bf)) <= 1e-12
    rows = list(range(w.total_tokens))
    pr = O.prefill_rows(q, k, v, w.intervals, rows)
    assert np.max(np.abs(pr - out)) <= 1e-12


def test_brute_force_decode_one_matches_oracle_decode():
    rng = np.random.default_rng(5)
    pk = rng.standard_normal((2, 1, 8, 4)).astype(np.float32)
    pv = rng.standard_normal((2, 1, 8, 4)).astype(np.float32)
    qn = rng.standard_normal((1, 2, 4)).astype(np.float32)
    kn = rng.standard_normal((1, 1, 4)).astype(np.float32)
    vn = rng.standard_normal((1, 1, 4)).astype(np.float32)
    o, pk2, pv2 = O.decode(qn, kn, vn, pk, pv, [1], [5], [1], "fp32")
    kr = pk2[1, 0, :6].astype(np.float64).tolist()
    vr = pv2[1, 0, :6].astype(np.float64).tolist()
    for h in range(2):
        ref = brute.decode_one(qn[0, h].astype(np.float64).tolist(), kr, vr, 0.5)
        assert np.max(np.abs(np.array(ref) - o[0, h])) <= 1e-12


# ---------------------------------------------------------------------------
# a library routine: torch scaled-dot-product attention in float64
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("h_q,h_kv", [(4, 4), (8, 2), (7, 1)])
def test_single_question_matches_torch_sdpa(h_q, h_kv):
    rng = np.random.default_rng(h_q * 10 + h_kv)
    T, d = 23, 16
    q = rng.standard_normal((T, h_q, d))
    k = rng.standard_normal((T, h_kv, d))
    v = rng.standard_normal((T, h_kv, d))
    out = O.prefill(q, k, v, [(0, T)])
    tq = torch.from_numpy(q).permute(1, 0, 2)[None]
    tk = torch.from_numpy(k).permute(1, 0, 2)[None]
    tv = torch.from_numpy(v).permute(1, 0, 2)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True,
                                                          enable_gqa=(h_q != h_kv))
    ref = ref[0].permute(1, 0, 2).numpy()
    assert np.max(np.abs(out - ref)) < 1e-12


def test_packed_matches_torch_sdpa_with_block_mask():
    w = W.random_case(51, [7, 13, 5], 4, 2, 8, "fp32", gaps=[1, 0, 2])
    q, k, v = _f64(w, "q"), _f64(w, "k"), _f64(w, "v")
    out = O.prefill(q, k, v, w.intervals)
    for s, e in w.intervals:
        tq = torch.from_numpy(q[s:e]).permute(1, 0, 2)[None]
        tk = torch.from_numpy(k[s:e]).permute(1, 0, 2)[None]
        tv = torch.from_numpy(v[s:e]).permute(1, 0, 2)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True,
                                                              enable_gqa=True)
        assert np.max(np.abs(out[s:e] - ref[0].permute(1, 0, 2).numpy())) < 1e-12


# ---------------------------------------------------------------------------
# slot pool and validation
# ---------------------------------------------------------------------------

def test_slot_write_is_bit_copy_and_keeps_sentinels():
    w = W.random_case(61, [3, 0, 5], 2, 2, 8, "bf16", n_slots=5, permute_slots=True, cap=6)
    sent = np.uint16(0x7FC1)
    pk = np.full((5, 2, 6, 8), sent, np.uint16)
    pv = np.full((5, 2, 6, 8), sent, np.uint16)
    nk, nv = O.slot_write(pk, pv, w.k, w.v, w.intervals, w.slot_ids)
    for (s, e), slot in zip(w.intervals, w.slot_ids):
        n = e - s
        assert np.array_equal(nk[slot, :, :n], np.swapaxes(w.k[s:e], 0, 1))
        assert np.array_equal(nv[slot, :, :n], np.swapaxes(w.v[s:e], 0, 1))
        assert (nk[slot, :, n:] == sent).all() and (nv[slot, :, n:] == sent).all()
    unused = sorted(set(range(5)) - set(int(x) for x, (s, e) in zip(w.slot_ids, w.intervals) if e > s))
    for slot in unused:
        assert (nk[slot] == sent).all()


def test_validate_prefill_cases():
    V = O.validate_prefill
    assert V([(0, 3), (3, 5)], 5) is None
    assert V([(0, 3), (2, 5)], 5) == O.INTERVALS          # overlap
    assert V([(0, 6)], 5) == O.INTERVALS                   # past T
    assert V([(3, 2)], 5) == O.INTERVALS                   # reversed
    assert V([(-1, 2)], 5) == O.INTERVALS
    assert V([(2, 2), (0, 5)], 5) is None                  # empty interval overlaps nothing
    assert V([(0, 3), (3, 5)], 5, [0, 2], 2, 4) == O.SLOT  # slot out of range
    assert V([(0, 3), (3, 5)], 5, [1, 1], 2, 4) == O.SLOT  # shared slot
    assert V([(0, 3), (3, 3)], 5, [1, 1], 2, 4) is None    # empty question's slot may repeat
    assert V([(0, 5)], 5, [0], 1, 4) == O.SLOT_OVERFLOW    # L > cap
    assert V([(0, 4)], 5, [0], 1, 4) is None               # L == cap fits exactly


def test_validate_decode_cases():
    V = O.validate_decode
    assert V([0, 1], [3, 3], [1, 1], 2, 4) is None
    assert V([0, 1], [4, 3], [1, 1], 2, 4) == O.SLOT_OVERFLOW   # no room for the new row
    assert V([0, 1], [4, 3], [0, 1], 2, 4) is None              # dropped question not checked
    assert V([1, 1], [1, 1], [1, 1], 2, 4) == O.SLOT
    assert V([1, 1], [1, 1], [1, 0], 2, 4) is None
    assert V([0, 5], [1, 1], [1, 1], 2, 4) == O.SLOT
    assert V([0, 1], [0, 0], [0, 0], 2, 4) is None              # every question dropped


def test_config_realisations():
    """The seeded procedure gives the workloads quoted in the design notes."""
    w2 = W.qwen25_7b_prefill()
    assert w2.lengths.tolist() == [1757, 725, 451, 791, 997, 1715, 1065, 420]
    assert w2.total_tokens == 7921
    rng = np.random.default_rng(3)
    L3 = np.clip(np.rint(np.exp(rng.normal(np.log(512.0), 0.8, size=32))), 1, 4096)
    assert int(L3.sum()) == 24100 and int(L3.max()) == 4096 and int(L3.min()) == 66
    s = W.stress()
    assert s.prefill.total_tokens == 19483
    assert int((s.n_decoded > 0).sum()) == 256 and int(s.n_decoded.max()) == 116


# ---------------------------------------------------------------------------
# planted mistakes: each must be caught by a pin above
# ---------------------------------------------------------------------------

def _pins_pass(prefill_fn):
    """Re-run a representative subset of the pins against a replacement prefill."""
    ok = []
    g = _golden("online_softmax_worked_example.txt")
    k = np.array(g["k"]).reshape(4, 1, 1)
    v = np.array(g["v"]).reshape(4, 1, 1)
    q = np.ones((4, 1, 1))
    ok.append(round(float(prefill_fn(q, k, v, [(0, 4)], 1.0)[3, 0, 0]), 6) == g["output"][0])
    w = W.random_case(31, [17, 3, 29, 1, 12], 6, 2, 16, "fp32", gaps=[0, 4, 1, 2, 0], tail=3)
    qq, kk, vv = _f64(w, "q"), _f64(w, "k"), _f64(w, "v")
    packed = prefill_fn(qq, kk, vv, w.intervals, None)
    good = True
    for s, e in w.intervals:
        alone = prefill_fn(qq[s:e], kk[s:e], vv[s:e], [(0, e - s)], None)
        good &= bool(np.max(np.abs(packed[s:e] - alone)) <= 1e-12)
    ok.append(good)
    bf = np.array(brute.prefill(_nested(qq), _nested(kk), _nested(vv), w.intervals.tolist(), 0.25))
    ok.append(bool(np.max(np.abs(packed - bf)) <= 1e-12))
    return all(ok)


def test_planted_mistakes_are_caught(monkeypatch):
    assert _pins_pass(lambda q, k, v, iv, sc: O.prefill(q, k, v, iv, scale=sc))

    def future_mask(intervals, T):          # causal direction reversed
        return np.triu(np.ones((T, T), bool)) & _iso(intervals, T)

    def no_isolation(intervals, T):          # isolation dropped
        return np.tril(np.ones((T, T), bool)) & (O.segment_ids(intervals, T)[:, None] >= 0)

    def _iso(intervals, T):
        m = np.zeros((T, T), bool)
        for s, e in intervals:
            m[s:e, s:e] = True
        return m

    for bad in (future_mask, no_isolation):
        monkeypatch.setattr(O, "allowed_mask", bad)
        assert not _pins_pass(lambda q, k, v, iv, sc: O.prefill(q, k, v, iv, scale=sc))
        monkeypatch.undo()

    def wrong_gqa(q, k, v, iv, sc):          # h % H_kv instead of h // G
        kk = np.tile(k, (1, q.shape[1] // k.shape[1], 1))
        vv = np.tile(v, (1, q.shape[1] // v.shape[1], 1))
        return O.prefill(q, kk, vv, iv, scale=sc)
    assert not _pins_pass(wrong_gqa)

    # the 1/sqrt(d_h) factor dropped when no scale is given
    assert not _pins_pass(lambda q, k, v, iv, sc: O.prefill(q, k, v, iv, scale=sc or 1.0))

    plain_softmax = O.softmax_rows

    def transposed_pv(scores):               # weights normalised over the wrong axis
        return plain_softmax(scores.T).T
    monkeypatch.setattr(O, "softmax_rows", transposed_pv)
    assert not _pins_pass(lambda q, k, v, iv, sc: O.prefill(q, k, v, iv, scale=sc))


# ---------------------------------------------------------------------------
# rotary position encoding with per-question positions (KV-cache isolation
# article, hnwysp.cn, §7.2)
# ---------------------------------------------------------------------------

def _rope_case(seed, P=5, H=3, d=8):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((P, H, d)), rng.integers(0, 3000, P)


def test_rope_is_the_complex_rotation():
    """Pair (x_j, x_{j+d/2}) as the complex number x_j + i x_{j+d/2}: RoPE multiplies it by
    exp(i p w_j).  Complex arithmetic, not the oracle's real-valued formula."""
    x, pos = _rope_case(1)
    d = x.shape[-1]
    theta = 10000.0
    z = x[..., :d // 2] + 1j * x[..., d // 2:]
    w = np.exp(-np.log(theta) * np.arange(d // 2) * 2.0 / d)
    zr = z * np.exp(1j * pos[:, None, None] * w[None, None, :])
    want = np.concatenate([zr.real, zr.imag], axis=-1)
    np.testing.assert_allclose(O.rope_rotate(x, pos, theta), want, rtol=0, atol=1e-12)


def test_rope_brute_force_scalar_loops():
    x, pos = _rope_case(2, P=4, H=2, d=16)
    pos[1] = -1  # a token in no question: unchanged
    want = np.array(brute.rope_rows(x.tolist(), pos.tolist(), 1e6))
    np.testing.assert_allclose(O.rope_rotate(x, pos, 1e6), want, rtol=0, atol=1e-12)


def test_rope_closed_forms():
    d, theta = 128, 1e6
    w = O.rope_freqs(d, theta)
    assert w[0] == 1.0 and len(w) == d // 2
    assert math.isclose(w[-1], theta ** (-(d - 2) / d), rel_tol=1e-14)
    np.testing.assert_allclose(w[1:] / w[:-1], theta ** (-2.0 / d), rtol=1e-13)
    x, _ = _rope_case(3)
    np.testing.assert_array_equal(O.rope_rotate(x, np.zeros(len(x), int), theta), x)  # position 0: identity
    np.testing.assert_array_equal(O.rope_rotate(x, -np.ones(len(x), int), theta), x)  # no question: unchanged
    y = O.rope_rotate(x, np.arange(len(x)) * 977, theta)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)


def test_rope_scores_depend_on_the_position_difference_only():
    rng = np.random.default_rng(4)
    q, k = rng.standard_normal((1, 2, 64)), rng.standard_normal((1, 2, 64))
    for p1, p2, shift in [(5, 3, 100), (0, 0, 2457), (1000, 17, 3)]:
        a = (O.rope_rotate(q, [p1], 1e6) * O.rope_rotate(k, [p2], 1e6)).sum(-1)
        b = (O.rope_rotate(q, [p1 + shift], 1e6) * O.rope_rotate(k, [p2 + shift], 1e6)).sum(-1)
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-11)


def test_rope_positions_restart_in_every_question():
    iv = np.array([[5, 8], [0, 3], [10, 10], [11, 13]])  # unsorted, an empty one, gaps at 3, 4, 8, 9, 10
    pos = O.prefill_positions(iv, 14)
    assert pos.tolist() == [0, 1, 2, -1, -1, 0, 1, 2, -1, -1, -1, 0, 1, -1]


def test_rope_packed_equals_alone_and_the_cache_needs_per_question_positions():
    """Invariant (b) with RoPE: with positions counted per question, each question's output rows
    and rotated K rows in the packed batch equal those of the question run alone.  Positions
    counted over the packed sequence shift a question's positions by a constant: its attention
    output stays the same (scores see position differences only), but the K it would cache is
    rotated differently from the K it caches alone, so a later decode at position lens (the cache
    length) would no longer match -- the reason positions restart in every question."""
    rng = np.random.default_rng(5)
    lengths, h_q, h_kv, d, theta = [6, 9, 4], 4, 2, 16, 1e4
    iv = W.pack_intervals(lengths, gaps=[1, 0, 2])
    T = int(iv[-1, 1])
    q, k, v = (rng.standard_normal((T, h, d)) for h in (h_q, h_kv, h_kv))
    out, _, k_rot = O.prefill_rope(q, k, v, iv, theta)
    k_glob = O.rope_rotate(k, np.arange(T), theta)
    out_glob = O.prefill(O.rope_rotate(q, np.arange(T), theta), k_glob, v, iv)
    for s, e in iv:
        alone, _, k_alone = O.prefill_rope(q[s:e], k[s:e], v[s:e], np.array([[0, e - s]]), theta)
        np.testing.assert_allclose(out[s:e], alone, rtol=0, atol=1e-12)
        np.testing.assert_allclose(k_rot[s:e], k_alone, rtol=0, atol=1e-12)
        np.testing.assert_allclose(out_glob[s:e], alone, rtol=0, atol=1e-9)
        if s > 0:
            assert np.abs(k_glob[s:e] - k_alone).max() > 1e-3
    seg = O.segment_ids(iv, T)
    assert (out[seg < 0] == 0).all()
    np.testing.assert_array_equal(k_rot[seg < 0], k[seg < 0])


def test_rope_decode_with_rotated_cache_equals_last_row_of_recompute():
    """Invariant (c) with RoPE: the cache holds K rotated at its own positions 0..n-1, the new
    token is rotated at position n = lens (the cache length), and the decode output equals the
    last row of the full recompute with RoPE."""
    rng = np.random.default_rng(6)
    n, h_q, h_kv, d, cap, theta = 11, 4, 2, 16, 16, 1e6
    q, k, v = (rng.standard_normal((n + 1, h, d)) for h in (h_q, h_kv, h_kv))
    full, _, k_rot = O.prefill_rope(q, k, v, np.array([[0, n + 1]]), theta)
    pool_k = np.zeros((1, h_kv, cap, d))
    pool_v = np.zeros((1, h_kv, cap, d))
    pool_k[0, :, :n] = np.swapaxes(k_rot[:n], 0, 1)
    pool_v[0, :, :n] = np.swapaxes(v[:n], 0, 1)
    q_new = O.rope_rotate(q[n:], [n], theta)
    k_new = O.rope_rotate(k[n:], [n], theta)
    o, pk, _ = O.decode(q_new, k_new, v[n:], pool_k, pool_v, [0], [n], [1], "fp64")
    np.testing.assert_allclose(o[0], full[n], rtol=0, atol=1e-12)
    np.testing.assert_allclose(pk[0, :, n], k_rot[n], rtol=0, atol=1e-12)


def test_round_to_stored_is_one_rounding_to_nearest_even():
    one = 1.0
    ulp = 2.0 ** -7  # bf16 spacing in [1, 2)
    xs = np.array([one + ulp / 2, one + 1.5 * ulp, one + ulp / 2 + 2.0 ** -40, -(one + 1.5 * ulp), 0.0])
    got = W.bf16_bits_to_f32(O.round_to_stored(xs, "bf16")).astype(np.float64)
    assert got.tolist() == [1.0, 1.0 + 2 * ulp, 1.0 + ulp, -(1.0 + 2 * ulp), 0.0]
    # values a float32 holds exactly are rounded once either way
    x32 = np.random.default_rng(7).standard_normal(1000).astype(np.float32)
    np.testing.assert_array_equal(O.round_to_stored(x32.astype(np.float64), "bf16"), W.f32_to_bf16_bits(x32))


def test_rope_planted_mistakes_are_caught(monkeypatch):
    """Each plausible RoPE mistake -- the frequency exponent -j/d instead of -2j/d, the rotation
    turned the other way, adjacent (interleaved) pairs instead of (j, j + d/2) -- disagrees with
    the scalar-loop brute force the oracle is pinned to."""
    x, pos = _rope_case(8, P=3, H=2, d=8)
    theta = 1e4
    ref = np.array(brute.rope_rows(x.tolist(), pos.tolist(), theta))

    def agrees(y):
        return np.allclose(y, ref, rtol=0, atol=1e-12)

    assert agrees(O.rope_rotate(x, pos, theta))
    good = O.rope_freqs
    monkeypatch.setattr(O, "rope_freqs", lambda d, th: good(2 * d, th)[: d // 2])
    assert not agrees(O.rope_rotate(x, pos, theta))
    monkeypatch.undo()
    assert not agrees(O.rope_rotate(x, -pos, theta))  # turned the other way
    perm = np.arange(8).reshape(4, 2).T.reshape(-1)    # (0, 1), (2, 3), ... as the pairs
    inter = O.rope_rotate(x[..., perm], pos, theta)[..., np.argsort(perm)]
    assert not agrees(inter)


# ---------------------------------------------------------------------------
# paged slot pool (inference-engine notes, sakurs2.com, §2.5; Kev pipeline
# article, gsyq.cn, §4.3)
# ---------------------------------------------------------------------------

def _paged_case(seed, lengths, h_kv=2, d=8, page=O.PAGE, extra=0):
    """Random block tables: every question gets blocks for its length + ``extra`` positions."""
    rng = np.random.default_rng(seed)
    iv = W.pack_intervals(lengths, gaps=[1] * len(lengths))
    T = int(iv[-1, 1])
    k = rng.standard_normal((T, h_kv, d))
    v = rng.standard_normal((T, h_kv, d))
    need = [(L + extra + page - 1) // page for L in lengths]
    mb = max(need + [1]) + 1
    n_blocks = sum(need) + 5
    perm = rng.permutation(n_blocks)
    table = np.full((len(lengths), mb), -1, np.int64)
    at = 0
    for i, m in enumerate(need):
        table[i, :m] = perm[at:at + m]
        at += m
    return iv, k, v, table, n_blocks, mb


def test_paged_write_then_gather_equals_the_contiguous_slot():
    lengths = [300, 129, 1, 0, 256]
    iv, k, v, table, n_blocks, mb = _paged_case(1, lengths)
    pool = np.full((n_blocks, 2, O.PAGE, 8), -7.0)
    pk, pv = O.paged_slot_write(pool, pool, k, v, iv, table)
    ck, cv = O.slot_write(np.zeros((len(lengths), 2, 512, 8)), np.zeros((len(lengths), 2, 512, 8)), k, v, iv,
                          np.arange(len(lengths)))
    for i, L in enumerate(lengths):
        np.testing.assert_array_equal(O.paged_gather(pk, table[i], L), ck[i, :, :L])
        np.testing.assert_array_equal(O.paged_gather(pv, table[i], L), cv[i, :, :L])
    used = {int(b) for i, L in enumerate(lengths) for b in table[i, :(L + 127) // 128]}
    for b in set(range(n_blocks)) - used:  # blocks no question uses keep their contents
        assert (pk[b] == -7.0).all() and (pv[b] == -7.0).all()


def test_paged_identity_table_is_the_contiguous_layout_reshaped():
    """With block i * mb + b for block b of question i, the paged pool [n * mb, H, page, d] holds
    exactly the contiguous pool [n, H, mb * page, d] split along positions."""
    lengths = [200, 77, 300]
    iv, k, v, _, _, mb = _paged_case(2, lengths)
    n = len(lengths)
    table = np.arange(n * mb).reshape(n, mb)
    pk, _ = O.paged_slot_write(np.zeros((n * mb, 2, O.PAGE, 8)), np.zeros((n * mb, 2, O.PAGE, 8)), k, v, iv, table)
    ck, _ = O.slot_write(np.zeros((n, 2, mb * O.PAGE, 8)), np.zeros((n, 2, mb * O.PAGE, 8)), k, v, iv, np.arange(n))
    as_contig = pk.reshape(n, mb, 2, O.PAGE, 8).transpose(0, 2, 1, 3, 4).reshape(n, 2, mb * O.PAGE, 8)
    np.testing.assert_array_equal(as_contig, ck)


def test_paged_decode_equals_contiguous_decode():
    rng = np.random.default_rng(3)
    lengths = [300, 129, 7, 0, 255]
    h_q, h_kv, d = 4, 2, 8
    iv, k, v, table, n_blocks, mb = _paged_case(3, lengths, h_kv, d, extra=1)  # room for the new row
    N = len(lengths)
    pk, pv = O.paged_slot_write(np.zeros((n_blocks, h_kv, O.PAGE, d)), np.zeros((n_blocks, h_kv, O.PAGE, d)), k, v,
                                iv, table)
    cap = mb * O.PAGE
    ck, cv = O.slot_write(np.zeros((N, h_kv, cap, d)), np.zeros((N, h_kv, cap, d)), k, v, iv, np.arange(N))
    q_new, k_new, v_new = (rng.standard_normal((N, h, d)) for h in (h_q, h_kv, h_kv))
    lens = np.array(lengths)
    active = np.array([1, 0, 1, 1, 1])
    assert O.validate_paged(lens + 1, table, n_blocks, live=active) is None
    o_p, pk2, _ = O.decode_paged(q_new, k_new, v_new, pk, pv, table, lens, active, "fp64")
    o_c, ck2, _ = O.decode(q_new, k_new, v_new, ck, cv, np.arange(N), lens, active, "fp64")
    np.testing.assert_array_equal(np.isnan(o_p), np.isnan(o_c))
    live = active.astype(bool)
    np.testing.assert_allclose(o_p[live], o_c[live], rtol=0, atol=1e-12)
    for i in np.nonzero(live)[0]:
        np.testing.assert_array_equal(O.paged_gather(pk2, table[i], lens[i] + 1), ck2[i, :, :lens[i] + 1])


def test_validate_paged_cases():
    table = np.array([[3, 4, -1], [5, -1, -1], [0, 1, 2]])
    assert O.validate_paged([200, 100, 300], table, 6) is None
    assert O.validate_paged([257, 100, 300], table, 6) == O.SLOT  # a third block: -1
    assert O.validate_paged([200, 100, 385], table, 6) == O.SLOT_OVERFLOW  # 4 blocks, rows hold 3
    assert O.validate_paged([200, 100, 300], table, 5) == O.SLOT  # block 5 out of range
    dup = np.array([[3, 4, -1], [4, -1, -1], [0, 1, 2]])
    assert O.validate_paged([200, 100, 300], dup, 6) == O.SLOT  # block 4 shared
    assert O.validate_paged([200, 100, 300], dup, 6, live=[1, 0, 1]) is None  # the sharer is dropped
    same = np.array([[3, 3, -1]])
    assert O.validate_paged([200], same, 6) == O.SLOT  # twice in one question
    assert O.validate_paged([0, 0], np.full((2, 1), -1), 1) is None  # empty questions use no block


def test_assign_blocks_contiguous_first_example_and_invariants():
    free = np.array([1, 1, 0, 1, 1, 1, 0, 1], bool)
    table, fr = O.assign_blocks([2, 2, 2], free, 3)
    assert table.tolist() == [[0, 1, -1], [3, 4, -1], [5, 7, -1]]  # the last one has no run of 2 left
    assert fr.tolist() == [False] * 8
    table, _ = O.assign_blocks([2, 2, 2], free, 3, contiguous_first=False)
    assert table.tolist() == [[0, 1, -1], [3, 4, -1], [5, 7, -1]]
    table, _ = O.assign_blocks([1, 3], free, 3)
    assert table.tolist() == [[0, -1, -1], [3, 4, 5]]  # lowest run of 3, not blocks 1, 3, 4
    table, _ = O.assign_blocks([1, 3], free, 3, contiguous_first=False)
    assert table.tolist() == [[0, -1, -1], [1, 3, 4]]
    assert O.assign_blocks([3, 4], free, 4) is None  # 6 free blocks for 7
    assert O.assign_blocks([4], free, 3) is None     # a row holds 3
    rng = np.random.default_rng(4)
    for _ in range(20):
        free = rng.random(64) < 0.7
        need = rng.integers(0, 5, 6)
        res = O.assign_blocks(need, free, 5)
        if res is None:
            assert need.sum() > free.sum()
            continue
        table, fr = res
        used = [int(b) for i, m in enumerate(need) for b in table[i, :m]]
        assert len(set(used)) == len(used) and all(free[b] for b in used)
        assert (table[np.arange(5)[None, :] >= need[:, None]] == -1).all()
        assert sorted(np.nonzero(free & ~fr)[0].tolist()) == sorted(used)
        assert O.validate_paged(need * O.PAGE, table, 64) is None


# ---------------------------------------------------------------------------
# chunked prefill into slots (inference-engine notes, sakurs2.com, §2.6)
# ---------------------------------------------------------------------------

def _chunk_case(seed, lengths, h_q=4, h_kv=2, d=8):
    rng = np.random.default_rng(seed)
    iv = W.pack_intervals(lengths, gaps=[1] * len(lengths))
    T = int(iv[-1, 1])
    q, k, v = (rng.standard_normal((T, h, d)) for h in (h_q, h_kv, h_kv))
    return iv, q, k, v


def test_chunk_with_empty_prefixes_is_the_plain_prefill():
    lengths = [30, 17, 0, 45]
    iv, q, k, v = _chunk_case(1, lengths)
    n, cap = len(lengths), 64
    pool = np.full((n + 1, 2, cap, 8), -3.0)
    slots = np.array([2, 0, 4, 1])
    out, pk, pv = O.prefill_chunk(q, k, v, iv, np.zeros(n, int), slots, pool, pool, "fp64")
    np.testing.assert_allclose(out, O.prefill(q, k, v, iv), rtol=0, atol=1e-12)
    ek, ev = O.slot_write(pool, pool, k, v, iv, slots)
    np.testing.assert_array_equal(pk, ek)
    np.testing.assert_array_equal(pv, ev)


@pytest.mark.parametrize("split", [1, 7, 20, 29])
def test_chunks_in_sequence_equal_one_prefill(split):
    """A question prefilled as chunk [0, split) then chunk [split, L) with prefix = split gives the
    one-shot prefill's rows and the same slot contents."""
    L = 30
    iv, q, k, v = _chunk_case(2, [L])
    s = int(iv[0, 0])
    full = O.prefill(q, k, v, iv)
    pool = np.zeros((1, 2, 40, 8))
    a_iv = np.array([[s, s + split]])
    out1, pk, pv = O.prefill_chunk(q, k, v, a_iv, [0], [0], pool, pool, "fp64")
    b_iv = np.array([[s + split, s + L]])
    out2, pk, pv = O.prefill_chunk(q, k, v, b_iv, [split], [0], pk, pv, "fp64")
    np.testing.assert_allclose(out1[s:s + split], full[s:s + split], rtol=0, atol=1e-12)
    np.testing.assert_allclose(out2[s + split:s + L], full[s + split:s + L], rtol=0, atol=1e-12)
    ek, ev = O.slot_write(pool, pool, k, v, iv, [0])
    np.testing.assert_array_equal(pk, ek)
    np.testing.assert_array_equal(pv, ev)


def test_one_token_chunk_is_a_decode_step():
    rng = np.random.default_rng(3)
    n, h_q, h_kv, d, cap = 3, 4, 2, 8, 32
    pool_k = rng.standard_normal((n, h_kv, cap, d))
    pool_v = rng.standard_normal((n, h_kv, cap, d))
    prefix = np.array([5, 0, 17])
    q, k, v = (rng.standard_normal((n, h, d)) for h in (h_q, h_kv, h_kv))
    iv = np.array([[0, 1], [1, 2], [2, 3]])
    slots = np.array([1, 2, 0])
    out, pk, pv = O.prefill_chunk(q, k, v, iv, prefix, slots, pool_k, pool_v, "fp64")
    o, dk, dv = O.decode(q, k, v, pool_k, pool_v, slots, prefix, np.ones(n), "fp64")
    np.testing.assert_allclose(out, o, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(pk, dk)
    np.testing.assert_array_equal(pv, dv)


def test_validate_chunk_cases():
    iv = np.array([[0, 100], [100, 100], [105, 300]])
    ok = dict(total_tokens=300, slot_ids=[0, 1, 2], n_slots=3, cap=512)
    assert O.validate_chunk(iv, prefix_lens=[0, 0, 256], **ok) is None
    assert O.validate_chunk(iv, prefix_lens=[0, 0, 100], **ok) == O.PREFIX       # not on a tile boundary
    assert O.validate_chunk(iv, prefix_lens=[-128, 0, 0], **ok) == O.PREFIX
    assert O.validate_chunk(iv, prefix_lens=[0, 0, 384], **ok) == O.SLOT_OVERFLOW  # 384 + 195 > 512
    assert O.validate_chunk(iv, prefix_lens=[0, 0, 0], total_tokens=300, slot_ids=[0, 0, 2], n_slots=3,
                            cap=512) is None  # the empty chunk's slot is not used
    assert O.validate_chunk(iv, prefix_lens=[0, 0, 0], total_tokens=300, slot_ids=[2, 1, 2], n_slots=3,
                            cap=512) == O.SLOT
    assert O.validate_chunk(iv, prefix_lens=[0, 0, 0], total_tokens=300, slot_ids=[0, 1, 3], n_slots=3,
                            cap=512) == O.SLOT
    assert O.validate_chunk(np.array([[0, 100], [50, 120]]), 300, prefix_lens=[0, 0], slot_ids=[0, 1], n_slots=3,
                            cap=512) == O.INTERVALS


# ---------------------------------------------------------------------------
# per-question temperature sampling (Kev architecture article, icman.com.cn, §4.1)
# ---------------------------------------------------------------------------

def test_sampling_closed_form_two_tokens():
    # logits (0, ln 3) at T = 1: p = (1/4, 3/4); at T = 2: p = (1, sqrt 3) / (1 + sqrt 3)
    lg = np.array([[0.0, np.log(3.0)]] * 4)
    got = O.sample_tokens(lg, [1.0, 1.0, 2.0, 2.0], [0.2499, 0.2501, 0.366, 0.367])
    assert got.tolist() == [0, 1, 0, 1]  # 1 / (1 + sqrt 3) = 0.36603


def test_sampling_frequencies_over_a_uniform_grid_are_the_probabilities():
    """Inverse CDF: the share of a fine grid of u in [0, 1) that picks token k is p_k (up to the grid step)."""
    rng = np.random.default_rng(1)
    lg = rng.standard_normal(7) * 2
    for T in (0.5, 1.0, 3.0):
        grid = (np.arange(20000) + 0.5) / 20000
        toks = O.sample_tokens(np.tile(lg, (len(grid), 1)), np.full(len(grid), T), grid)
        freq = np.bincount(toks, minlength=7) / len(grid)
        p = np.exp(lg / T) / np.exp(lg / T).sum()  # the plain softmax, not the oracle's stable form
        np.testing.assert_allclose(freq, p, atol=1.0 / 20000 + 1e-12)


def test_sampling_greedy_ties_and_temperature_identity():
    lg = np.array([[1.0, 5.0, 5.0, 2.0], [0.0, 0.0, 0.0, 0.0]])
    assert O.sample_tokens(lg, [0.0, 0.0], [0.9, 0.9]).tolist() == [1, 0]  # lowest index among maxima
    rng = np.random.default_rng(2)
    x = rng.standard_normal((6, 50))
    T = np.array([0.3, 0.7, 1.0, 1.5, 2.0, 4.0])
    u = rng.random(6)
    # sampling x at temperature T is sampling x / T at temperature 1
    assert O.sample_tokens(x, T, u).tolist() == O.sample_tokens(x / T[:, None], np.ones(6), u).tolist()
    # dropped questions: -1
    assert O.sample_tokens(x, T, u, active=[1, 0, 1, 0, 1, 0]).tolist()[1::2] == [-1, -1, -1]


def test_validate_sampling_cases():
    assert O.validate_sampling([0.0, 1.0], [0.0, 0.999]) is None
    assert O.validate_sampling([-1.0, 1.0], [0.5, 0.5]) == O.SAMPLING
    assert O.validate_sampling([np.inf, 1.0], [0.5, 0.5]) == O.SAMPLING
    assert O.validate_sampling([1.0, 1.0], [1.0, 0.5]) == O.SAMPLING
    assert O.validate_sampling([1.0, 1.0], [np.nan, 0.5]) == O.SAMPLING
    assert O.validate_sampling([1.0, -1.0], [0.5, 0.5], active=[1, 0]) is None


# ---------------------------------------------------------------------------
# token-grouped LoRA (Kev architecture article, icman.com.cn, §3.2, §3.3)
# ---------------------------------------------------------------------------

def _lora_case(seed, lengths, d_in=24, d_out=20, r=4, n_ad=3):
    rng = np.random.default_rng(seed)
    iv = W.pack_intervals(lengths, gaps=[1] * len(lengths))
    T = int(iv[-1, 1]) + 2
    x = rng.standard_normal((T, d_in))
    y = rng.standard_normal((T, d_out))
    A = rng.standard_normal((n_ad, r, d_in))
    B = rng.standard_normal((n_ad, d_out, r))
    scales = rng.random(n_ad) + 0.5
    return iv, x, y, A, B, scales


def test_lora_grouped_equals_the_routed_form():
    iv, x, y, A, B, sc = _lora_case(1, [5, 9, 0, 7, 3])
    ids = np.array([2, -1, 0, 0, 1])  # two questions share adapter 0, one has none
    np.testing.assert_allclose(O.lora_apply(y, x, iv, ids, A, B, sc), O.lora_router(y, x, iv, ids, A, B, sc),
                               rtol=0, atol=1e-12)


def test_lora_is_the_merged_weight_and_leaves_other_rows():
    """For a question with adapter a, base output x W^T plus the delta is x (W + s B A)^T (the
    article's merged alternative); rows without an adapter, and gap rows, keep the base output."""
    iv, x, _, A, B, sc = _lora_case(2, [6, 4])
    Wb = np.random.default_rng(3).standard_normal((20, 24))
    y0 = x @ Wb.T
    got = O.lora_apply(y0, x, iv, [1, -1], A, B, sc)
    s0, e0 = iv[0]
    np.testing.assert_allclose(got[s0:e0], x[s0:e0] @ (Wb + sc[1] * B[1] @ A[1]).T, rtol=0, atol=1e-11)
    mask = np.ones(len(x), bool)
    mask[s0:e0] = False
    np.testing.assert_array_equal(got[mask], y0[mask])


def test_validate_lora_cases():
    assert O.validate_lora([-1, 0, 2], 3) is None
    assert O.validate_lora([-2, 0], 3) == O.ADAPTER
    assert O.validate_lora([0, 3], 3) == O.ADAPTER
