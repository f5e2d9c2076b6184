"""GPU parity of the paged slot pool (block tables) against the CPU oracle: prefill with the
paged write, the paged write alone, decode over a paged pool (including bitwise equality with
the contiguous decode of the same logical cache), and the table errors that must write
nothing."""
import numpy as np
import pytest
import torch

import packed_question_isolated_gb300 as kev
import workloads as W
from oracle import kev_oracle as O

from kev_harness import PrefillRun, compare, dev, f64, host, shape_of, tdtype

pytestmark = pytest.mark.gpu

PAGE = O.PAGE


def _scattered_tables(rng, need, n_blocks, max_blocks, contiguous_first=False):
    """Tables from the library's host assignment over a random free map (scattered blocks)."""
    free = (rng.random(n_blocks) < 0.8).astype(np.uint8)
    short = int(np.sum(need)) - int(free.sum())
    if short > 0:  # free some more, still scattered
        free[rng.permutation(np.nonzero(free == 0)[0])[:short]] = 1
    table = kev.kev_assign_blocks(need, free, max_blocks, contiguous_first=contiguous_first)
    assert table is not None
    return table


def _itensor(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


CASES = [
    # lengths, h_q, h_kv, d, dtype, gaps, tail
    ([300, 129, 1, 0, 517], 8, 2, 128, "bf16", [0, 3, 0, 5, 1], 7),
    ([200, 77, 640], 7, 1, 128, "bf16", [2, 0, 1], 3),
    ([65, 190, 3, 129], 8, 2, 64, "bf16", [1, 1, 1, 1], 1),
    ([40, 7, 130], 4, 2, 64, "fp32", [0, 2, 1], 2),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_prefill_attn_paged_full_parity(case):
    lengths, h_q, h_kv, d, dtype, gaps, tail = CASES[case]
    w = W.random_case(600 + case, lengths, h_q, h_kv, d, dtype, gaps=gaps, tail=tail)
    rng = np.random.default_rng(601 + case)
    need = [(L + PAGE - 1) // PAGE for L in lengths]
    max_blocks, n_blocks = max(need) + 1, 3 * sum(need) + 4
    table = _scattered_tables(rng, need, n_blocks, max_blocks)
    assert O.validate_paged(lengths, table, n_blocks) is None
    run = PrefillRun(w, slots=False)
    td = tdtype(dtype)
    pk = torch.full((n_blocks, h_kv, PAGE, d), -7.0, dtype=td, device="cuda")
    pv = torch.full((n_blocks, h_kv, PAGE, d), -9.0, dtype=td, device="cuda")
    pk0, pv0 = host(pk), host(pv)
    kev.kev_prefill_attn_paged(run.q, run.k, run.v, w.total_tokens, run.intervals, run.n_questions, _itensor(table),
                               max_blocks, pk, pv, n_blocks, run.out, shape_of(w), run.ws, run.ws_bytes, run.status)
    assert run.device_status() == 0
    T = w.total_tokens
    ref = O.prefill(W.to_float64(w.q, dtype), W.to_float64(w.k, dtype), W.to_float64(w.v, dtype), w.intervals,
                    scale=w.scale or None)
    got = f64(run.out, dtype)[:T]
    compare(got, ref, dtype, f"paged case {case}")
    assert (got[O.segment_ids(w.intervals, T) < 0] == 0).all()
    ek, ev = O.paged_slot_write(pk0, pv0, w.k, w.v, w.intervals, table)
    np.testing.assert_array_equal(host(pk), ek)
    np.testing.assert_array_equal(host(pv), ev)


def test_kv_write_paged_alone_is_a_bit_copy():
    lengths = [129, 128, 1, 300]
    w = W.random_case(610, lengths, 4, 2, 128, "bf16", gaps=[1, 0, 2, 0], tail=3)
    rng = np.random.default_rng(611)
    need = [(L + PAGE - 1) // PAGE for L in lengths]
    max_blocks, n_blocks = 4, 16
    table = _scattered_tables(rng, need, n_blocks, max_blocks, contiguous_first=True)
    run = PrefillRun(w, slots=False)
    pk = torch.full((n_blocks, 2, PAGE, 128), -7.0, dtype=torch.bfloat16, device="cuda")
    pv = torch.full((n_blocks, 2, PAGE, 128), -9.0, dtype=torch.bfloat16, device="cuda")
    pk0, pv0 = host(pk), host(pv)
    kev.kev_kv_write_paged(run.k, run.v, w.total_tokens, run.intervals, run.n_questions, _itensor(table), max_blocks,
                           pk, pv, n_blocks, shape_of(w), run.ws, run.ws_bytes, run.status)
    assert run.device_status() == 0
    ek, ev = O.paged_slot_write(pk0, pv0, w.k, w.v, w.intervals, table)
    np.testing.assert_array_equal(host(pk), ek)
    np.testing.assert_array_equal(host(pv), ev)


def _paged_decode_case(seed, lens, active, h_q, h_kv, extra_blocks=8, contiguous_first=False):
    rng = np.random.default_rng(seed)
    d = 128
    lens = np.asarray(lens, np.int32)
    N = len(lens)
    need = [(int(n) + 1 + PAGE - 1) // PAGE for n in lens]  # room for the new row
    max_blocks = max(need) + 1
    n_blocks = sum(need) + extra_blocks
    table = _scattered_tables(rng, need, n_blocks, max_blocks, contiguous_first)
    pool_k = W.f32_to_bf16_bits(rng.standard_normal((n_blocks, h_kv, PAGE, d), dtype=np.float32))
    pool_v = W.f32_to_bf16_bits(rng.standard_normal((n_blocks, h_kv, PAGE, d), dtype=np.float32))
    q_new = W.f32_to_bf16_bits(rng.standard_normal((N, h_q, d), dtype=np.float32))
    k_new = W.f32_to_bf16_bits(rng.standard_normal((N, h_kv, d), dtype=np.float32))
    v_new = W.f32_to_bf16_bits(rng.standard_normal((N, h_kv, d), dtype=np.float32))
    return dict(lens=lens, active=np.asarray(active, np.uint8), table=table, n_blocks=n_blocks, max_blocks=max_blocks,
                pool_k=pool_k, pool_v=pool_v, q_new=q_new, k_new=k_new, v_new=v_new, h_q=h_q, h_kv=h_kv, d=d, N=N)


def _run_paged_decode(c, table=None):
    shape = kev.make_shape(c["h_q"], c["h_kv"], c["d"], "bf16")
    pk, pv = dev(c["pool_k"]), dev(c["pool_v"])
    out = torch.full((c["N"], c["h_q"], c["d"]), float("nan"), dtype=torch.bfloat16, device="cuda")
    nb = kev.kev_decode_workspace_size(c["N"], c["max_blocks"] * PAGE, shape)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    tb = c["table"] if table is None else table
    kev.kev_decode_attn_paged(dev(c["q_new"]), dev(c["k_new"]), dev(c["v_new"]), pk, pv, c["n_blocks"], _itensor(tb),
                              c["max_blocks"], _itensor(c["lens"]), torch.from_numpy(c["active"]).cuda(), c["N"], out,
                              shape, ws, nb, st)
    return kev.kev_read_status(st), out, pk, pv


@pytest.mark.parametrize("h_q,h_kv", [(32, 8), (28, 4), (16, 2)])
def test_decode_attn_paged_against_oracle(h_q, h_kv):
    lens = [127, 128, 255, 256, 0, 1000, 2047, 64]  # block boundaries, an empty cache, long ones
    active = [1, 1, 0, 1, 1, 1, 1, 0]
    c = _paged_decode_case(7 + h_q, lens, active, h_q, h_kv)
    assert O.validate_paged(c["lens"] + 1, c["table"], c["n_blocks"], live=c["active"]) is None
    status, out, pk, pv = _run_paged_decode(c)
    assert status == 0
    o_ref, pk_ref, pv_ref = O.decode_paged(c["q_new"], c["k_new"], c["v_new"], c["pool_k"], c["pool_v"], c["table"],
                                           c["lens"], c["active"], "bf16")
    got = f64(out, "bf16")
    live = c["active"].astype(bool)
    compare(got[live], o_ref[live], "bf16", f"paged decode G={h_q // h_kv}")
    assert np.isnan(got[~live]).all()
    np.testing.assert_array_equal(host(pk), pk_ref)  # the new rows, and nothing else
    np.testing.assert_array_equal(host(pv), pv_ref)


def test_paged_decode_is_bitwise_the_contiguous_decode():
    """The Qwen3-8B decode workload (64 slots of cap 2458, 32 live) copied into a paged pool with
    scattered blocks: the paged decode reads the same chunks in the same order, so its output and
    appended rows equal the contiguous decode's bit for bit."""
    dw = W.qwen3_8b_decode()
    N, h_q, h_kv, d = dw.n_questions, dw.h_q, dw.h_kv, dw.d
    shape = kev.make_shape(h_q, h_kv, d, "bf16")
    rng = np.random.default_rng(8)
    lens = np.asarray(dw.lens)
    live = np.asarray(dw.active).astype(bool)
    need = [(int(n) + 1 + PAGE - 1) // PAGE if a else 0 for n, a in zip(lens, live)]
    max_blocks = (dw.cap + PAGE - 1) // PAGE
    n_blocks = sum(need) + 32
    table = _scattered_tables(rng, need, n_blocks, max_blocks)
    # the paged copy of every live question's positions 0..lens (what the contiguous pool holds there)
    pool_k = np.zeros((n_blocks, h_kv, PAGE, d), np.uint16)
    pool_v = np.zeros((n_blocks, h_kv, PAGE, d), np.uint16)
    for i in np.nonzero(live)[0]:
        slot = int(dw.slot_ids[i])
        for b in range(need[i]):
            rows = slice(b * PAGE, min((b + 1) * PAGE, dw.cap))
            n_rows = rows.stop - rows.start
            pool_k[table[i, b], :, :n_rows] = dw.pool_k[slot, :, rows]
            pool_v[table[i, b], :, :n_rows] = dw.pool_v[slot, :, rows]
    # contiguous run
    ck, cv = dev(dw.pool_k), dev(dw.pool_v)
    out_c = torch.empty((N, h_q, d), dtype=torch.bfloat16, device="cuda")
    nb = kev.kev_decode_workspace_size(N, dw.cap, shape)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kev.kev_decode_attn(dev(dw.q_new), dev(dw.k_new), dev(dw.v_new), ck, cv, dw.n_slots, dw.cap, _itensor(dw.slot_ids),
                        _itensor(lens), torch.from_numpy(np.asarray(dw.active, np.uint8)).cuda(), N, out_c, shape, ws,
                        nb, st)
    assert kev.kev_read_status(st) == 0
    # paged run
    pk, pv = dev(pool_k), dev(pool_v)
    out_p = torch.empty((N, h_q, d), dtype=torch.bfloat16, device="cuda")
    nbp = kev.kev_decode_workspace_size(N, max_blocks * PAGE, shape)
    wsp = torch.zeros(nbp, dtype=torch.uint8, device="cuda")
    stp = torch.zeros(1, dtype=torch.int32, device="cuda")
    kev.kev_decode_attn_paged(dev(dw.q_new), dev(dw.k_new), dev(dw.v_new), pk, pv, n_blocks, _itensor(table),
                              max_blocks, _itensor(lens), torch.from_numpy(np.asarray(dw.active, np.uint8)).cuda(), N,
                              out_p, shape, wsp, nbp, stp)
    assert kev.kev_read_status(stp) == 0
    np.testing.assert_array_equal(host(out_p)[live], host(out_c)[live])
    hk, hck = host(pk), host(ck)
    for i in np.nonzero(live)[0]:  # the appended row landed at position lens_i of the question
        n = int(lens[i])
        np.testing.assert_array_equal(hk[table[i, n // PAGE], :, n % PAGE], hck[int(dw.slot_ids[i]), :, n])


def test_paged_table_errors_write_nothing():
    c = _paged_decode_case(21, [300, 129, 200], [1, 1, 1], 8, 2)
    # a block shared by two live questions
    bad = c["table"].copy()
    bad[1, 0] = bad[0, 1]
    assert O.validate_paged(c["lens"] + 1, bad, c["n_blocks"], live=c["active"]) == O.SLOT
    status, out, pk, pv = _run_paged_decode(c, bad)
    assert status == kev.binding.KEV_ERR_SLOT
    assert torch.isnan(out.float()).all()
    np.testing.assert_array_equal(host(pk), c["pool_k"])
    np.testing.assert_array_equal(host(pv), c["pool_v"])
    # the same sharing with the sharer dropped is valid
    c2 = dict(c, active=np.array([1, 0, 1], np.uint8))
    assert _run_paged_decode(c2, bad)[0] == 0
    # a table row too short for the new row
    short = c["table"].copy()
    short[0, (300 // PAGE):] = -1
    assert O.validate_paged(c["lens"] + 1, short, c["n_blocks"], live=c["active"]) == O.SLOT  # -1 entry
    c3 = dict(c, max_blocks=2, table=np.ascontiguousarray(c["table"][:, :2]))
    assert O.validate_paged(c["lens"] + 1, c3["table"], c["n_blocks"], live=c["active"]) == O.SLOT_OVERFLOW
    assert _run_paged_decode(c3)[0] == kev.binding.KEV_ERR_SLOT_OVERFLOW
    # prefill: a shared block writes neither the output nor the pool
    lengths = [200, 100]
    w = W.random_case(22, lengths, 4, 2, 128, "bf16", gaps=[1, 1], tail=1)
    run = PrefillRun(w, slots=False)
    table = np.array([[3, 4], [4, -1]], np.int32)
    pk = torch.full((6, 2, PAGE, 128), -7.0, dtype=torch.bfloat16, device="cuda")
    pv = torch.full((6, 2, PAGE, 128), -9.0, dtype=torch.bfloat16, device="cuda")
    kev.kev_prefill_attn_paged(run.q, run.k, run.v, w.total_tokens, run.intervals, run.n_questions, _itensor(table), 2,
                               pk, pv, 6, run.out, shape_of(w), run.ws, run.ws_bytes, run.status)
    assert run.device_status() == kev.binding.KEV_ERR_SLOT
    assert torch.isnan(run.out.float()).all()
    assert (host(pk) == host(torch.full_like(pk, -7.0))).all() and (host(pv) == host(torch.full_like(pv, -9.0))).all()
