"""Device-detected errors: the status code matches the oracle's validation and nothing is written."""
import numpy as np
import pytest
import torch

import packed_question_isolated_gb300 as kev
import workloads as W
from oracle import kev_oracle as O

from kev_harness import DecodeRun, PrefillRun, host

pytestmark = pytest.mark.gpu

CODE = {None: kev.binding.KEV_OK, O.INTERVALS: kev.binding.KEV_ERR_INTERVALS, O.SLOT: kev.binding.KEV_ERR_SLOT,
        O.SLOT_OVERFLOW: kev.binding.KEV_ERR_SLOT_OVERFLOW}

PREFILL_BAD = [
    # intervals, slot_ids, cap
    ([[0, 40], [30, 60]], [0, 1], 64),     # overlap
    ([[0, 40], [40, 70]], [0, 1], 64),     # past T (T = 64)
    ([[10, 5], [20, 30]], [0, 1], 64),     # reversed
    ([[0, 20], [20, 40]], [0, 3], 64),     # slot out of range (n_slots = 3)
    ([[0, 20], [20, 40]], [1, 1], 64),     # shared slot
    ([[0, 20], [20, 40]], [1, 2], 16),     # longer than the slot
    ([[0, 20], [20, 20]], [1, 1], 64),     # empty question may share a slot: valid
    ([[0, 16], [16, 40]], [2, 0], 24),     # exactly cap: valid
    ([[20, 40], [0, 20]], [0, 1], 64),     # not in index order: valid
    ([[24, 40], [0, 20]], [2, 2], 64),     # not in index order, shared slot
]


@pytest.mark.parametrize("case", range(len(PREFILL_BAD)))
def test_prefill_errors_match_oracle_and_write_nothing(case):
    iv, slots, cap = PREFILL_BAD[case]
    w = W.random_case(400 + case, [40, 24], 4, 2, 64, "bf16", cap=cap, n_slots=3)
    w.cap = cap
    iv = np.array(iv, np.int32)
    expect = O.validate_prefill(iv, w.total_tokens, slots, w.n_slots, cap)
    run = PrefillRun(w, intervals=iv, slot_ids=np.array(slots, np.int32))
    st = run.run(check=False)
    assert st == 0  # host-side checks pass; the error is data dependent
    code = run.device_status()
    assert code == CODE[expect]
    if expect is not None:
        assert torch.isnan(run.out.float()).all(), "out written despite an error"
        assert torch.equal(run.pool_k, run.pool_k0) and torch.equal(run.pool_v, run.pool_v0)


DECODE_BAD = [
    # slot_ids, lens, active
    ([0, 1, 2], [3, 7, 5], [1, 1, 1]),     # valid
    ([0, 1, 2], [3, 8, 5], [1, 1, 1]),     # lens == cap: no room
    ([0, 1, 2], [3, 8, 5], [1, 0, 1]),     # ... but that question is dropped: valid
    ([0, 0, 2], [3, 1, 5], [1, 1, 1]),     # two live questions on one slot
    ([0, 0, 2], [3, 1, 5], [1, 0, 1]),     # shared only with a dropped question: valid
    ([0, 4, 2], [3, 1, 5], [1, 1, 1]),     # slot out of range
    ([0, 1, 2], [-1, 1, 5], [1, 1, 1]),    # negative length
]


@pytest.mark.parametrize("case", range(len(DECODE_BAD)))
def test_decode_errors_match_oracle_and_write_nothing(case):
    slots, lens, active = DECODE_BAD[case]
    rng = np.random.default_rng(case)
    cap, n_slots = 8, 4
    pool = W.f32_to_bf16_bits(rng.standard_normal((n_slots, 2, cap, 64), dtype=np.float32))
    q = W.f32_to_bf16_bits(rng.standard_normal((3, 4, 64), dtype=np.float32))
    kv = W.f32_to_bf16_bits(rng.standard_normal((3, 2, 64), dtype=np.float32))
    expect = O.validate_decode(slots, lens, active, n_slots, cap)
    run = DecodeRun("bf16", 4, 2, 64, pool, pool.copy(), slots, lens, active, q, kv, kv, cap, n_slots)
    assert run.run(check=False) == 0
    assert run.device_status() == CODE[expect]
    if expect is not None:
        assert torch.isnan(run.out.float()).all()
        assert np.array_equal(host(run.pool_k), pool)


def test_host_side_errors_launch_nothing():
    w = W.random_case(7, [10, 12], 4, 2, 64, "bf16")
    run = PrefillRun(w)
    bad_shape = kev.make_shape(4, 3, 64, "bf16")
    st = kev.kev_prefill_attn(run.q, run.k, run.v, w.total_tokens, run.intervals, 2, run.slot_ids, run.pool_k,
                              run.pool_v, w.n_slots, w.cap, run.out, bad_shape, run.ws, run.ws_bytes, run.status,
                              check=False)
    assert st == kev.binding.KEV_ERR_UNSUPPORTED
    st = kev.kev_prefill_attn(run.q, run.k, run.v, w.total_tokens, run.intervals, 2, run.slot_ids, run.pool_k,
                              run.pool_v, w.n_slots, w.cap, run.out, kev.make_shape(4, 2, 96), run.ws,
                              run.ws_bytes, run.status, check=False)
    assert st == kev.binding.KEV_ERR_UNSUPPORTED
    st = kev.kev_prefill_attn(run.q, run.k, run.v, w.total_tokens, run.intervals, 2, run.slot_ids, run.pool_k,
                              run.pool_v, w.n_slots, w.cap, run.out, kev.make_shape(4, 2, 64), run.ws, 16,
                              run.status, check=False)
    assert st == kev.binding.KEV_ERR_INVALID_ARG
    st = kev.kev_prefill_attn(run.q.data_ptr() + 2, run.k, run.v, w.total_tokens, run.intervals, 2, run.slot_ids,
                              run.pool_k, run.pool_v, w.n_slots, w.cap, run.out, kev.make_shape(4, 2, 64),
                              run.ws, run.ws_bytes, run.status, check=False)
    assert st == kev.binding.KEV_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert int(run.status.item()) == -1, "a launch happened for a call rejected on the host"
    assert torch.isnan(run.out.float()).all()
