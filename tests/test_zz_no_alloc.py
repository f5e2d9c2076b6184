"""kev_decode_attn_static: the decode step for callers that cannot allocate device memory.

Such callers (a plugin inside a framework that owns the whole device-memory budget, or a
latency-critical path where cudaMalloc/cudaFree are not allowed) get a variant of
kev_decode_attn that keeps its scratch (split-K partials and arrival counters) in a fixed
array inside the library instead of a caller workspace.  This file checks, through the C ABI,
that two calls in a row match the oracle and kev_decode_attn with a workspace, on the
tensor-core path (bf16, d = 128) and on the CUDA-core path (fp32, and bf16 at d = 64), whose
arrival counters the shared array carries from call to call; and that a call needing more
scratch than the fixed maximum is refused without launching anything, after the same
argument checks as kev_decode_attn.

The file name sorts last so that a run stopping at the first failure has already run every
other test; it also passes alone in a fresh process (the first call sets the scratch up).
"""
import numpy as np
import pytest
import torch

import packed_question_isolated_gb300 as kev
import workloads as W
from oracle import kev_oracle as O

from kev_harness import DecodeRun, compare, f64, host

pytestmark = pytest.mark.gpu


def _case(seed, lens, active, dtype="bf16", d=128, G=4):
    rng = np.random.default_rng(seed)
    h_kv, cap, n_slots = 4, 1100, 12
    n = len(lens)
    f = W.f32_to_bf16_bits if dtype == "bf16" else (lambda x: x)
    pool_k = f(rng.standard_normal((n_slots, h_kv, cap, d), dtype=np.float32))
    pool_v = f(rng.standard_normal((n_slots, h_kv, cap, d), dtype=np.float32))
    slot_ids = rng.permutation(n_slots)[:n].astype(np.int32)
    q = f(rng.standard_normal((n, h_kv * G, d), dtype=np.float32))
    k = f(rng.standard_normal((n, h_kv, d), dtype=np.float32))
    v = f(rng.standard_normal((n, h_kv, d), dtype=np.float32))
    return (dtype, h_kv * G, h_kv, d, pool_k, pool_v, slot_ids, np.array(lens, np.int32),
            np.array(active, np.uint8), q, k, v, cap, n_slots)


def _static_call(run):
    return kev.kev_decode_attn_static(run.q_new, run.k_new, run.v_new, run.pool_k, run.pool_v, run.n_slots,
                                      run.cap, run.slot_ids, run.lens, run.active, run.n, run.out, run.shape,
                                      run.status, check=False)


CASES = [
    (11, [0, 1, 255, 256, 257, 700, 1099, 40], [1, 1, 1, 1, 1, 1, 1, 1], "bf16", 128, 4),
    (12, [900, 3, 512, 513, 64, 1000, 17, 255], [1, 0, 1, 1, 0, 1, 1, 1], "bf16", 128, 4),
    (13, [900, 3, 512, 513, 64, 1000, 17, 255], [1, 1, 1, 0, 1, 1, 0, 1], "fp32", 64, 4),
    (14, [1099, 0, 129, 600, 31, 1000, 256, 2], [1, 1, 1, 1, 1, 0, 1, 1], "bf16", 64, 8),
    (15, [640, 77, 1, 1098, 300, 512, 5, 900], [1, 1, 0, 1, 1, 1, 1, 1], "fp32", 128, 16),
]


@pytest.mark.parametrize("seed,lens,active,dtype,d,G", CASES)
def test_static_scratch_matches_oracle_and_workspace_path_on_two_calls_in_a_row(seed, lens, active, dtype, d, G):
    case = _case(seed, lens, active, dtype, d, G)
    _, h_q, h_kv, d, pool_k, pool_v, slots, ln, act, q, k, v, cap, n_slots = case
    o_ref, ek, ev = O.decode(q, k, v, pool_k, pool_v, slots, ln, act, dtype)
    live = act.astype(bool)
    ref = DecodeRun(*case)
    assert ref.run() == 0 and ref.device_status() == 0
    for call in range(2):  # the shared array carries the previous call's contents
        got = DecodeRun(*case)
        assert _static_call(got) == 0
        assert got.device_status() == 0
        compare(f64(got.out, dtype)[live], o_ref[live], dtype, f"static vs oracle, seed {seed}, call {call}")
        compare(f64(got.out, dtype)[live], f64(ref.out, dtype)[live], dtype, f"static vs workspace, seed {seed}")
        assert torch.isnan(got.out.float()[torch.from_numpy(~live)]).all(), "dropped rows must stay untouched"
        assert np.array_equal(host(got.pool_k), ek) and np.array_equal(host(got.pool_v), ev)


def test_static_scratch_refuses_sizes_beyond_its_maximum():
    h_q, h_kv, d = 32, 8, 128
    shape = kev.make_shape(h_q, h_kv, d, "bf16")
    n, cap = 256, 4224
    assert kev.kev_decode_workspace_size(n, cap, shape) > kev.binding.KEV_STATIC_SCRATCH_BYTES
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    # valid buffers of the refused size: the refusal comes from the scratch limit alone
    q = torch.zeros((n, h_q, d), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((n, h_kv, d), dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros((1, h_kv, cap, d), dtype=torch.bfloat16, device="cuda")
    slots = torch.zeros(n, dtype=torch.int32, device="cuda")
    lens = torch.zeros(n, dtype=torch.int32, device="cuda")
    act = torch.zeros(n, dtype=torch.uint8, device="cuda")
    out = torch.zeros((n, h_q, d), dtype=torch.bfloat16, device="cuda")
    st = kev.kev_decode_attn_static(q, kv, kv, pool, pool, 1, cap, slots, lens, act, n, out, shape, status,
                                    check=False)
    assert st == kev.binding.KEV_ERR_UNSUPPORTED
    # argument errors are reported first, with kev_decode_attn's codes
    st = kev.kev_decode_attn_static(q, kv, kv, pool, pool, 1, cap, slots, lens, None, n, out, shape, status,
                                    check=False)
    assert st == kev.binding.KEV_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert int(status.item()) == -1, "nothing may run for a refused call"
