"""kev_decode_attn_static: the decode step for callers that cannot allocate device memory.

Such callers (a plugin inside a framework that owns the whole device-memory budget, or a
latency-critical path where cudaMalloc/cudaFree are not allowed) get a variant of
kev_decode_attn that keeps its scratch (split-K partials and arrival counters) in a fixed
array inside the library instead of a caller workspace.  This file checks, through the C ABI,
that two calls in a row give the same results as kev_decode_attn with a workspace, and that
a call needing more scratch than the fixed maximum is refused without launching anything.

The file name sorts last so that a run stopping at the first failure has already run every
other test; it also passes alone in a fresh process (the first call sets the scratch up).
"""
import numpy as np
import pytest
import torch

import packed_question_isolated_gb300 as kev
import workloads as W

from kev_harness import DecodeRun, compare, f64, host

pytestmark = pytest.mark.gpu


def _case(seed, lens, active):
    rng = np.random.default_rng(seed)
    h_kv, G, d, cap, n_slots = 4, 4, 128, 1100, 12
    n = len(lens)
    pool_k = W.f32_to_bf16_bits(rng.standard_normal((n_slots, h_kv, cap, d), dtype=np.float32))
    pool_v = W.f32_to_bf16_bits(rng.standard_normal((n_slots, h_kv, cap, d), dtype=np.float32))
    slot_ids = rng.permutation(n_slots)[:n].astype(np.int32)
    q = W.f32_to_bf16_bits(rng.standard_normal((n, h_kv * G, d), dtype=np.float32))
    k = W.f32_to_bf16_bits(rng.standard_normal((n, h_kv, d), dtype=np.float32))
    v = W.f32_to_bf16_bits(rng.standard_normal((n, h_kv, d), dtype=np.float32))
    return (h_kv * G, h_kv, d, pool_k, pool_v, slot_ids, np.array(lens, np.int32), np.array(active, np.uint8),
            q, k, v, cap, n_slots)


def _static_call(run):
    return kev.kev_decode_attn_static(run.q_new, run.k_new, run.v_new, run.pool_k, run.pool_v, run.n_slots,
                                      run.cap, run.slot_ids, run.lens, run.active, run.n, run.out, run.shape,
                                      run.status, check=False)


def test_static_scratch_matches_workspace_path_on_two_calls_in_a_row():
    cases = [
        (11, [0, 1, 255, 256, 257, 700, 1099, 40], [1, 1, 1, 1, 1, 1, 1, 1]),
        (12, [900, 3, 512, 513, 64, 1000, 17, 255], [1, 0, 1, 1, 0, 1, 1, 1]),
    ]
    for seed, lens, active in cases:
        h_q, h_kv, d, pool_k, pool_v, slots, ln, act, q, k, v, cap, n_slots = _case(seed, lens, active)
        ref = DecodeRun("bf16", h_q, h_kv, d, pool_k, pool_v, slots, ln, act, q, k, v, cap, n_slots)
        assert ref.run() == 0 and ref.device_status() == 0
        got = DecodeRun("bf16", h_q, h_kv, d, pool_k, pool_v, slots, ln, act, q, k, v, cap, n_slots)
        assert _static_call(got) == 0
        assert got.device_status() == 0
        live = act.astype(bool)
        compare(f64(got.out, "bf16")[live], f64(ref.out, "bf16")[live], "bf16", f"static vs workspace, seed {seed}")
        assert torch.isnan(got.out.float()[torch.from_numpy(~live)]).all()
        assert np.array_equal(host(got.pool_k), host(ref.pool_k))
        assert np.array_equal(host(got.pool_v), host(ref.pool_v))


def test_static_scratch_refuses_sizes_beyond_its_maximum():
    h_q, h_kv, d = 32, 8, 128
    shape = kev.make_shape(h_q, h_kv, d, "bf16")
    n, cap = 256, 4224
    assert kev.kev_decode_workspace_size(n, cap, shape) > kev.binding.KEV_STATIC_SCRATCH_BYTES
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    st = kev.kev_decode_attn_static(dummy, dummy, dummy, dummy, dummy, n, cap, status, status, status, n, dummy,
                                    shape, status, check=False)
    assert st == kev.binding.KEV_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert int(status.item()) == -1, "nothing may run for a refused call"
