"""The bounded-wait timeout path of the attention kernels, made to run out on purpose.

Every wait inside the kernels has a cycle budget; when one runs out the kernel stores
KEV_ERR_TIMEOUT, raises its CTA's abort flag, waits (again bounded) for its own copies and
MMAs, frees its tensor memory and returns, so the context stays usable.  Here the library's
test hook (KEV_TEST_STALL=1) makes CTA 0 of each kernel wait on an mbarrier that nothing
arrives on, with the budget shortened to about a millisecond (KEV_TEST_WAIT_LIMIT).  Nothing
faults, traps or hangs.

In a child process (the variables are read at every launch): the tensor-core prefill, the
tensor-core decode and the CUDA-core decode each report KEV_ERR_TIMEOUT and return; then,
with the hook off, the same calls (the decode workspace zeroed again, as the header asks)
match the oracle.  The workspace-free decode entry point on the CUDA-core path, whose
arrival counters a timeout leaves behind, recovers by itself on the next call.
"""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.join(ROOT, "tests")

CHILD = textwrap.dedent(r"""
    import os, sys
    sys.path[:0] = [ROOT, TESTS]
    import numpy as np
    import torch
    import packed_question_isolated_gb300 as kev
    import workloads as W
    from oracle import kev_oracle as O
    from kev_harness import DecodeRun, PrefillRun, compare, f64, host

    TIMEOUT = kev.binding.KEV_ERR_TIMEOUT

    def stall(on):
        if on:
            os.environ["KEV_TEST_STALL"] = "1"
            os.environ["KEV_TEST_WAIT_LIMIT"] = "2000000"  # ~1 ms at the top SM clock
        else:
            os.environ.pop("KEV_TEST_STALL", None)
            os.environ.pop("KEV_TEST_WAIT_LIMIT", None)

    # ---- tensor-core prefill: several CTAs of work, CTA 0 stalls
    w = W.random_case(41, [700, 130, 1, 513, 256, 90], 8, 2, 128, "bf16", cap=800)
    run = PrefillRun(w)
    stall(True)
    assert run.run() == 0
    assert run.device_status() == TIMEOUT, "prefill: expected KEV_ERR_TIMEOUT"
    stall(False)
    run.status.fill_(-1)
    assert run.run() == 0 and run.device_status() == 0
    ref = O.prefill(W.to_float64(w.q, "bf16"), W.to_float64(w.k, "bf16"), W.to_float64(w.v, "bf16"), w.intervals)
    compare(f64(run.out, "bf16"), ref, "bf16", "prefill after a timeout")
    print("prefill ok", flush=True)

    def decode_case(seed, dtype, d, G):
        rng = np.random.default_rng(seed)
        h_kv, cap, n_slots = 2, 1200, 10
        f = (lambda x: W.f32_to_bf16_bits(x)) if dtype == "bf16" else (lambda x: x)
        pk = f(rng.standard_normal((n_slots, h_kv, cap, d), dtype=np.float32))
        pv = f(rng.standard_normal((n_slots, h_kv, cap, d), dtype=np.float32))
        sl = rng.permutation(n_slots)[:8].astype(np.int32)
        lens = np.array([1100, 5, 640, 300, 0, 999, 128, 1150], np.int32)
        act = np.array([1, 1, 1, 0, 1, 1, 1, 1], np.uint8)
        q = f(rng.standard_normal((8, h_kv * G, d), dtype=np.float32))
        k = f(rng.standard_normal((8, h_kv, d), dtype=np.float32))
        v = f(rng.standard_normal((8, h_kv, d), dtype=np.float32))
        return (dtype, h_kv * G, h_kv, d, pk, pv, sl, lens, act, q, k, v, cap, n_slots)

    def check(run, case):
        dtype, h_q, h_kv, d, pk, pv, sl, lens, act, q, k, v, cap, n_slots = case
        o_ref, ek, ev = O.decode(q, k, v, pk, pv, sl, lens, act, dtype)
        live = act.astype(bool)
        compare(f64(run.out, dtype)[live], o_ref[live], dtype, f"decode {dtype} d={d} after a timeout")
        assert np.array_equal(host(run.pool_k), ek) and np.array_equal(host(run.pool_v), ev)

    def fresh(case):
        return DecodeRun(*case)

    # ---- decode through a caller workspace: tensor cores (bf16 d=128), CUDA cores (fp32 d=64)
    for case in (decode_case(42, "bf16", 128, 4), decode_case(43, "fp32", 64, 4)):
        run = fresh(case)
        stall(True)
        assert run.run() == 0
        assert run.device_status() == TIMEOUT, f"decode {case[0]}: expected KEV_ERR_TIMEOUT"
        stall(False)
        run = fresh(case)  # pools as before the failed call; the workspace zeroed again
        assert run.run() == 0 and run.device_status() == 0
        check(run, case)
        print(f"decode {case[0]} ok", flush=True)

    # ---- the workspace-free entry point: a timeout, then a normal call on the same scratch
    def static_call(run):
        return kev.kev_decode_attn_static(run.q_new, run.k_new, run.v_new, run.pool_k, run.pool_v, run.n_slots,
                                          run.cap, run.slot_ids, run.lens, run.active, run.n, run.out, run.shape,
                                          run.status, check=False)

    for case in (decode_case(44, "fp32", 64, 4), decode_case(45, "bf16", 128, 8)):
        run = fresh(case)
        stall(True)
        assert static_call(run) == 0
        assert run.device_status() == TIMEOUT, f"static {case[0]}: expected KEV_ERR_TIMEOUT"
        stall(False)
        for rep in range(2):
            run = fresh(case)
            assert static_call(run) == 0 and run.device_status() == 0
            check(run, case)
        print(f"static {case[0]} ok", flush=True)
    print("ALL OK", flush=True)
""").replace("ROOT", repr(ROOT)).replace("TESTS", repr(TESTS))


def test_timeouts_are_reported_and_the_next_call_is_correct():
    env = {k: v for k, v in os.environ.items() if k not in ("KEV_TEST_STALL", "KEV_TEST_WAIT_LIMIT")}
    r = subprocess.run([sys.executable, "-c", CHILD], capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0 and "ALL OK" in r.stdout, f"child failed:\n{r.stdout}\n{r.stderr[-4000:]}"
