"""The bench's N > 1 path on CPU: max-over-ranks timing and whole-job aggregation over two gloo
ranks, and the reference arm under a torchrun-style environment (rank 0 prints, others exit)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        local_ms = [120.0, 180.0][rank]  # rank 1 is the slow one
        m = bench.max_over_ranks(local_ms, world, "cpu")
        q.put((rank, m, bench.aggregate_rate(1000.0, 10, world, m)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_aggregate_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, m, rate in got:
        assert m == 180.0, "every rank sees the slowest rank's time"
        # 2 ranks x 10 steps x 1000 units in 180 ms
        assert rate == pytest.approx(2 * 10 * 1000.0 / 0.180)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.aggregate_rate(5.0, 4, 1, 2.0) == pytest.approx(5.0 * 4 / 0.002)


def _run_reference(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1")
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                           "--steps", "1", "--warmup", "3"], cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=300)


def test_reference_arm_under_torchrun_rank0_prints_others_exit():
    r1 = _run_reference(1)
    assert r1.returncode == 0 and r1.stdout.strip() == "", "ranks other than 0 exit 0 without work"
    r0 = _run_reference(0)
    assert r0.returncode == 0, r0.stderr[-2000:]
    lines = [l for l in r0.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
