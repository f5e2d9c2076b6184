"""Benchmark of the packed, question-isolated attention hot path on GB300.

One step = the whole hot path over one batch of 8 Qwen2.5-7B-shaped questions
(lengths U{256..2048}, T = 7921, H_q 28 / H_kv 4, d 128, bf16, slot cap 2458):
segment build + prefill attention + slot write + one decode step of every
question, all through the C ABI of libkev.  The headline value is useful
prefill TFLOP/s over the whole step (sum_i 2 d H_q L_i (L_i + 1) per step).
Decode GB/s is measured on its own workload (64-slot pool of cap 2458, 32 of
64 questions live) and reported in the same JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

With torchrun, every rank runs its own batch (questions are independent:
weak scaling, no collective on the data path); rank 0 prints one JSON line.
``--impl reference`` times the CPU oracle (dense-mask fp64 attention) on a
bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402
from packed_question_isolated_gb300 import roofline as RL  # noqa: E402

METRIC = "prefill useful TFLOP/s & decode HBM GB/s vs GB300 roofline, 1 GPU"
WORKLOAD = ("qwen25_7b_prefill: 8 questions, lengths U{256..2048} seed 2 (T=7921), H_q 28, H_kv 4, d 128, bf16, "
            "slot cap 2458; step = segment build + prefill attention + slot write + 1 decode step per question")
DECODE_WORKLOAD = ("qwen3_8b_decode: [64, 8, 2458, 128] bf16 pools, lens U{64..2400} seed 4, 32 of 64 questions "
                   "live, 1 new token each")
PREFILL3_WORKLOAD = ("qwen3_8b_prefill: 32 questions, lengths clip(rint(exp(N(ln 512, 0.8))), 1, 4096) seed 3 "
                     "(T=24100), H_q 32, H_kv 8, d 128, bf16; one call = segment build + prefill attention + slot "
                     "write into [32, 8, 4096, 128] pools")
STEP_COPIES = 3           # buffer sets the back-to-back steps cycle through
DECODE_COPIES = 2


def max_over_ranks(x: float, world: int, device="cpu") -> float:
    """The largest of every rank's value (the slowest rank's elapsed time); x itself on one rank."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(units_per_rank: float, steps: int, world: int, max_ms: float) -> float:
    """Whole-job throughput under weak scaling: every rank processes units_per_rank per step, the
    job takes as long as its slowest rank (max_ms for all steps)."""
    return units_per_rank * steps * world / (max_ms * 1e-3)


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def _traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel source is unchanged."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        fields = dict(kv.split("=", 1) for kv in line.split() if "=" in kv)
        if fields.get("kernel") != kernel:
            continue
        src = os.path.join(ROOT, "packed_question_isolated_gb300", "csrc", fields.get("source", ""))
        if not os.path.exists(src):
            return None
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        if h != fields.get("sha"):
            return None
        return float(fields["bytes_per_launch"])
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled in the background."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"kev_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "100"], stdout=open(self.path, "w"),
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        time.sleep(0.2)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        mx = max(r[1] for r in rows)
        load = [r for r in rows if r[0] > 0.5 * mx] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[j] for r in load for j, v in enumerate(r[2]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in load), "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------------------
# CPU oracle legs (bounded samples)
# ---------------------------------------------------------------------------------------

_W_CACHE = {}


def _oracle_sample(heads):
    """Time the oracle's dense-mask prefill for the given q-heads over the whole packed batch."""
    from oracle import kev_oracle as O
    if "w" not in _W_CACHE:
        _W_CACHE["w"] = W.qwen25_7b_prefill()
    w = _W_CACHE["w"]
    G = w.h_q // w.h_kv
    kv_heads = sorted({h // G for h in heads})
    q = W.to_float64(w.q[:, heads], "bf16")
    k = W.to_float64(w.k[:, kv_heads], "bf16")
    v = W.to_float64(w.v[:, kv_heads], "bf16")
    # keep the GQA mapping of the sampled heads: a sample of G' q-heads per kv head
    t0 = time.perf_counter()
    O.prefill(q, k, v, w.intervals)
    dt = time.perf_counter() - t0
    flops = RL.prefill_useful_flops(w.lengths, len(heads), w.d)
    return flops, dt


def cpu_baseline(heads=tuple(range(14))):
    heads = list(heads)
    flops, dt = _oracle_sample(heads)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"oracle dense-mask fp64 prefill of q-heads {heads[0]}-{heads[-1]} (of 28; kv-heads 0-1) "
                      f"over the full 8-question packed batch (T=7921); {dt:.2f} s"}


def cpu_fair_baseline():
    """A labelled second CPU number (not the oracle): per-question fp32 attention with BLAS
    matmuls over each question's own causal block, all q-heads of the packed batch."""
    import numpy as np
    if "w" not in _W_CACHE:
        _W_CACHE["w"] = W.qwen25_7b_prefill()
    w = _W_CACHE["w"]
    G = w.h_q // w.h_kv
    q = W.to_float64(w.q, "bf16").astype(np.float32)
    k = W.to_float64(w.k, "bf16").astype(np.float32)
    v = W.to_float64(w.v, "bf16").astype(np.float32)
    scale = np.float32(1.0 / np.sqrt(w.d))
    t0 = time.perf_counter()
    for s0, e0 in w.intervals:
        L = e0 - s0
        tri = np.triu(np.ones((L, L), dtype=bool), 1)
        for h in range(w.h_q):
            g = h // G
            sc = (q[s0:e0, h] @ k[s0:e0, g].T) * scale
            sc[tri] = -np.inf
            sc -= sc.max(axis=1, keepdims=True)
            np.exp(sc, out=sc)
            sc /= sc.sum(axis=1, keepdims=True)
            _ = sc @ v[s0:e0, g]
    dt = time.perf_counter() - t0
    flops = RL.prefill_useful_flops(w.lengths, w.h_q, w.d)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "fair (not the oracle)",
            "sample": f"per-question fp32 numpy/BLAS causal attention, all 28 q-heads of the 8-question batch "
                      f"(T=7921), useful flops only; {dt:.2f} s"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    heads = [0]
    for _ in range(args.warmup):
        _oracle_sample(heads)
    times = []
    flops = 0.0
    for _ in range(args.steps):
        f, dt = _oracle_sample(heads)
        flops += f
        times.append(dt)
    total = sum(times)
    value = flops / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": "q-head 0 of 28 per step"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": "oracle dense-mask fp64 prefill of q-head 0 over the full packed batch "
                                   "(T=7921), one per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------------------

def _stress_decode_graph(kev, torch, dev, tdev, tf_peak, hbm_peak):
    """The stress batch: prefill into the slot pools, then its 128-step decode loop with early
    stop (kev_decode_step per step: decode with the lens advance folded in, each step with its own
    live set and inputs) captured once as a CUDA graph and replayed.  L2 is not flushed between
    the steps of a replay."""
    import numpy as np
    s = W.stress()
    w = s.prefill
    shape = kev.make_shape(w.h_q, w.h_kv, w.d, "bf16")
    N = w.n_questions
    q, k, v, iv, sl = tdev(w.q), tdev(w.k), tdev(w.v), tdev(w.intervals), tdev(w.slot_ids)
    pk = torch.zeros((w.n_slots, w.h_kv, w.cap, w.d), dtype=torch.bfloat16, device=dev)
    pv = torch.zeros_like(pk)
    out = torch.empty((w.total_tokens, w.h_q, w.d), dtype=torch.bfloat16, device=dev)
    pws_bytes = kev.kev_prefill_workspace_size(N, w.total_tokens, shape)
    pws = torch.empty(pws_bytes, dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    pre_ms = []
    for it in range(4):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        kev.kev_prefill_attn(q, k, v, w.total_tokens, iv, N, sl, pk, pv, w.n_slots, w.cap, out, shape, pws, pws_bytes, st)
        b.record()
        pre_ms.append((a, b))
    torch.cuda.synchronize()
    assert kev.kev_read_status(st) == 0
    pre_avg = statistics.mean(a.elapsed_time(b) for a, b in pre_ms[1:])
    steps = s.n_steps
    act = tdev(np.stack([s.active_at(t) for t in range(steps)]))
    ins = [s.step_inputs(t) for t in range(steps)]
    qn = tdev(np.stack([x[0] for x in ins]))
    kn = tdev(np.stack([x[1] for x in ins]))
    vn = tdev(np.stack([x[2] for x in ins]))
    del ins
    lens0 = tdev(s.lens_at(0))
    lens = lens0.clone()
    dout = torch.empty((N, w.h_q, w.d), dtype=torch.bfloat16, device=dev)
    dws_bytes = kev.kev_decode_workspace_size(N, w.cap, shape)
    dws = torch.zeros(dws_bytes, dtype=torch.uint8, device=dev)
    pk0, pv0 = pk.clone(), pv.clone()

    def loop():  # one fused call per step: decode, then the lens advance folded into its merge kernel
        for t in range(steps):
            kev.kev_decode_step(qn[t], kn[t], vn[t], pk, pv, w.n_slots, w.cap, sl, lens, act[t], N, dout, shape, dws,
                                dws_bytes, st)

    loop()  # eager pass: first-call work happens outside the capture
    torch.cuda.synchronize()
    assert kev.kev_read_status(st) == 0
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        loop()
    reps = []
    for _ in range(3):
        pk.copy_(pk0)
        pv.copy_(pv0)
        lens.copy_(lens0)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        reps.append(a.elapsed_time(b))
    assert kev.kev_read_status(st) == 0
    total_bytes = sum(RL.decode_bytes(s.lens_at(t), s.active_at(t), w.h_q, w.h_kv, w.d, 2) for t in range(steps))
    ms = statistics.mean(reps)
    useful = RL.prefill_useful_flops(w.lengths, w.h_q, w.d)
    # short questions make this prefill memory-bound: its intensity (useful FLOP per algorithmic
    # byte: q, k, v read, out and both slot rows written) is below the ridge point peak / bandwidth
    pre_bytes = RL.prefill_bytes(w.total_tokens, w.h_q, w.h_kv, w.d, 2)
    intensity = RL.arithmetic_intensity(useful, pre_bytes)
    ridge = tf_peak * 1e12 / (hbm_peak * 1e9)
    return {"workload": "stress: 256 questions (T=19483), H_q 32, H_kv 8, d 128, bf16, cap 4224; prefill with slot "
                        "write, then 128 decode steps with early stop (116 with live questions)",
            "prefill_tflops": useful / (pre_avg * 1e-3) / 1e12, "prefill_ms": pre_avg,
            "prefill_frac": useful / (pre_avg * 1e-3) / 1e12 / tf_peak,
            "prefill_bytes": pre_bytes, "prefill_gbs": pre_bytes / (pre_avg * 1e-3) / 1e9,
            "prefill_intensity_flop_per_byte": intensity, "ridge_flop_per_byte": ridge,
            "prefill_bound": "hbm" if intensity < ridge else "tensor",
            "prefill_bound_frac": (RL.ideal_time(useful, pre_bytes, tf_peak * 1e12, hbm_peak * 1e9) * 1e3) / pre_avg,
            "decode_graph_ms": ms, "decode_steps": steps, "decode_bytes": total_bytes,
            "decode_gbs": total_bytes / (ms * 1e-3) / 1e9, "decode_frac": total_bytes / (ms * 1e-3) / 1e9 / hbm_peak,
            "launches_per_step": kev.kev_launch_count(15),
            "l2": "not flushed between the steps of a graph replay (L2 may hold part of the working set)"}


ROPE_THETA = 1e6  # Qwen2.5 / Qwen3 rotary base


def _rope_step(kev, torch, w, shape, copies, step_buffers, ws_bytes, dws_bytes, K, warmup, useful, hbm_peak):
    """The headline step with RoPE: segment build, prefill-side RoPE with the slot write, attention
    (no second slot write), then decode-side RoPE and the decode of one new token per question;
    back to back over the same buffer sets (q, k, q_new, k_new are rotated in place every step)."""
    N, T = w.n_questions, w.total_tokens
    table = torch.empty(kev.kev_rope_table_size(w.cap, w.d) // 4, dtype=torch.float32, device=copies[0]["q"].device)
    kev.kev_rope_table(table, w.cap, w.d, ROPE_THETA)

    def rstep(c, ev_a=None, ev_b=None):
        kev.kev_build_segments(c["iv"], N, T, c["sl"], w.n_slots, w.cap, shape, c["ws"], ws_bytes, c["st"])
        if ev_a is not None:
            ev_a.record()
        kev.kev_rope_prefill(c["q"], c["k"], c["v"], T, c["iv"], N, c["sl"], c["pk"], c["pv"], w.n_slots, w.cap,
                             shape, table, w.cap, c["ws"], ws_bytes, c["st"])
        if ev_b is not None:
            ev_b.record()
        kev.kev_prefill_from_segments(c["q"], c["k"], c["v"], T, c["iv"], N, None, None, None, 0, 0, c["out"],
                                      shape, c["ws"], ws_bytes, c["st"])
        kev.kev_decode_attn_rope(c["qn"], c["kn"], c["vn"], c["pk"], c["pv"], w.n_slots, w.cap, c["sl"], c["ln"],
                                 c["act"], N, c["on"], shape, table, w.cap, c["dws"], dws_bytes, c["dst"])

    for _ in range(warmup):
        for c in copies:
            rstep(c)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for s in range(K):
        rstep(copies[s % len(copies)])
    b.record()
    torch.cuda.synchronize()
    step_ms = a.elapsed_time(b) / K
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for s in range(K):
        rstep(copies[s % len(copies)], ev[s][0], ev[s][1])
    torch.cuda.synchronize()
    ok = all(kev.kev_read_status(c["st"]) == 0 and kev.kev_read_status(c["dst"]) == 0 for c in copies)
    rope_ms = statistics.mean(x.elapsed_time(y) for x, y in ev)
    rbytes = RL.rope_prefill_bytes(w.lengths, w.h_q, w.h_kv, w.d, 2, slots=True)
    return {"workload": "the step above with RoPE (theta 1e6, positions restart in every question): segment build, "
                        "prefill-side RoPE with the slot write, attention, decode-side RoPE and decode",
            "value": useful / (step_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": step_ms, "status_ok": ok,
            "roofline": {"kernel": "rope_prefill_kernel (rotation in place + slot write)", "bound": "hbm",
                         "achieved": rbytes / (rope_ms * 1e-3) / 1e9, "peak": hbm_peak, "unit": "GB/s",
                         "frac": rbytes / (rope_ms * 1e-3) / 1e9 / hbm_peak, "algorithmic_bytes": rbytes,
                         "launch_ms": rope_ms, "traffic": _traffic("rope")}}


def _chunked_prefill(kev, torch, tdev, dev, K, warmup):
    """The Qwen2.5-7B-shaped batch prefilled as two chunks per question (the first ending on the
    last tile boundary at or below half the question, the second attending to it from the slot),
    back to back over two buffer sets; useful FLOPs as for one prefill."""
    w = W.qwen25_7b_prefill()
    N, T = w.n_questions, w.total_tokens
    shape = kev.make_shape(w.h_q, w.h_kv, w.d, "bf16")
    cap = (w.cap + 127) // 128 * 128
    iv = np.asarray(w.intervals)
    L = iv[:, 1] - iv[:, 0]
    cut = ((L // 2) // 128 * 128).astype(np.int32)
    parts = [(np.stack([iv[:, 0], iv[:, 0] + cut], 1), np.zeros(N, np.int32)),
             (np.stack([iv[:, 0] + cut, iv[:, 1]], 1), cut)]
    nb = kev.kev_prefill_workspace_size(N, T, shape)
    copies = []
    for _ in range(2):
        c = {"q": tdev(w.q), "k": tdev(w.k), "v": tdev(w.v), "sl": tdev(w.slot_ids),
             "out": torch.empty((T, w.h_q, w.d), dtype=torch.bfloat16, device=dev),
             "pk": torch.zeros((w.n_slots, w.h_kv, cap, w.d), dtype=torch.bfloat16, device=dev),
             "ws": torch.empty(nb, dtype=torch.uint8, device=dev), "st": torch.zeros(1, dtype=torch.int32, device=dev),
             "iv": [tdev(pi.astype(np.int32)) for pi, _ in parts], "pre": [tdev(pp) for _, pp in parts]}
        c["pv"] = torch.zeros_like(c["pk"])
        copies.append(c)

    def call(c, part):
        kev.kev_prefill_chunk(c["q"], c["k"], c["v"], T, c["iv"][part], N, c["pre"][part], c["sl"], c["pk"], c["pv"],
                              w.n_slots, cap, c["out"], shape, c["ws"], nb, c["st"])

    for _ in range(warmup):
        for c in copies:
            call(c, 0)
            call(c, 1)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for s in range(K):
        call(copies[s % 2], 0)
        call(copies[s % 2], 1)
    b.record()
    torch.cuda.synchronize()
    pair_ms = a.elapsed_time(b) / K
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for s in range(K):
        call(copies[s % 2], 0)
        ev[s][0].record()
        call(copies[s % 2], 1)
        ev[s][1].record()
    torch.cuda.synchronize()
    assert all(kev.kev_read_status(c["st"]) == 0 for c in copies)
    second_ms = statistics.mean(x.elapsed_time(y) for x, y in ev)
    useful = RL.prefill_useful_flops(w.lengths, w.h_q, w.d)
    second = RL.prefill_useful_flops(L, w.h_q, w.d) - RL.prefill_useful_flops(cut, w.h_q, w.d)
    return {"workload": "qwen25_7b_prefill batch as two chunks per question (cut at the last 128-row boundary at or "
                        "below half), the second reading the first from the slot", "unit": "TFLOP/s",
            "value": useful / (pair_ms * 1e-3) / 1e12, "ms_per_pair": pair_ms,
            "second_chunk": {"value": second / (second_ms * 1e-3) / 1e12, "ms": second_ms,
                             "useful_gflop": second / 1e9}}


def _sampling(kev, torch, tdev, dev, K, warmup):
    """Per-question temperature sampling of the decode batch: 32 live questions, a 151,936-token
    bf16 vocabulary (Qwen3), temperatures 0.3 .. 1.5, uniforms from a seeded generator; calls back
    to back over two logit buffers (19 MB)."""
    rng = np.random.default_rng(50)
    n, vocab = 32, 151936
    sets = []
    for _ in range(2):
        lg = W.f32_to_bf16_bits(rng.standard_normal((n, vocab), dtype=np.float32) * 2)
        sets.append({"lg": tdev(lg), "t": tdev(rng.choice([0.3, 0.7, 1.0, 1.5], n).astype(np.float32)),
                     "u": tdev(rng.random(n).astype(np.float32)), "a": tdev(np.ones(n, np.uint8)),
                     "tok": torch.empty(n, dtype=torch.int32, device=dev),
                     "st": torch.zeros(1, dtype=torch.int32, device=dev)})

    def call(c):
        kev.kev_sample(c["lg"], n, vocab, "bf16", c["t"], c["u"], c["a"], c["tok"], c["st"])

    for _ in range(warmup):
        for c in sets:
            call(c)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for s in range(K):
        call(sets[s % 2])
    b.record()
    torch.cuda.synchronize()
    assert all(kev.kev_read_status(c["st"]) == 0 for c in sets)
    ms = a.elapsed_time(b) / K
    logit_bytes = n * vocab * 2
    return {"workload": "32 questions x 151,936 bf16 logits, per-question temperatures, inverse CDF",
            "ms_per_step": ms, "value": logit_bytes / (ms * 1e-3) / 1e9, "unit": "GB/s (logits read once)"}


def _lora(kev, torch, tdev, dev, K, warmup):
    """The Qwen2.5-7B-shaped batch (T = 7921) through a 3584 -> 3584 projection's rank-16 LoRA
    adapters (4 adapters over 8 questions, one question without), back to back over two buffer
    sets of x and y (2 x 113 MB)."""
    w = W.qwen25_7b_prefill()
    d, rank, n_ad = 3584, 16, 4
    T, N = w.total_tokens, w.n_questions
    rng = np.random.default_rng(60)
    bf = lambda a: W.f32_to_bf16_bits(a.astype(np.float32))
    shape = kev.make_shape(w.h_q, w.h_kv, w.d, "bf16")
    nb = kev.kev_prefill_workspace_size(N, T, shape)
    A = tdev(bf(rng.standard_normal((n_ad, rank, d)) / np.sqrt(d)))
    B = tdev(bf(rng.standard_normal((n_ad, d, rank)) / np.sqrt(rank)))
    sc = tdev(np.full(n_ad, 2.0, np.float32))
    ids = tdev(np.array([0, 1, 2, 3, -1, 0, 1, 2], np.int32))
    sets = []
    for _ in range(2):
        c = {"x": tdev(bf(rng.standard_normal((T, d)))), "y": tdev(bf(rng.standard_normal((T, d)))),
             "iv": tdev(w.intervals), "ws": torch.empty(nb, dtype=torch.uint8, device=dev),
             "st": torch.zeros(1, dtype=torch.int32, device=dev)}
        kev.kev_build_segments(c["iv"], N, T, None, 0, 0, shape, c["ws"], nb, c["st"])
        sets.append(c)

    def call(c):
        kev.kev_lora_apply(c["x"], c["y"], T, d, d, c["iv"], N, ids, A, B, sc, n_ad, rank, c["ws"], nb, c["st"])

    for _ in range(warmup):
        for c in sets:
            call(c)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for s in range(K):
        call(sets[s % 2])
    b.record()
    torch.cuda.synchronize()
    assert all(kev.kev_read_status(c["st"]) == 0 for c in sets)
    ms = a.elapsed_time(b) / K
    rows = int(sum(L for L, i in zip(w.lengths, [0, 1, 2, 3, -1, 0, 1, 2]) if i >= 0))
    moved = rows * (d + 2 * d) * 2  # x read, y read and written (adapter rows only)
    flops = 2.0 * rows * (d * rank + rank * d)
    return {"workload": "qwen25_7b_prefill batch (T=7921), 3584 x 3584 projection, rank-16 adapters, 7 of 8 "
                        "questions with an adapter", "ms_per_step": ms, "value": moved / (ms * 1e-3) / 1e9,
            "unit": "GB/s", "tflops": flops / (ms * 1e-3) / 1e12}


def _paged_decode(kev, torch, tdev, dev, K, warmup):
    """The decode workload over a paged pool (128-position blocks, block tables from the library's
    host assignment): contiguous-first tables on an empty pool, and scattered tables (a pool with
    every other block taken); calls back to back over two pool sets."""
    dw = W.qwen3_8b_decode()
    N, h_q, h_kv, d, page = dw.n_questions, dw.h_q, dw.h_kv, dw.d, kev.binding.KEV_PAGE
    shape = kev.make_shape(h_q, h_kv, d, "bf16")
    lens = np.asarray(dw.lens)
    live = np.asarray(dw.active).astype(bool)
    need = np.array([(int(n) + 1 + page - 1) // page if a else 0 for n, a in zip(lens, live)], np.int32)
    max_blocks = (dw.cap + page - 1) // page
    dec_bytes = RL.decode_bytes(dw.lens, dw.active, h_q, h_kv, d, 2)
    out = {"workload": DECODE_WORKLOAD + ", copied into 128-position blocks", "unit": "GB/s"}
    for policy in ("contiguous_first", "scattered"):
        if policy == "contiguous_first":
            n_blocks = int(need.sum())
            free = np.ones(n_blocks, np.uint8)
        else:
            n_blocks = 2 * int(need.sum())
            free = (np.arange(n_blocks) % 2).astype(np.uint8)  # every other block already taken
        table = kev.kev_assign_blocks(need, free, max_blocks, contiguous_first=(policy == "contiguous_first"))
        pk = np.zeros((n_blocks, h_kv, page, d), np.uint16)
        pv = np.zeros((n_blocks, h_kv, page, d), np.uint16)
        for i in np.nonzero(live)[0]:
            for b in range(int(need[i])):
                rows = slice(b * page, min((b + 1) * page, dw.cap))
                pk[table[i, b], :, :rows.stop - rows.start] = dw.pool_k[int(dw.slot_ids[i]), :, rows]
                pv[table[i, b], :, :rows.stop - rows.start] = dw.pool_v[int(dw.slot_ids[i]), :, rows]
        nb = kev.kev_decode_workspace_size(N, max_blocks * page, shape)
        copies = []
        for _ in range(DECODE_COPIES):
            copies.append({"pk": tdev(pk), "pv": tdev(pv), "tb": tdev(table), "ln": tdev(lens.astype(np.int32)),
                           "act": tdev(np.asarray(dw.active, np.uint8)), "q": tdev(dw.q_new), "k": tdev(dw.k_new),
                           "v": tdev(dw.v_new),
                           "out": torch.empty((N, h_q, d), dtype=torch.bfloat16, device=dev),
                           "ws": torch.zeros(nb, dtype=torch.uint8, device=dev),
                           "st": torch.zeros(1, dtype=torch.int32, device=dev)})
        del pk, pv

        def call(c):
            kev.kev_decode_attn_paged(c["q"], c["k"], c["v"], c["pk"], c["pv"], n_blocks, c["tb"], max_blocks,
                                      c["ln"], c["act"], N, c["out"], shape, c["ws"], nb, c["st"])

        for _ in range(warmup):
            for c in copies:
                call(c)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for s in range(K):
            call(copies[s % DECODE_COPIES])
        b.record()
        torch.cuda.synchronize()
        assert all(kev.kev_read_status(c["st"]) == 0 for c in copies)
        ms = a.elapsed_time(b) / K
        out[policy] = {"ms_per_step": ms, "value": dec_bytes / (ms * 1e-3) / 1e9, "n_blocks": n_blocks}
        del copies
    return out


def _prefill_qwen3_8b(kev, torch, tdev, dev, K, warmup, tf_peak, peak_src):
    """The Qwen3-8B-shaped batch (T = 24,100) as the workload states it: prefill + slot write.
    One call = kev_prefill_attn (segment build, attention, slot write into [32, 8, 4096, 128]
    pools), back to back over two buffer sets of ~1 GB each (inputs, output, pools), so no call
    finds its inputs in L2.  Also reported: the attention kernel alone over a prebuilt work list."""
    w3 = W.qwen3_8b_prefill()
    N3, T3 = w3.n_questions, w3.total_tokens
    shape3 = kev.make_shape(w3.h_q, w3.h_kv, w3.d, "bf16")
    ws3_bytes = kev.kev_prefill_workspace_size(N3, T3, shape3)
    p3 = []
    for _ in range(2):
        c = {"q": tdev(w3.q), "k": tdev(w3.k), "v": tdev(w3.v), "iv": tdev(w3.intervals), "sl": tdev(w3.slot_ids),
             "out": torch.empty((T3, w3.h_q, w3.d), dtype=torch.bfloat16, device=dev),
             "pk": torch.zeros((w3.n_slots, w3.h_kv, w3.cap, w3.d), dtype=torch.bfloat16, device=dev),
             "ws": torch.empty(ws3_bytes, dtype=torch.uint8, device=dev),
             "st": torch.zeros(1, dtype=torch.int32, device=dev)}
        c["pv"] = torch.zeros_like(c["pk"])
        p3.append(c)
    set_bytes = sum(t.numel() * t.element_size() for t in p3[0].values())

    def call(c):
        kev.kev_prefill_attn(c["q"], c["k"], c["v"], T3, c["iv"], N3, c["sl"], c["pk"], c["pv"], w3.n_slots, w3.cap,
                             c["out"], shape3, c["ws"], ws3_bytes, c["st"])

    def attn_only(c):
        kev.kev_prefill_from_segments(c["q"], c["k"], c["v"], T3, c["iv"], N3, None, None, None, 0, 0, c["out"],
                                      shape3, c["ws"], ws3_bytes, c["st"])

    for fn in (call, attn_only):
        for _ in range(warmup):
            for c in p3:
                fn(c)
    torch.cuda.synchronize()
    assert all(kev.kev_read_status(c["st"]) == 0 for c in p3)
    timed = {}
    for name, fn in (("call", call), ("attn", attn_only)):
        a3, b3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a3.record()
        for it in range(K):
            fn(p3[it % 2])
        b3.record()
        torch.cuda.synchronize()
        timed[name] = a3.elapsed_time(b3) / K
    assert all(kev.kev_read_status(c["st"]) == 0 for c in p3)
    useful3 = RL.prefill_useful_flops(w3.lengths, w3.h_q, w3.d)
    tf = useful3 / (timed["call"] * 1e-3) / 1e12
    tf_attn = useful3 / (timed["attn"] * 1e-3) / 1e12
    del p3
    return {"workload": PREFILL3_WORKLOAD, "value": tf, "unit": "TFLOP/s", "ms_per_call": timed["call"],
            "useful_gflop": useful3 / 1e9,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": tf_peak, "unit": "TFLOP/s", "frac": tf / tf_peak,
                         "kernel": "kev_prefill_attn: segment build + attention + slot write",
                         "peak_source": f"bf16_tflops burst, {peak_src}"},
            "attention_alone": {"value": tf_attn, "ms_per_launch": timed["attn"], "frac": tf_attn / tf_peak},
            "l2": f"not flushed; {K} calls back to back over 2 buffer sets of {set_bytes / 1e6:.0f} MB"}


def _decode_setup(kev, torch, dev, tdev):
    """The decode workload's buffer sets (DECODE_COPIES of them) and its call."""
    dwl = W.qwen3_8b_decode()
    dshape = kev.make_shape(dwl.h_q, dwl.h_kv, dwl.d, "bf16")
    d_bytes = kev.kev_decode_workspace_size(dwl.n_questions, dwl.cap, dshape)
    copies = []
    for _ in range(DECODE_COPIES):
        copies.append({"pk": tdev(dwl.pool_k), "pv": tdev(dwl.pool_v), "sl": tdev(dwl.slot_ids),
                       "ln": tdev(dwl.lens), "act": tdev(dwl.active), "q": tdev(dwl.q_new), "k": tdev(dwl.k_new),
                       "v": tdev(dwl.v_new),
                       "out": torch.empty((dwl.n_questions, dwl.h_q, dwl.d), dtype=torch.bfloat16, device=dev),
                       "ws": torch.zeros(d_bytes, dtype=torch.uint8, device=dev),
                       "st": torch.zeros(1, dtype=torch.int32, device=dev)})

    def dstep(c):
        kev.kev_decode_attn(c["q"], c["k"], c["v"], c["pk"], c["pv"], dwl.n_slots, dwl.cap, c["sl"], c["ln"],
                            c["act"], dwl.n_questions, c["out"], dshape, c["ws"], d_bytes, c["st"])

    return dwl, copies, dstep


def _decode_only(args, kev, torch, dev, tdev):
    """Warm-up and timed loop of the decode workload alone (profiling aid)."""
    _, copies, dstep = _decode_setup(kev, torch, dev, tdev)
    for s in range(args.warmup + args.steps):
        dstep(copies[s % DECODE_COPIES])
    torch.cuda.synchronize()
    assert all(kev.kev_read_status(c["st"]) == 0 for c in copies)
    return None


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="kev", choices=["kev", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["step", "decode", "rope", "sampling", "lora", "stress", "prefill3"],
                    default=None,
                    help="run only one workload's warm-up and timed loop (for profiling); prints no JSON line")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist
    import packed_question_isolated_gb300 as kev

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            dist.barrier()

    def tdev(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        return (t.view(torch.bfloat16) if a.dtype == np.uint16 else t).to(dev)

    # ---- main workload -----------------------------------------------------------------
    w = W.qwen25_7b_prefill()
    shape = kev.make_shape(w.h_q, w.h_kv, w.d, "bf16")
    N, T = w.n_questions, w.total_tokens
    ws_bytes = kev.kev_prefill_workspace_size(N, T, shape)
    dws_bytes = kev.kev_decode_workspace_size(N, w.cap, shape)

    def step_buffers():
        """One full set of the step's device buffers: inputs, outputs, pools and workspaces."""
        c = {"q": tdev(w.q), "k": tdev(w.k), "v": tdev(w.v), "iv": tdev(w.intervals), "sl": tdev(w.slot_ids),
             "qn": tdev(w.q_new), "kn": tdev(w.k_new), "vn": tdev(w.v_new), "ln": tdev(w.lengths),
             "act": torch.ones(N, dtype=torch.uint8, device=dev)}
        c["out"] = torch.empty((T, w.h_q, w.d), dtype=torch.bfloat16, device=dev)
        c["on"] = torch.empty((N, w.h_q, w.d), dtype=torch.bfloat16, device=dev)
        c["pk"] = torch.zeros((w.n_slots, w.h_kv, w.cap, w.d), dtype=torch.bfloat16, device=dev)
        c["pv"] = torch.zeros_like(c["pk"])
        c["ws"] = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        c["st"] = torch.zeros(1, dtype=torch.int32, device=dev)
        c["dws"] = torch.zeros(dws_bytes, dtype=torch.uint8, device=dev)
        c["dst"] = torch.zeros(1, dtype=torch.int32, device=dev)
        return c

    def step(c, ev_a=None, ev_b=None):
        kev.kev_build_segments(c["iv"], N, T, c["sl"], w.n_slots, w.cap, shape, c["ws"], ws_bytes, c["st"])
        if ev_a is not None:
            ev_a.record()
        kev.kev_prefill_from_segments(c["q"], c["k"], c["v"], T, c["iv"], N, c["sl"], c["pk"], c["pv"], w.n_slots,
                                      w.cap, c["out"], shape, c["ws"], ws_bytes, c["st"])
        if ev_b is not None:
            ev_b.record()
        kev.kev_decode_attn(c["qn"], c["kn"], c["vn"], c["pk"], c["pv"], w.n_slots, w.cap, c["sl"], c["ln"],
                            c["act"], N, c["on"], shape, c["dws"], dws_bytes, c["dst"])

    def statuses_ok(cs):
        return all(kev.kev_read_status(c["st"]) == 0 and kev.kev_read_status(c["dst"]) == 0 for c in cs)

    if args.only == "decode":
        return _decode_only(args, kev, torch, dev, tdev)
    if args.only == "sampling":
        _sampling(kev, torch, tdev, dev, args.steps, args.warmup)
        return None
    if args.only == "lora":
        _lora(kev, torch, tdev, dev, args.steps, args.warmup)
        return None
    if args.only == "stress":
        _stress_decode_graph(kev, torch, dev, tdev, 1.0, 1.0)
        return None
    if args.only == "prefill3":
        _prefill_qwen3_8b(kev, torch, tdev, dev, args.steps, args.warmup, 1.0, "")
        return None
    # The timed steps run back to back, each on the next of R full sets of buffers: one cycle
    # touches R x ~170 MB, several times the 129 MB L2, so no step finds its inputs in L2.
    copies = [step_buffers() for _ in range(STEP_COPIES)]
    for _ in range(args.warmup):
        for c in copies:
            step(c)
    torch.cuda.synchronize()
    assert statuses_ok(copies)
    # kernels per step, as the library reports them for the calls just made
    launches_per_step = kev.kev_launch_count(2) + kev.kev_launch_count(1) + kev.kev_launch_count(4)
    if args.only == "step":
        for s in range(args.steps):
            step(copies[s % STEP_COPIES])
        torch.cuda.synchronize()
        return None
    if args.only == "rope":
        _rope_step(kev, torch, w, shape, copies, step_buffers, ws_bytes, dws_bytes, args.steps, args.warmup,
                   RL.prefill_useful_flops(w.lengths, w.h_q, w.d), 1.0)
        return None

    K = args.steps
    e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        e_a.record()
        for s in range(K):
            step(copies[s % STEP_COPIES])
        e_b.record()
        torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    assert statuses_ok(copies)
    total_ms = max_over_ranks(e_a.elapsed_time(e_b), world, dev)
    useful = RL.prefill_useful_flops(w.lengths, w.h_q, w.d)
    value = aggregate_rate(useful, K, world, total_ms) / 1e12
    hbm_peak, tf_peak, tf_sust, peak_src = _peaks()
    # the prefill call (attention kernel + slot-write kernel) on its own: the same back-to-back
    # loop with an event pair around each prefill call (the events cost the step ~10 us, so
    # this pass gives the kernel's duration and not the step's)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for s in range(K):
        step(copies[s % STEP_COPIES], ev[s][0], ev[s][1])
    torch.cuda.synchronize()
    attn_avg_ms = statistics.mean(x.elapsed_time(y) for x, y in ev)
    achieved = useful / (attn_avg_ms * 1e-3) / 1e12
    traffic = _traffic("prefill")
    step_bytes = sum(t.numel() * t.element_size() for t in copies[0].values())

    # ---- e2e: host buffers, copies inside the timed region ------------------------------
    # Every step copies its inputs from pinned host memory and its two outputs back.  Three
    # streams overlap step i's compute with step i+1's host-to-device copies and step i-1's
    # device-to-host copies; steps alternate between two device buffer sets and two pinned
    # output sets, and events order each copy after the last use of the buffers it overwrites.
    def pinned(t):
        return t.cpu().pin_memory()
    in_keys = ("q", "k", "v", "iv", "sl", "qn", "kn", "vn", "ln", "act")
    h_in = [pinned(copies[0][x]) for x in in_keys]
    h_outs = [[torch.empty(copies[0]["out"].shape, dtype=copies[0]["out"].dtype, pin_memory=True),
               torch.empty(copies[0]["on"].shape, dtype=copies[0]["on"].dtype, pin_memory=True)] for _ in range(2)]
    h2d = sum(x.numel() * x.element_size() for x in h_in)
    d2h = sum(x.numel() * x.element_size() for x in h_outs[0])
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    s_comp = torch.cuda.current_stream()

    def e2e_run(n_steps):
        ev_in = [torch.cuda.Event() for _ in range(n_steps)]
        ev_comp = [torch.cuda.Event() for _ in range(n_steps)]
        ev_out = [torch.cuda.Event() for _ in range(n_steps)]
        for i in range(n_steps):
            c, ho = copies[i % 2], h_outs[i % 2]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_comp[i - 2])  # step i-2 has finished reading this input set
                for hd, key in zip(h_in, in_keys):
                    c[key].copy_(hd, non_blocking=True)
                ev_in[i].record(s_in)
            s_comp.wait_event(ev_in[i])
            if i >= 2:
                s_comp.wait_event(ev_out[i - 2])  # step i-2's outputs are on the host
            step(c)
            ev_comp[i].record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[i])
                ho[0].copy_(c["out"], non_blocking=True)
                ho[1].copy_(c["on"], non_blocking=True)
                ev_out[i].record(s_out)
        s_comp.wait_stream(s_in)
        s_comp.wait_stream(s_out)

    e2e_run(args.warmup)
    torch.cuda.synchronize()
    assert statuses_ok(copies[:2])
    Ke = max(5, K // 2)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    e0.record()
    e2e_run(Ke)
    e1.record()
    torch.cuda.synchronize()
    assert statuses_ok(copies[:2])
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    e2e_value = aggregate_rate(useful, Ke, world, e2e_ms) / 1e12

    # ---- the same step with rotary position encoding (positions counted per question) ---------
    rope = _rope_step(kev, torch, w, shape, copies, step_buffers, ws_bytes, dws_bytes, K, args.warmup, useful,
                      hbm_peak)

    # ---- decode workload: calls back to back over DECODE_COPIES pools (2 x 178 MB read per cycle) --
    dwl, dcopies, dstep = _decode_setup(kev, torch, dev, tdev)
    for _ in range(args.warmup):
        for c in dcopies:
            dstep(c)
    torch.cuda.synchronize()
    Kd = max(10, K)
    barrier()
    torch.cuda.synchronize()
    d_a, d_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d_a.record()
    for s in range(Kd):
        dstep(dcopies[s % DECODE_COPIES])
    d_b.record()
    torch.cuda.synchronize()
    assert all(kev.kev_read_status(c["st"]) == 0 for c in dcopies)
    dec_ms = d_a.elapsed_time(d_b) / Kd
    dec_bytes = RL.decode_bytes(dwl.lens, dwl.active, dwl.h_q, dwl.h_kv, dwl.d, 2)
    dec_gbs = dec_bytes / (dec_ms * 1e-3) / 1e9  # this GPU's kernel rate (the roofline is per GPU)
    dec_job_gbs = aggregate_rate(dec_bytes, 1, world, max_over_ranks(dec_ms, world, dev)) / 1e9
    dec_traffic = _traffic("decode")
    del dcopies

    paged = _paged_decode(kev, torch, tdev, dev, Kd, args.warmup)
    chunked = _chunked_prefill(kev, torch, tdev, dev, max(10, K // 2), args.warmup)
    sampling = _sampling(kev, torch, tdev, dev, Kd, args.warmup)
    lora = _lora(kev, torch, tdev, dev, Kd, args.warmup)

    # ---- second prefill workload (Qwen3-8B-shaped batch) as the workload states it ----------
    prefill3 = _prefill_qwen3_8b(kev, torch, tdev, dev, max(6, K // 2), args.warmup, tf_peak, peak_src)

    stress = _stress_decode_graph(kev, torch, dev, tdev, tf_peak, hbm_peak)

    cpu = cpu_fair = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline()
        cpu_fair = cpu_fair_baseline()

    if rank == 0:
        clocks = clk.summary()
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "questions_per_gpu": N, "total_tokens_per_gpu": T,
                       "useful_gflop_per_step": useful / 1e9,
                       "l2": (f"not flushed; inputs larger than L2: the {K} steps run back to back, each on the next "
                              f"of {STEP_COPIES} full buffer sets of {step_bytes / 1e6:.0f} MB (inputs, outputs, pools, "
                              "workspaces) used in turn"),
                       "parallelism": f"replicas x{world} (independent question batches)"},
            "clocks": clocks,
            "decode": {"workload": DECODE_WORKLOAD, "value": dec_job_gbs, "unit": "GB/s", "ms_per_step": dec_ms,
                       "l2": (f"not flushed; {Kd} calls back to back over {DECODE_COPIES} pool sets "
                              f"({dec_bytes / 1e6:.0f} MB read per call)"),
                       "roofline": {"bound": "hbm", "achieved": dec_gbs, "peak": hbm_peak, "unit": "GB/s",
                                    "frac": dec_gbs / hbm_peak, "traffic": dec_traffic,
                                    "algorithmic_bytes": dec_bytes, "peak_source": f"hbm_gbs, {peak_src}"}},
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms / Ke,
                    "overlap": "H2D of step i+1 and D2H of step i-1 on their own streams during step i's compute "
                               "(two device buffer sets, two pinned output sets)"},
            "gpu_launches": launches_per_step * K,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": tf_peak, "unit": "TFLOP/s",
                         "frac": achieved / tf_peak, "traffic": traffic,
                         "kernel": "prefill attention (kev_prefill_from_segments)",
                         "peak_source": f"bf16_tflops burst, {peak_src}", "launch_ms": attn_avg_ms},
            "prefill_qwen3_8b": prefill3,
            "rope": rope,
            "paged_decode": paged,
            "chunked_prefill": chunked,
            "sampling": sampling,
            "lora": lora,
            "stress": stress,
            "cpu_baseline": cpu,
            "cpu_fair_baseline": cpu_fair,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
