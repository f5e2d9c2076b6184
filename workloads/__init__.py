"""Seeded synthetic inputs for packed, question-isolated attention.

This module only *draws* inputs: question lengths, packed intervals, slot
assignments, early-stop schedules and Q/K/V values.  It holds none of the
attention arithmetic, so both the CPU oracle (``oracle/``) and the GPU path
(tests, ``bench.py``) can take their inputs from here without sharing any
compute code.

Every generator uses ``numpy.random.default_rng(seed)`` with a fixed draw
order: lengths, then (decode / stress) cached lengths, active set and
max_new_tokens, then Q, K, V in float32 (scaled where the workload says so),
then rounded to the storage dtype, then the decode step inputs.

bf16 tensors are carried as ``uint16`` bit patterns (round-to-nearest-even
from the float32 draw), so the GPU receives exactly the values the oracle
upcasts to float64.

Workloads (the shapes come from the attention layers of the models named on
the pages: Qwen2.5-7B-Instruct in the Kev architecture article, §5, and
Qwen3-8B in the inference-engine notes, §2.1; the batch of 8 questions of at
most 2048 tokens is the Kev pipeline article's test setup, §1.1 and §3.1):

* ``tiny_fp32``          4 questions, lengths 7/13/5/11, 2/2 heads, d 64, fp32
* ``qwen25_7b_prefill``  8 questions, lengths U{256..2048}, 28/4 heads, d 128, bf16
* ``qwen3_8b_prefill``   32 questions, log-normal lengths, 32/8 heads, d 128, bf16
* ``qwen3_8b_decode``    64-slot pool of cap 2458, 32 of 64 questions live
* ``stress``             256 questions, Pareto lengths, prefill + 128 decode steps
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

__all__ = [
    "Workload", "DecodeWorkload", "StressWorkload",
    "f32_to_bf16_bits", "bf16_bits_to_f32", "to_float64",
    "pack_intervals", "random_case", "tiny_fp32", "qwen25_7b_prefill",
    "qwen3_8b_prefill", "qwen3_8b_decode", "stress", "by_name",
]


# ---------------------------------------------------------------------------
# storage-type helpers (bit handling only)
# ---------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return the bits as uint16."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def to_float64(arr: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 value of a stored tensor (``dtype`` is 'bf16', 'fp32' or 'fp64')."""
    if dtype == "bf16":
        return bf16_bits_to_f32(arr).astype(np.float64)
    if dtype == "fp32":
        return np.asarray(arr, dtype=np.float32).astype(np.float64)
    if dtype == "fp64":
        return np.asarray(arr, dtype=np.float64)
    raise ValueError(dtype)


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_bf16_bits(x) if dtype == "bf16" else np.ascontiguousarray(x, dtype=np.float32)


def pack_intervals(lengths, gaps=None) -> np.ndarray:
    """Half-open intervals [s_i, e_i) of questions laid end to end.

    ``gaps[i]`` tokens (boundary / padding tokens that belong to no question)
    are placed *before* question i when given.
    """
    lengths = np.asarray(lengths, dtype=np.int64)
    out = np.zeros((len(lengths), 2), dtype=np.int32)
    pos = 0
    for i, n in enumerate(lengths):
        if gaps is not None:
            pos += int(gaps[i])
        out[i] = (pos, pos + int(n))
        pos += int(n)
    return out


# ---------------------------------------------------------------------------
# workload records
# ---------------------------------------------------------------------------

@dataclass
class Workload:
    """One packed prefill batch (+ optionally one decode step for every question)."""
    name: str
    seed: int
    dtype: str                 # 'bf16' | 'fp32'
    h_q: int
    h_kv: int
    d: int
    lengths: np.ndarray        # int32 [N]
    intervals: np.ndarray      # int32 [N, 2], half-open, packed-token indices
    total_tokens: int          # T
    q: np.ndarray              # [T, h_q, d]   (uint16 bf16 bits or float32)
    k: np.ndarray              # [T, h_kv, d]
    v: np.ndarray              # [T, h_kv, d]
    slot_ids: np.ndarray       # int32 [N]
    n_slots: int
    cap: int
    # one decode step appended after prefill (lens = lengths, every question live)
    q_new: Optional[np.ndarray] = None   # [N, h_q, d]
    k_new: Optional[np.ndarray] = None   # [N, h_kv, d]
    v_new: Optional[np.ndarray] = None   # [N, h_kv, d]
    scale: float = 0.0                   # 0 => 1/sqrt(d)

    @property
    def n_questions(self) -> int:
        return int(len(self.lengths))


@dataclass
class DecodeWorkload:
    """One decode step over a pre-filled slot pool."""
    name: str
    seed: int
    dtype: str
    h_q: int
    h_kv: int
    d: int
    n_slots: int
    cap: int
    pool_k: np.ndarray         # [n_slots, h_kv, cap, d]
    pool_v: np.ndarray
    slot_ids: np.ndarray       # int32 [N]
    lens: np.ndarray           # int32 [N]  cached length before the step
    active: np.ndarray         # uint8 [N]  0 = early-stopped, dropped from the step
    q_new: np.ndarray          # [N, h_q, d]
    k_new: np.ndarray          # [N, h_kv, d]
    v_new: np.ndarray          # [N, h_kv, d]
    scale: float = 0.0

    @property
    def n_questions(self) -> int:
        return int(len(self.lens))


@dataclass
class StressWorkload:
    """Prefill of many short questions, then a decode loop with early stop."""
    prefill: Workload
    max_new: np.ndarray        # int32 [N]  per-question max_new_tokens
    eos: np.ndarray            # bool [steps, N]  EOS drawn after the token of that step
    n_steps: int
    n_decoded: np.ndarray      # int32 [N]  steps each question takes part in
    _rng_state: dict = field(default_factory=dict, repr=False)

    def active_at(self, step: int) -> np.ndarray:
        """uint8 [N]: 1 if the question still takes part in decode step ``step``."""
        return (self.n_decoded > step).astype(np.uint8)

    def lens_at(self, step: int) -> np.ndarray:
        """Cached length of every question before decode step ``step`` (live or not)."""
        done = np.minimum(self.n_decoded, step)
        return (self.prefill.lengths + done).astype(np.int32)

    def step_inputs(self, step: int):
        """(q_new, k_new, v_new) of decode step ``step`` (drawn for every question)."""
        w = self.prefill
        rng = np.random.default_rng([w.seed, 1000 + step])
        n = w.n_questions
        q = rng.standard_normal((n, w.h_q, w.d), dtype=np.float32)
        k = rng.standard_normal((n, w.h_kv, w.d), dtype=np.float32)
        v = rng.standard_normal((n, w.h_kv, w.d), dtype=np.float32)
        return _store(q, w.dtype), _store(k, w.dtype), _store(v, w.dtype)


# ---------------------------------------------------------------------------
# generators
# ---------------------------------------------------------------------------

def _draw_qkv(rng, T, h_q, h_kv, d, dtype, mul=1.0):
    q = rng.standard_normal((T, h_q, d), dtype=np.float32)
    k = rng.standard_normal((T, h_kv, d), dtype=np.float32)
    v = rng.standard_normal((T, h_kv, d), dtype=np.float32)
    if mul != 1.0:
        m = np.float32(mul)
        q *= m
        k *= m
        v *= m
    return _store(q, dtype), _store(k, dtype), _store(v, dtype)


def _draw_new(rng, n, h_q, h_kv, d, dtype, mul=1.0):
    q = rng.standard_normal((n, h_q, d), dtype=np.float32)
    k = rng.standard_normal((n, h_kv, d), dtype=np.float32)
    v = rng.standard_normal((n, h_kv, d), dtype=np.float32)
    if mul != 1.0:
        m = np.float32(mul)
        q *= m
        k *= m
        v *= m
    return _store(q, dtype), _store(k, dtype), _store(v, dtype)


def _prefill_workload(name, seed, rng, lengths, h_q, h_kv, d, dtype, cap, n_slots=None,
                      slot_ids=None, gaps=None, mul=1.0, tail=0, decode=True):
    lengths = np.asarray(lengths, dtype=np.int32)
    intervals = pack_intervals(lengths, gaps)
    T = int(intervals[:, 1].max()) + int(tail) if len(lengths) else int(tail)
    q, k, v = _draw_qkv(rng, T, h_q, h_kv, d, dtype, mul)
    n = len(lengths)
    if n_slots is None:
        n_slots = n
    if slot_ids is None:
        slot_ids = np.arange(n, dtype=np.int32)
    w = Workload(name=name, seed=seed, dtype=dtype, h_q=h_q, h_kv=h_kv, d=d,
                 lengths=lengths, intervals=intervals, total_tokens=T,
                 q=q, k=k, v=v, slot_ids=np.asarray(slot_ids, dtype=np.int32),
                 n_slots=int(n_slots), cap=int(cap))
    if decode:
        w.q_new, w.k_new, w.v_new = _draw_new(rng, n, h_q, h_kv, d, dtype, mul)
    return w


def tiny_fp32() -> Workload:
    """4 questions of 7/13/5/11 tokens (T=36), 2 q-heads / 2 kv-heads, d=64, float32, cap 16."""
    rng = np.random.default_rng(1)
    return _prefill_workload("tiny_fp32", 1, rng, [7, 13, 5, 11], 2, 2, 64, "fp32", cap=16)


def qwen25_7b_prefill() -> Workload:
    """Qwen2.5-7B-shaped layer: 8 questions, lengths U{256..2048}, 28/4 heads, d 128, bf16.

    Q, K and V are N(0,1) draws multiplied by 1/sqrt(d) before rounding; slot cap 2458.
    """
    rng = np.random.default_rng(2)
    lengths = rng.integers(256, 2049, size=8)
    return _prefill_workload("qwen25_7b_prefill", 2, rng, lengths, 28, 4, 128, "bf16",
                             cap=2458, mul=1.0 / np.sqrt(128.0))


def qwen3_8b_prefill() -> Workload:
    """Qwen3-8B-shaped layer: 32 questions, lengths clip(rint(exp(N(ln 512, 0.8))), 1, 4096)."""
    rng = np.random.default_rng(3)
    lengths = np.clip(np.rint(np.exp(rng.normal(np.log(512.0), 0.8, size=32))), 1, 4096)
    return _prefill_workload("qwen3_8b_prefill", 3, rng, lengths.astype(np.int32), 32, 8, 128,
                             "bf16", cap=4096)


def qwen3_8b_decode(n_slots: int = 64, cap: int = 2458, n_live: int = 32) -> DecodeWorkload:
    """One decode step: [64, 8, 2458, 128] bf16 pools, lens U{64..2400}, 32 of 64 questions live.

    Slot ``slot_ids[i]`` of question i is a seeded permutation of the pool, so the
    kernel's indirection is exercised.  Pool contents are N(0,1).
    """
    rng = np.random.default_rng(4)
    h_q, h_kv, d, dtype = 32, 8, 128, "bf16"
    n = n_slots
    lens = rng.integers(64, 2401, size=n).astype(np.int32)
    active = (rng.permutation(n) < n_live).astype(np.uint8)
    slot_ids = rng.permutation(n_slots).astype(np.int32)[:n]
    pool_k = f32_to_bf16_bits(rng.standard_normal((n_slots, h_kv, cap, d), dtype=np.float32))
    pool_v = f32_to_bf16_bits(rng.standard_normal((n_slots, h_kv, cap, d), dtype=np.float32))
    q_new, k_new, v_new = _draw_new(rng, n, h_q, h_kv, d, dtype)
    return DecodeWorkload(name="qwen3_8b_decode", seed=4, dtype=dtype, h_q=h_q, h_kv=h_kv, d=d,
                          n_slots=n_slots, cap=cap, pool_k=pool_k, pool_v=pool_v,
                          slot_ids=slot_ids, lens=lens, active=active,
                          q_new=q_new, k_new=k_new, v_new=v_new)


def stress(n_steps: int = 128) -> StressWorkload:
    """256 questions, L = min(4096, floor(32 (1 + Lomax(1.5)))), 32/8 heads, d 128, cap 4224.

    max_new_tokens ~ U{8..128}; after every produced token a question stops with
    probability 0.02 (EOS).  A question that draws EOS at step t has produced the
    token of step t and is dropped from step t+1 on; it also stops after
    max_new_tokens steps.
    """
    seed = 5
    rng = np.random.default_rng(seed)
    n = 256
    lengths = np.minimum(4096, np.floor(32 * (1 + rng.pareto(1.5, size=n)))).astype(np.int32)
    max_new = rng.integers(8, 129, size=n).astype(np.int32)
    eos = rng.random((n_steps, n)) < 0.02
    first_eos = np.where(eos.any(0), eos.argmax(0) + 1, np.iinfo(np.int32).max)
    n_decoded = np.minimum(np.minimum(max_new, first_eos), n_steps).astype(np.int32)
    cap = 4096 + 128
    w = _prefill_workload("stress", seed, rng, lengths, 32, 8, 128, "bf16", cap=cap, decode=False)
    return StressWorkload(prefill=w, max_new=max_new, eos=eos, n_steps=n_steps, n_decoded=n_decoded)


def random_case(seed: int, lengths, h_q: int, h_kv: int, d: int, dtype: str = "bf16", *,
                gaps=None, tail: int = 0, cap: Optional[int] = None, n_slots: Optional[int] = None,
                permute_slots: bool = False, order=None, mul: float = 1.0) -> Workload:
    """Small seeded case for tests.

    ``gaps`` puts tokens that belong to no question before each interval,
    ``tail`` adds such tokens at the end, ``order`` lists the intervals in a
    different order than their positions (the packing order need not be
    sorted), ``permute_slots`` assigns a seeded permutation of slots.
    """
    rng = np.random.default_rng(seed)
    lengths = np.asarray(lengths, dtype=np.int32)
    n = len(lengths)
    if cap is None:
        cap = int(lengths.max()) + 1 if n else 1
    if n_slots is None:
        n_slots = n
    slot_ids = (rng.permutation(n_slots)[:n] if permute_slots else np.arange(n)).astype(np.int32)
    w = _prefill_workload(f"random{seed}", seed, rng, lengths, h_q, h_kv, d, dtype, cap,
                          n_slots=n_slots, slot_ids=slot_ids, gaps=gaps, mul=mul, tail=tail)
    if order is not None:
        order = np.asarray(order)
        w.lengths = w.lengths[order]
        w.intervals = w.intervals[order]
        w.slot_ids = w.slot_ids[order]
        w.q_new, w.k_new, w.v_new = w.q_new[order], w.k_new[order], w.v_new[order]
    return w


def by_name(name: str):
    return {
        "tiny_fp32": tiny_fp32,
        "qwen25_7b_prefill": qwen25_7b_prefill,
        "qwen3_8b_prefill": qwen3_8b_prefill,
        "qwen3_8b_decode": qwen3_8b_decode,
        "stress": stress,
    }[name]()
