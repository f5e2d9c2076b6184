"""Work and roofline accounting for the measurement harness.

The roofline is the one on the inference-engine notes (sakurs2.com), §2.3:
arithmetic intensity I = F / D and the ideal time t = max(F / P, D / beta),
with F the operations, D the bytes moved, P the peak compute and beta the
peak memory bandwidth.

Algorithmic work counted for this path:

* prefill useful FLOPs = sum_i 2 * d * H_q * L_i * (L_i + 1): 4 d FLOPs (QK^T and
  PV multiply-adds) per allowed (query, key, head) pair, of which question i
  has L_i (L_i + 1) / 2.  Masked work, softmax and exponentials are not counted.
* prefill bytes = T (2 H_q + 4 H_kv) d * elem: read Q, K, V, write O and the
  two slot-pool rows.
* decode bytes = sum over live questions of 2 H_kv lens_i d elem (cached K, V)
  + 2 H_kv d elem (new K/V row) + 2 H_q d elem (query in, output out);
  dropped questions count zero.
* prefill-side RoPE bytes = sum_i L_i (2 H_q + 5 H_kv) d elem: q and k rows
  of question tokens read and written back rotated, and (with a slot pool)
  the v row read plus the rotated k row and the v row written to the slot.
"""
from __future__ import annotations

import numpy as np


def arithmetic_intensity(flops: float, bytes_moved: float) -> float:
    return float(flops) / float(bytes_moved)


def projection_intensity(n: int, d: int, bytes_per_value: int) -> float:
    """Intensity of a d x d projection over n positions (weight and input read, output written)."""
    flops = 2 * n * d * d
    moved = (d * d + 2 * n * d) * bytes_per_value
    return arithmetic_intensity(flops, moved)


def ideal_time(flops: float, bytes_moved: float, peak_flops: float, peak_bytes_per_s: float) -> float:
    return max(float(flops) / peak_flops, float(bytes_moved) / peak_bytes_per_s)


def prefill_useful_flops(lengths, h_q: int, d: int) -> float:
    L = np.asarray(lengths, dtype=np.float64)
    return float(np.sum(2.0 * d * h_q * L * (L + 1.0)))


def prefill_bytes(total_tokens: int, h_q: int, h_kv: int, d: int, elem: int) -> float:
    return float(total_tokens) * (2 * h_q + 4 * h_kv) * d * elem


def decode_bytes(lens, active, h_q: int, h_kv: int, d: int, elem: int) -> float:
    lens = np.asarray(lens, dtype=np.float64)
    live = np.asarray(active).astype(bool)
    per = 2.0 * h_kv * lens * d * elem + 2.0 * h_kv * d * elem + 2.0 * h_q * d * elem
    return float(np.sum(per[live]))


def rope_prefill_bytes(lengths, h_q: int, h_kv: int, d: int, elem: int, slots: bool = True) -> float:
    tokens = float(np.sum(np.asarray(lengths, dtype=np.float64)))
    per_token = 2 * (h_q + h_kv) + (3 * h_kv if slots else 0)
    return tokens * per_token * d * elem
