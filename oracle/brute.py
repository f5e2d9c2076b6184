"""Pure-Python brute force for tiny cases (invariant (d)).

TEST INFRASTRUCTURE ONLY (same rule as ``kev_oracle``: the product path never
imports it).  Deliberately written without NumPy and without any code of
``kev_oracle``: scalar loops over (token, head, key) with ``math.exp``, so
that a vectorisation, indexing or transposition mistake in the NumPy oracle
does not repeat here.

The rule it applies per output element is the same plain definition:
token t of question i attends to every token u of the same question with
u <= t (inference-engine notes, sakurs2.com, §2.1 causal mask; Kev
architecture article, icman.com.cn, §2.3 causal AND isolation), with the
softmax taken relative to the row maximum (§2.4 of the notes).
"""
from __future__ import annotations

import math


def prefill(q, k, v, intervals, scale):
    """q [T][H_q][d], k/v [T][H_kv][d] nested lists of floats -> out [T][H_q][d]."""
    T = len(q)
    h_q = len(q[0]) if T else 0
    h_kv = len(k[0]) if T else 1
    d = len(q[0][0]) if T else 0
    G = h_q // h_kv if h_kv else 1
    owner = [None] * T
    for i, (s, e) in enumerate(intervals):
        for t in range(s, e):
            owner[t] = i
    out = [[[0.0] * d for _ in range(h_q)] for _ in range(T)]
    for t in range(T):
        if owner[t] is None:
            continue
        keys = [u for u in range(t + 1) if owner[u] == owner[t]]
        for h in range(h_q):
            g = h // G
            scores = []
            for u in keys:
                acc = 0.0
                for c in range(d):
                    acc += q[t][h][c] * k[u][g][c]
                scores.append(acc * scale)
            top = max(scores)
            weights = [math.exp(s - top) for s in scores]
            total = sum(weights)
            for c in range(d):
                acc = 0.0
                for w, u in zip(weights, keys):
                    acc += w * v[u][g][c]
                out[t][h][c] = acc / total
    return out


def decode_one(q_row, k_rows, v_rows, scale):
    """One query row against a list of cached K/V rows (all visible)."""
    scores = [sum(a * b for a, b in zip(q_row, kr)) * scale for kr in k_rows]
    top = max(scores)
    weights = [math.exp(s - top) for s in scores]
    total = sum(weights)
    d = len(v_rows[0])
    return [sum(w * vr[c] for w, vr in zip(weights, v_rows)) / total for c in range(d)]


def rope_rows(x, positions, theta):
    """Rotary position encoding, one scalar at a time: x [P][H][d] nested lists,
    positions [P] ints (negative: row unchanged).  Element j < d/2 pairs with
    element j + d/2; the pair turns by the angle p * theta**(-2j/d) (KV-cache
    isolation article, hnwysp.cn, §7.2: the rotation multiplies Q and K)."""
    out = []
    for row, p in zip(x, positions):
        if p < 0:
            out.append([list(hv) for hv in row])
            continue
        new_row = []
        for hv in row:
            d = len(hv)
            half = d // 2
            nv = [0.0] * d
            for j in range(half):
                ang = p * theta ** (-(2.0 * j) / d)
                c, s = math.cos(ang), math.sin(ang)
                a, b = hv[j], hv[j + half]
                nv[j] = a * c - b * s
                nv[j + half] = b * c + a * s
            new_row.append(nv)
        out.append(new_row)
    return out
