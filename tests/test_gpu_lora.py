"""GPU parity of token-grouped LoRA against the CPU oracle: several adapters (shared, absent),
ranks 16 / 32 / 64, the Qwen2.5-7B-shaped projection on sampled rows, and the adapter-id error
that must write nothing.

Tolerance, from the kernel's arithmetic (bf16 operands, fp32 accumulation): h = scale x A^T is
accumulated in fp32 over d_in products (at most d_in 2^-24 sum_k |x_k A_rk| off, the worst-case
bound of a sum of that length) and rounded to bf16 for the second product (bf16 keeps 8
significant bits, so round-to-nearest moves it by at most the unit roundoff 2^-8 |h_r|); the new
y is rounded once to bf16 (half a unit in the last place of the larger of the computed and exact
values).  So per element
  |got - ref| <= ulp(max(|ref|, |got|)) / 2 + sum_r |B[col, r]| (2^-8 |h_r| + d_in 2^-24 h1_r) + 1e-5,
h1_r = scale sum_k |x_k| |A_rk|, all in float64; the relative L2 error over all elements stays
within 5e-3."""
import numpy as np
import pytest
import torch

import packed_question_isolated_gb300 as kev
import workloads as W
from oracle import kev_oracle as O

from kev_harness import TOL_BF16_REL_L2, dev, f64, host

pytestmark = pytest.mark.gpu


def _case(seed, lengths, d_in, d_out, rank, n_ad, gaps=None, tail=0):
    rng = np.random.default_rng(seed)
    iv = W.pack_intervals(lengths, gaps=gaps).astype(np.int32)
    T = int(iv[-1, 1]) + tail
    bf = lambda a: W.f32_to_bf16_bits(a.astype(np.float32))
    x = bf(rng.standard_normal((T, d_in)))
    y = bf(rng.standard_normal((T, d_out)))
    A = bf(rng.standard_normal((n_ad, rank, d_in)) / np.sqrt(d_in))
    B = bf(rng.standard_normal((n_ad, d_out, rank)) / np.sqrt(rank))
    scales = (rng.random(n_ad) + 0.5).astype(np.float32)
    return iv, T, x, y, A, B, scales


def _assert_lora_close(got, ref, x64, iv, ids, A64, B64, scales, what):
    bound = np.zeros_like(ref)
    mag = np.maximum(np.abs(ref), np.abs(got))
    ulp_half = np.ldexp(1.0, (np.floor(np.log2(np.maximum(mag, 1e-30))) - 8).astype(int))
    d_in = x64.shape[1]
    for (s, e), a in zip(iv, ids):
        if a < 0 or e <= s:
            continue
        sc = abs(float(scales[a]))
        h = sc * np.abs(x64[s:e] @ A64[a].T)          # [rows, r]
        h1 = sc * np.abs(x64[s:e]) @ np.abs(A64[a]).T  # sum_k |x_k| |A_rk|
        bound[s:e] = (2.0 ** -8 * h + d_in * 2.0 ** -24 * h1) @ np.abs(B64[a]).T
    bound += ulp_half + 1e-5
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert (err <= bound).all(), f"{what}: {int((err > bound).sum())} elements beyond the rounding bound"
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))
    assert rel <= TOL_BF16_REL_L2, f"{what}: rel L2 {rel:.3e}"


def _run(iv, T, x, y, A, B, scales, ids, rank, d_in, d_out, n_ad):
    n = len(iv)
    shape = kev.make_shape(1, 1, 128, "bf16")  # any shape: only the intervals' cu_seqlens are used
    nb = kev.kev_prefill_workspace_size(n, T, shape)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    div = torch.from_numpy(np.ascontiguousarray(iv)).cuda()
    kev.kev_build_segments(div, n, T, None, 0, 0, shape, ws, nb, st)
    dy = dev(y)
    kev.kev_lora_apply(dev(x), dy, T, d_in, d_out, div, n, torch.tensor(ids, dtype=torch.int32).cuda(), dev(A),
                       dev(B), torch.from_numpy(scales).cuda(), n_ad, rank, ws, nb, st)
    return kev.kev_read_status(st), dy


@pytest.mark.parametrize("rank", [16, 32, 64])
def test_lora_against_oracle(rank):
    lengths, d_in, d_out, n_ad = [70, 129, 0, 64, 33], 256, 192, 3
    iv, T, x, y, A, B, sc = _case(80 + rank, lengths, d_in, d_out, rank, n_ad, gaps=[1, 0, 2, 0, 1], tail=3)
    ids = [2, -1, 0, 0, 1]  # two questions share adapter 0, one has none
    status, dy = _run(iv, T, x, y, A, B, sc, ids, rank, d_in, d_out, n_ad)
    assert status == 0
    x64, A64, B64 = W.to_float64(x, "bf16"), W.to_float64(A, "bf16"), W.to_float64(B, "bf16")
    ref = O.lora_apply(W.to_float64(y, "bf16"), x64, iv, ids, A64, B64, sc.astype(np.float64))
    got = f64(dy, "bf16")
    _assert_lora_close(got, ref, x64, iv, ids, A64, B64, sc, f"lora rank {rank}")
    untouched = np.ones(T, bool)
    for (s, e), a in zip(iv, ids):
        if a >= 0:
            untouched[s:e] = False
    np.testing.assert_array_equal(host(dy)[untouched], y[untouched])  # no adapter, gaps: bit for bit


@pytest.mark.parametrize("rank", [16, 64])
def test_lora_smallest_dimensions(rank):
    """d_in 64 and d_out 32 (one chunk each, fewer 32-column blocks than warps), one-row questions
    and a question whose last tile has a single row."""
    lengths, d_in, d_out, n_ad = [1, 17, 1, 40], 64, 32, 2
    iv, T, x, y, A, B, sc = _case(120 + rank, lengths, d_in, d_out, rank, n_ad, gaps=[0, 1, 0, 3], tail=1)
    ids = [0, 1, 1, 0]
    status, dy = _run(iv, T, x, y, A, B, sc, ids, rank, d_in, d_out, n_ad)
    assert status == 0
    x64, A64, B64 = W.to_float64(x, "bf16"), W.to_float64(A, "bf16"), W.to_float64(B, "bf16")
    ref = O.lora_apply(W.to_float64(y, "bf16"), x64, iv, ids, A64, B64, sc.astype(np.float64))
    _assert_lora_close(f64(dy, "bf16"), ref, x64, iv, ids, A64, B64, sc, f"lora small rank {rank}")
    untouched = np.ones(T, bool)
    for s, e in iv:
        untouched[s:e] = False
    np.testing.assert_array_equal(host(dy)[untouched], y[untouched])


def test_lora_most_questions():
    """4096 questions of 1 to 40 rows (the most a call takes), adapters drawn at random, some
    questions without one."""
    rng = np.random.default_rng(130)
    n, d_in, d_out, rank, n_ad = 4096, 64, 64, 16, 5
    lengths = rng.integers(1, 41, n).tolist()
    iv, T, x, y, A, B, sc = _case(131, lengths, d_in, d_out, rank, n_ad)
    ids = rng.integers(-1, n_ad, n).tolist()
    status, dy = _run(iv, T, x, y, A, B, sc, ids, rank, d_in, d_out, n_ad)
    assert status == 0
    x64, A64, B64 = W.to_float64(x, "bf16"), W.to_float64(A, "bf16"), W.to_float64(B, "bf16")
    ref = O.lora_apply(W.to_float64(y, "bf16"), x64, iv, ids, A64, B64, sc.astype(np.float64))
    _assert_lora_close(f64(dy, "bf16"), ref, x64, iv, ids, A64, B64, sc, "lora 4096 questions")


def test_lora_qwen25_7b_projection_sampled_rows():
    """The Qwen2.5-7B-shaped batch through a 3584 -> 3584 projection's rank-16 adapters: 4 adapters
    over 8 questions (one without), sampled rows against the oracle."""
    w = W.qwen25_7b_prefill()
    d, rank, n_ad = 3584, 16, 4
    rng = np.random.default_rng(90)
    iv = np.asarray(w.intervals, np.int32)
    T = w.total_tokens
    bf = lambda a: W.f32_to_bf16_bits(a.astype(np.float32))
    x = bf(rng.standard_normal((T, d)))
    y = bf(rng.standard_normal((T, d)))
    A = bf(rng.standard_normal((n_ad, rank, d)) / np.sqrt(d))
    B = bf(rng.standard_normal((n_ad, d, rank)) / np.sqrt(rank))
    sc = np.full(n_ad, 2.0, np.float32)  # alpha 32 over rank 16
    ids = [0, 1, 2, 3, -1, 0, 1, 2]
    status, dy = _run(iv, T, x, y, A, B, sc, ids, rank, d, d, n_ad)
    assert status == 0
    rows = sorted({int(s) for s, _ in iv} | {int(e) - 1 for _, e in iv} |
                  set(rng.integers(0, T, 64).tolist()))
    sub = np.zeros(T, bool)
    sub[rows] = True
    # the oracle on the sampled rows: every row is independent
    x64, A64, B64 = W.to_float64(x, "bf16")[sub], W.to_float64(A, "bf16"), W.to_float64(B, "bf16")
    (riv,) = _restrict(iv, rows)
    ref = O.lora_apply(W.to_float64(y, "bf16")[sub], x64, riv, ids, A64, B64, sc.astype(np.float64))
    _assert_lora_close(f64(dy, "bf16")[rows], ref, x64, riv, ids, A64, B64, sc, "lora qwen25 rows")


def _restrict(iv, rows):
    """Intervals over the sampled rows (in order): question i keeps its sampled rows."""
    rows = np.asarray(rows)
    out, pos = [], 0
    for s, e in iv:
        k = int(((rows >= s) & (rows < e)).sum())
        out.append((pos, pos + k))
        pos += k
    return (np.array(out, np.int32),)


def test_lora_bad_adapter_id_writes_nothing():
    iv, T, x, y, A, B, sc = _case(95, [40, 50], 128, 64, 16, 2)
    assert O.validate_lora([0, 2], 2) == O.ADAPTER
    status, dy = _run(iv, T, x, y, A, B, sc, [0, 2], 16, 128, 64, 2)
    assert status == kev.binding.KEV_ERR_ADAPTER
    np.testing.assert_array_equal(host(dy), y)
