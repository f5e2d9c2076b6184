"""CPU float64 oracle for packed, question-isolated attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
link this module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline legs of ``bench.py`` use it.  It shares no code with the CUDA
library (no kernels, headers, helpers, tables or constants); its only
common dependency with the GPU side is the seeded input module
``workloads`` (which draws numbers and holds none of the arithmetic).

What it computes is the plain definition, written out with an explicit
dense T x T mask, in float64:

* Attention (inference-engine notes, sakurs2.com, §2.1, the Z = softmax(QK^T /
  sqrt(d_h) + M) V equation and its causal mask M_ij = 0 for j <= i, -inf
  otherwise); the softmax is taken in its stable form, subtracting the row
  maximum (same page, §2.4, the p_i = e^{s_i - m} / sum_j e^{s_j - m} equation).
* Isolation (Kev architecture article, icman.com.cn, §2.1 end and §2.3: each
  question owns one contiguous interval, the isolation mask is block
  diagonal and is combined with the causal mask by a logical AND; Kev
  pipeline article, gsyq.cn, §2.2: attention stays inside the question's
  visible domain, causal within it, and crosses no boundary).
* KV slot pool (Kev pipeline article, §2.2: a preallocated pool cut into
  fixed-size slots, one slot per question).
* Decode with a cache (inference-engine notes, §2.2: only K/V are cached, the
  new K/V row is appended and the new query attends to every cached
  position plus itself, with no mask; the result equals the last row of a
  full recompute).
* Early stop (Kev pipeline article, §1.2 and §2.3: a question that has
  finished takes no further part in attention).
* Paged slot pool (inference-engine notes, §2.5: K/V kept in fixed-size
  blocks allocated on demand, a block table records where each block is and
  attention reads K/V through it; Kev pipeline article, §4.3: blocks of one
  batch placed at neighbouring addresses first).
* Chunked prefill into slots (inference-engine notes, §2.6: a long input is
  prefilled in pieces that share rounds with decode steps, each later piece
  using the K/V of the pieces before it).
* Per-question temperature sampling (Kev architecture article, §4.1: each
  question brings its own temperature, applied to the softmax of its logits
  at every decode step; nothing else in the model changes).
* Token-grouped LoRA (Kev architecture article, §3.2: the base layer stays
  fixed and each token takes the low-rank delta of its own question's
  adapter, computed per adapter group rather than for every adapter over the
  whole sequence; §3.3: the scale is the adapter's alpha / rank).
* Rotary position encoding with per-question positions (KV-cache isolation
  article, hnwysp.cn, §7.2: the rotation multiplies Q and K, a cached K
  keeps the rotation of its own position, and the new token's position is
  the cache length counted from 0).  Packed with isolation, every question
  counts its positions from 0 as if it ran alone.

Readings taken where the pages are silent or garbled (each listed in the
design notes): intervals are half-open [s, e); scale = 1/sqrt(d_h) unless
given; a q-head h uses kv-head h // (H_q / H_kv); tokens in no interval are
keys for nobody and their own output row is 0; an empty interval is allowed;
a decode step attends over lens + 1 positions, the new K/V written first;
sampling takes token k, the smallest index whose cumulative probability under
softmax(logits / T_i) exceeds the question's uniform u_i in [0, 1) (inverse
CDF; the uniforms are inputs), and T_i = 0 means the greedy argmax, ties to
the lowest index;
RoPE is the rotate-half form (pair (x_i, x_{i+d/2}) turned by p * w_i with
w_i = theta^(-2i/d), theta given by the caller), the position of token t of
question i is t - s_i, that of a decode token is lens_i, tokens in no
question are not rotated.

Pinned by ``tests/test_oracle.py`` against the pages' worked example, closed
forms, invariants (a)-(d), a library routine and a pure-Python brute force.
"""
from __future__ import annotations

import numpy as np

from workloads import to_float64

# Error kinds, in the order they are checked.
INTERVALS = "intervals"
SLOT = "slot"
SLOT_OVERFLOW = "slot_overflow"
PREFIX = "prefix"


# ---------------------------------------------------------------------------
# mask
# ---------------------------------------------------------------------------

def segment_ids(intervals, total_tokens: int) -> np.ndarray:
    """seg[t] = i if t lies in question i's interval [s_i, e_i), else -1."""
    seg = np.full(int(total_tokens), -1, dtype=np.int64)
    for i, (s, e) in enumerate(np.asarray(intervals, dtype=np.int64).reshape(-1, 2)):
        seg[s:e] = i
    return seg


def allowed_mask(intervals, total_tokens: int) -> np.ndarray:
    """Boolean T x T mask: row t may attend to column u.

    The causal lower triangle (u <= t) AND the block-diagonal isolation
    mask (same question); a token in no question is allowed nothing.
    """
    T = int(total_tokens)
    causal = np.tril(np.ones((T, T), dtype=bool))
    iso = np.zeros((T, T), dtype=bool)
    for s, e in np.asarray(intervals, dtype=np.int64).reshape(-1, 2):
        iso[s:e, s:e] = True
    return causal & iso


def additive_mask(allowed: np.ndarray) -> np.ndarray:
    """The additive form of the same mask: 0 where allowed, -inf where blocked."""
    m = np.full(allowed.shape, -np.inf, dtype=np.float64)
    m[allowed] = 0.0
    return m


def _check_forms_agree(allowed: np.ndarray, add: np.ndarray) -> None:
    # A 0/1 mask handed to code that expects an additive mask fails silently
    # (Kev architecture article, §2.3 end); both forms must say the same.
    if not np.array_equal(np.isfinite(add), allowed):
        raise AssertionError("boolean and additive masks disagree")


# ---------------------------------------------------------------------------
# softmax
# ---------------------------------------------------------------------------

def softmax_rows(scores: np.ndarray) -> np.ndarray:
    """Row softmax in the stable form exp(s - max) / sum exp(s - max).

    A row whose entries are all -inf (a token that may attend to nothing)
    gets all-zero weights.
    """
    m = np.max(scores, axis=-1, keepdims=True)
    empty = ~np.isfinite(m)
    m = np.where(empty, 0.0, m)
    w = np.exp(scores - m)
    z = np.sum(w, axis=-1, keepdims=True)
    z = np.where(empty, 1.0, z)
    return w / z


def online_softmax_row(q_row, k, v, scale: float, block: int):
    """One query row processed block by block with a running max m, sum l and
    weighted sum u, each block rescaling the old state by alpha = exp(m_old - m_new)
    (inference-engine notes, §2.4, online softmax).

    Returns (output, list of alpha values, one per block).  Equal to the
    plain softmax up to rounding; kept here to pin the kernel's algorithm
    against the page's worked example.
    """
    q_row = np.asarray(q_row, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    m = -np.inf
    ell = 0.0
    u = np.zeros(v.shape[-1], dtype=np.float64)
    alphas = []
    for start in range(0, k.shape[0], block):
        s = (k[start:start + block] @ q_row) * scale
        m_new = max(m, float(np.max(s)))
        alpha = np.exp(m - m_new)
        w = np.exp(s - m_new)
        ell = alpha * ell + float(np.sum(w))
        u = alpha * u + w @ v[start:start + block]
        m = m_new
        alphas.append(float(alpha))
    return u / ell, alphas


# ---------------------------------------------------------------------------
# prefill
# ---------------------------------------------------------------------------

def _scale(scale, d):
    return 1.0 / np.sqrt(d) if (scale is None or scale == 0) else float(scale)


def _group(h_q: int, h_kv: int) -> int:
    if h_kv <= 0 or h_q % h_kv:
        raise ValueError("H_q must be a multiple of H_kv")
    return h_q // h_kv


def prefill(q, k, v, intervals, scale=None, return_probs: bool = False):
    """Packed prefill attention, float64.

    q [T, H_q, d], k/v [T, H_kv, d] (float64 values); intervals int [N, 2].
    Returns out [T, H_q, d]; with ``return_probs`` also the weights
    P [H_q, T, T].
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    T, h_q, d = q.shape
    h_kv = k.shape[1]
    G = _group(h_q, h_kv)
    sc = _scale(scale, d)
    allowed = allowed_mask(intervals, T)
    M = additive_mask(allowed)
    _check_forms_agree(allowed, M)
    out = np.zeros((T, h_q, d), dtype=np.float64)
    probs = np.zeros((h_q, T, T), dtype=np.float64) if return_probs else None
    for h in range(h_q):
        g = h // G
        S = (q[:, h, :] @ k[:, g, :].T) * sc + M
        P = softmax_rows(S)
        out[:, h, :] = P @ v[:, g, :]
        if return_probs:
            probs[h] = P
    if return_probs:
        return out, probs
    return out


def prefill_rows(q, k, v, intervals, rows, heads=None, scale=None):
    """The same definition evaluated for selected output rows only.

    Row t of the dense mask is built from the same rule (same question and
    u <= t) over all T columns.  Returns [len(rows), len(heads), d].
    ``q``/``k``/``v`` may be stored arrays; pass float64 values.
    """
    q = np.asarray(q)
    k = np.asarray(k)
    v = np.asarray(v)
    T, h_q, d = q.shape
    h_kv = k.shape[1]
    G = _group(h_q, h_kv)
    sc = _scale(scale, d)
    heads = list(range(h_q)) if heads is None else list(heads)
    seg = segment_ids(intervals, T)
    cols = np.arange(T)
    out = np.zeros((len(rows), len(heads), d), dtype=np.float64)
    for r, t in enumerate(rows):
        allowed = (seg[t] >= 0) & (seg == seg[t]) & (cols <= t)
        M = np.where(allowed, 0.0, -np.inf)
        for j, h in enumerate(heads):
            g = h // G
            s = (np.asarray(k[:, g, :], dtype=np.float64) @ np.asarray(q[t, h, :], dtype=np.float64)) * sc + M
            p = softmax_rows(s[None, :])[0]
            out[r, j] = p @ np.asarray(v[:, g, :], dtype=np.float64)
    return out


# ---------------------------------------------------------------------------
# KV slot pool
# ---------------------------------------------------------------------------

def validate_prefill(intervals, total_tokens, slot_ids=None, n_slots=0, cap=0):
    """Return None if the call is valid, else the error kind.

    Intervals lie in [0, T] with s <= e and non-empty ones do not overlap.
    With a slot write: every slot id is in [0, n_slots), every question fits
    (L_i <= cap) and the slots of non-empty questions are distinct (two live
    questions sharing one cache is the shared-state bug of the KV-cache
    isolation article, hnwysp.cn, §2.3 and §6.1).
    """
    iv = np.asarray(intervals, dtype=np.int64).reshape(-1, 2)
    T = int(total_tokens)
    for s, e in iv:
        if not (0 <= s <= e <= T):
            return INTERVALS
    ne = iv[iv[:, 1] > iv[:, 0]]
    order = np.argsort(ne[:, 0], kind="stable")
    ne = ne[order]
    for a in range(1, len(ne)):
        if ne[a, 0] < ne[a - 1, 1]:
            return INTERVALS
    if slot_ids is None:
        return None
    sl = np.asarray(slot_ids, dtype=np.int64)
    if np.any((sl < 0) | (sl >= n_slots)):
        return SLOT
    L = iv[:, 1] - iv[:, 0]
    if np.any(L > cap):
        return SLOT_OVERFLOW
    used = sl[L > 0]
    if len(np.unique(used)) != len(used):
        return SLOT
    return None


def slot_write(pool_k, pool_v, k, v, intervals, slot_ids):
    """pool[slot_i, g, j, :] = k/v[s_i + j, g, :] for j < L_i (a bit copy).

    Works on the stored arrays (any dtype); positions >= L_i and slots no
    question uses keep their previous contents.  Returns new arrays.
    """
    pk = np.array(pool_k, copy=True)
    pv = np.array(pool_v, copy=True)
    for (s, e), slot in zip(np.asarray(intervals).reshape(-1, 2), np.asarray(slot_ids)):
        n = int(e - s)
        if n <= 0:
            continue
        pk[slot, :, :n, :] = np.swapaxes(np.asarray(k)[s:e], 0, 1)
        pv[slot, :, :n, :] = np.swapaxes(np.asarray(v)[s:e], 0, 1)
    return pk, pv


# ---------------------------------------------------------------------------
# decode
# ---------------------------------------------------------------------------

def validate_decode(slot_ids, lens, active, n_slots, cap):
    """Return None if the step is valid, else the error kind.

    Only live questions are checked: a dropped question's slot may already
    be back in the pool.  A live question needs a slot in [0, n_slots),
    0 <= lens_i and room for the new row (lens_i < cap), and live slots are
    distinct.
    """
    sl = np.asarray(slot_ids, dtype=np.int64)
    ln = np.asarray(lens, dtype=np.int64)
    live = np.asarray(active).astype(bool)
    if np.any(live & ((sl < 0) | (sl >= n_slots))):
        return SLOT
    if np.any(live & ((ln < 0) | (ln >= cap))):
        return SLOT_OVERFLOW
    used = sl[live]
    if len(np.unique(used)) != len(used):
        return SLOT
    return None


def decode(q_new, k_new, v_new, pool_k, pool_v, slot_ids, lens, active, dtype: str,
           scale=None, inplace: bool = False):
    """One decode step over the slot pool.

    For every live question i with n = lens_i: first the new K/V row is
    written at position n of its slot, then for every q-head h (kv-head
    g = h // G) o_new[i, h] = softmax(scale * q_new[i, h] . K[0..n]) V[0..n].
    Dropped questions are skipped: no output, no write.

    ``pool_k``/``pool_v``/``k_new``/``v_new``/``q_new`` are stored arrays of
    ``dtype`` ('bf16' bits or 'fp32').  Returns (o_new [N, H_q, d] float64
    with NaN rows for dropped questions, pool_k', pool_v').
    """
    pk = pool_k if inplace else np.array(pool_k, copy=True)
    pv = pool_v if inplace else np.array(pool_v, copy=True)
    N, h_q, d = np.asarray(q_new).shape
    h_kv = np.asarray(k_new).shape[1]
    G = _group(h_q, h_kv)
    sc = _scale(scale, d)
    o = np.full((N, h_q, d), np.nan, dtype=np.float64)
    for i in range(N):
        if not active[i]:
            continue
        slot, n = int(slot_ids[i]), int(lens[i])
        pk[slot, :, n, :] = k_new[i]
        pv[slot, :, n, :] = v_new[i]
        for h in range(h_q):
            g = h // G
            K = to_float64(pk[slot, g, :n + 1, :], dtype)
            V = to_float64(pv[slot, g, :n + 1, :], dtype)
            qv = to_float64(np.asarray(q_new)[i, h], dtype)
            p = softmax_rows(((K @ qv) * sc)[None, :])[0]
            o[i, h] = p @ V
    return o, pk, pv


# ---------------------------------------------------------------------------
# rotary position encoding, positions counted per question
# ---------------------------------------------------------------------------

def rope_freqs(d: int, theta: float) -> np.ndarray:
    """w_i = theta^(-2i/d) for i = 0 .. d/2 - 1 (float64)."""
    return np.power(float(theta), -np.arange(0, d, 2, dtype=np.float64) / d)


def rope_rotate(x, positions, theta: float) -> np.ndarray:
    """Rotate-half RoPE of x [P, H, d] (float64 values) at positions[P].

    The pair (x_i, x_{i+d/2}) of every head turns by the angle p * w_i:
    (a, b) -> (a cos - b sin, b cos + a sin).  Rows whose position is
    negative (tokens in no question) are returned unchanged.
    """
    x = np.asarray(x, dtype=np.float64)
    half = x.shape[-1] // 2
    pos = np.asarray(positions, dtype=np.float64).reshape(-1)
    ang = pos[:, None] * rope_freqs(x.shape[-1], theta)[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    out = np.concatenate([a * c - b * s, b * c + a * s], axis=-1)
    keep = pos < 0
    out[keep] = x[keep]
    return out


def prefill_positions(intervals, total_tokens: int) -> np.ndarray:
    """Position of token t inside its own question, t - s_i (-1 for a token in
    no question): each question counts from 0, as it would alone."""
    pos = np.full(int(total_tokens), -1, dtype=np.int64)
    for s, e in np.asarray(intervals, dtype=np.int64).reshape(-1, 2):
        pos[s:e] = np.arange(e - s)
    return pos


def prefill_rope(q, k, v, intervals, theta: float, scale=None):
    """Packed prefill with RoPE: q and k rotated at their per-question
    positions, then the isolated causal attention of ``prefill``.  Returns
    (out, q_rot, k_rot), float64."""
    pos = prefill_positions(intervals, np.asarray(q).shape[0])
    q_rot = rope_rotate(q, pos, theta)
    k_rot = rope_rotate(k, pos, theta)
    return prefill(q_rot, k_rot, v, intervals, scale=scale), q_rot, k_rot


def round_to_stored(x64: np.ndarray, dtype: str) -> np.ndarray:
    """float64 values -> the stored array of ``dtype``: bfloat16 bits rounded
    once, to nearest with ties to even, from the float64 value (8 significant
    bits: x = m 2^e with 1/2 <= |m| < 1 becomes rint(256 m) 2^(e-8), which
    float32 then holds exactly), or float32."""
    from workloads import f32_to_bf16_bits
    x64 = np.asarray(x64, dtype=np.float64)
    if dtype == "bf16":
        m, e = np.frexp(x64)
        r = np.ldexp(np.rint(m * 256.0), e - 8)
        return f32_to_bf16_bits(r.astype(np.float32))  # exact: r has at most 8 significant bits
    return x64.astype(np.float32)


# ---------------------------------------------------------------------------
# paged slot pool
# ---------------------------------------------------------------------------

PAGE = 128  # positions per block


def paged_gather(pool, table_row, n: int, page: int = PAGE) -> np.ndarray:
    """Positions 0..n-1 of one question through its block table row: [H_kv, n, d]
    (position p lives in block table_row[p // page], row p % page)."""
    pool = np.asarray(pool)
    if n == 0:
        return pool[:0, :, :0].reshape(pool.shape[1], 0, pool.shape[3])
    assert all(int(table_row[p // page]) >= 0 for p in range(n)), "a position without a block"
    rows = [pool[int(table_row[p // page]), :, p % page, :] for p in range(n)]
    return np.stack(rows, axis=1)


def paged_slot_write(pool_k, pool_v, k, v, intervals, block_table, page: int = PAGE):
    """pool[table_i[j // page], g, j % page, :] = k/v[s_i + j, g, :] for j < L_i (a bit
    copy); every other row keeps its contents.  Returns new arrays."""
    pk = np.array(pool_k, copy=True)
    pv = np.array(pool_v, copy=True)
    for (s, e), row in zip(np.asarray(intervals).reshape(-1, 2), np.asarray(block_table)):
        for j in range(int(e - s)):
            blk, r = int(row[j // page]), j % page
            assert blk >= 0, "a position without a block"
            pk[blk, :, r, :] = np.asarray(k)[s + j]
            pv[blk, :, r, :] = np.asarray(v)[s + j]
    return pk, pv


def validate_paged(lengths, block_table, n_blocks: int, live=None, page: int = PAGE):
    """Return None if the tables are valid for questions of the given lengths (positions
    0..length-1 are used), else the error kind: a question needing more blocks than its
    table row holds -> SLOT_OVERFLOW; a used entry outside [0, n_blocks) -> SLOT; one
    block used by two questions, or twice by one -> SLOT.  ``live`` masks the questions
    that are checked (all when None)."""
    tb = np.asarray(block_table, dtype=np.int64)
    ln = np.asarray(lengths, dtype=np.int64)
    live = np.ones(len(ln), bool) if live is None else np.asarray(live).astype(bool)
    need = (ln + page - 1) // page
    if np.any(live & (need > tb.shape[1])):
        return SLOT_OVERFLOW
    used = [int(tb[i, b]) for i in range(len(ln)) if live[i] for b in range(int(need[i]))]
    if any(b < 0 or b >= n_blocks for b in used):
        return SLOT
    if len(set(used)) != len(used):
        return SLOT
    return None


def decode_paged(q_new, k_new, v_new, pool_k, pool_v, block_table, lens, active, dtype: str,
                 scale=None, page: int = PAGE):
    """One decode step over the paged pool: for every live question the new K/V
    row goes to position n = lens_i (block table_i[n // page], row n % page), then
    the question's positions 0..n, gathered through its table, are attended as in
    ``decode``.  Returns (o_new, pool_k', pool_v')."""
    pk = np.array(pool_k, copy=True)
    pv = np.array(pool_v, copy=True)
    N, h_q, d = np.asarray(q_new).shape
    h_kv = np.asarray(k_new).shape[1]
    G = _group(h_q, h_kv)
    sc = _scale(scale, d)
    o = np.full((N, h_q, d), np.nan, dtype=np.float64)
    for i in range(N):
        if not active[i]:
            continue
        n = int(lens[i])
        row = np.asarray(block_table)[i]
        assert int(row[n // page]) >= 0, "no block for the new row"
        pk[int(row[n // page]), :, n % page, :] = np.asarray(k_new)[i]
        pv[int(row[n // page]), :, n % page, :] = np.asarray(v_new)[i]
        K = to_float64(paged_gather(pk, row, n + 1, page), dtype)
        V = to_float64(paged_gather(pv, row, n + 1, page), dtype)
        for h in range(h_q):
            qv = to_float64(np.asarray(q_new)[i, h], dtype)
            p = softmax_rows(((K[h // G] @ qv) * sc)[None, :])[0]
            o[i, h] = p @ V[h // G]
    return o, pk, pv


def assign_blocks(need, free, max_blocks: int, contiguous_first: bool = True):
    """Block tables for questions needing need[i] blocks, taken from the free map
    ``free`` (bool per block, True = free), in question order.  Contiguous first (Kev
    pipeline article, §4.3): a question takes the lowest run of need[i] consecutive
    free blocks; without such a run, or with contiguous_first False, its lowest free
    blocks one by one.  Returns (table [N, max_blocks] with -1 past each row's blocks,
    free') or None when the free blocks do not suffice or a row would not fit."""
    fr = np.array(free, dtype=bool, copy=True)
    table = np.full((len(need), max_blocks), -1, dtype=np.int32)
    for i, m in enumerate(need):
        m = int(m)
        if m > max_blocks:
            return None
        if m == 0:
            continue
        pick = None
        if contiguous_first:
            run = 0
            for b in range(len(fr)):
                run = run + 1 if fr[b] else 0
                if run == m:
                    pick = list(range(b - m + 1, b + 1))
                    break
        if pick is None:
            idx = np.nonzero(fr)[0]
            if len(idx) < m:
                return None
            pick = [int(x) for x in idx[:m]]
        table[i, :m] = pick
        fr[pick] = False
    return table, fr


# ---------------------------------------------------------------------------
# chunked prefill into slots
# ---------------------------------------------------------------------------

def validate_chunk(intervals, total_tokens, prefix_lens, slot_ids, n_slots, cap, align: int = PAGE):
    """Return None if a chunked prefill is valid, else the error kind, in this order:
    intervals (as ``validate_prefill``); a slot id outside [0, n_slots) -> SLOT; a cached
    prefix length that is negative or not a multiple of ``align`` (the library's
    restriction: chunks start on a tile boundary) -> PREFIX; prefix + chunk longer than the
    slot -> SLOT_OVERFLOW; a slot shared by two non-empty chunks -> SLOT."""
    err = validate_prefill(intervals, total_tokens)
    if err is not None:
        return err
    iv = np.asarray(intervals, dtype=np.int64).reshape(-1, 2)
    sl = np.asarray(slot_ids, dtype=np.int64)
    pre = np.asarray(prefix_lens, dtype=np.int64)
    L = iv[:, 1] - iv[:, 0]
    if np.any((sl < 0) | (sl >= n_slots)):
        return SLOT
    if np.any((pre < 0) | (pre % align != 0)):
        return PREFIX
    if np.any(pre + L > cap):
        return SLOT_OVERFLOW
    used = sl[L > 0]
    if len(np.unique(used)) != len(used):
        return SLOT
    return None


def prefill_chunk(q, k, v, intervals, prefix_lens, slot_ids, pool_k, pool_v, dtype: str, scale=None):
    """Chunked prefill into slots.  Question i's chunk is packed tokens [s_i, e_i): its
    positions P_i .. P_i + L_i - 1, after the P_i = prefix_lens[i] positions already in slot
    slot_ids[i].  The chunk's K/V rows go into the slot first (positions P_i + j, bit copies),
    then token s_i + j attends to positions 0 .. P_i + j of its slot: the cached prefix and its
    own chunk causally, nothing of another question.  Rows of tokens in no chunk are 0.

    ``q``/``k``/``v`` and the pools are stored arrays of ``dtype``.  Returns (out [T, H_q, d]
    float64, pool_k', pool_v')."""
    pk = np.array(pool_k, copy=True)
    pv = np.array(pool_v, copy=True)
    q = np.asarray(q)
    T, h_q, d = q.shape
    h_kv = np.asarray(k).shape[1]
    G = _group(h_q, h_kv)
    sc = _scale(scale, d)
    out = np.zeros((T, h_q, d), dtype=np.float64)
    for (s, e), P, slot in zip(np.asarray(intervals).reshape(-1, 2), np.asarray(prefix_lens), np.asarray(slot_ids)):
        s, e, P, slot = int(s), int(e), int(P), int(slot)
        L = e - s
        if L <= 0:
            continue
        pk[slot, :, P:P + L, :] = np.swapaxes(np.asarray(k)[s:e], 0, 1)
        pv[slot, :, P:P + L, :] = np.swapaxes(np.asarray(v)[s:e], 0, 1)
        allowed = np.arange(P + L)[None, :] <= (P + np.arange(L))[:, None]  # key u for chunk row j: u <= P + j
        for h in range(h_q):
            g = h // G
            K = to_float64(pk[slot, g, :P + L, :], dtype)
            V = to_float64(pv[slot, g, :P + L, :], dtype)
            Q = to_float64(q[s:e, h], dtype)
            scores = np.where(allowed, (Q @ K.T) * sc, -np.inf)
            out[s:e, h] = softmax_rows(scores) @ V
    return out, pk, pv


# ---------------------------------------------------------------------------
# per-question temperature sampling
# ---------------------------------------------------------------------------

SAMPLING = "sampling"


def sample_probs(logits_row, temperature: float) -> np.ndarray:
    """softmax(logits / T) in float64 (T > 0), the stable form of ``softmax_rows``."""
    z = np.asarray(logits_row, dtype=np.float64) / float(temperature)
    return softmax_rows(z[None, :])[0]


def sample_tokens(logits, temperature, uniforms, active=None):
    """Token per question: argmax of its logits (lowest index among equal maxima) when its
    temperature is 0, else the smallest k with sum_{j <= k} p_j > u, p = softmax(logits / T)
    (the last k with p_k > 0 if rounding leaves no such k).  ``logits`` [N, V] float64
    values.  Dropped questions get -1.  Returns int64 [N]."""
    lg = np.asarray(logits, dtype=np.float64)
    N = lg.shape[0]
    live = np.ones(N, bool) if active is None else np.asarray(active).astype(bool)
    out = np.full(N, -1, dtype=np.int64)
    for i in range(N):
        if not live[i]:
            continue
        if float(temperature[i]) == 0.0:
            out[i] = int(np.argmax(lg[i]))  # numpy: the first maximum
            continue
        p = sample_probs(lg[i], temperature[i])
        cdf = np.cumsum(p)
        k = int(np.searchsorted(cdf, float(uniforms[i]), side="right"))
        if k >= len(p):
            k = int(np.nonzero(p > 0)[0][-1])
        out[i] = k
    return out


def validate_sampling(temperature, uniforms, active=None):
    """None, or SAMPLING when a live question's temperature is negative or not finite or its
    uniform lies outside [0, 1)."""
    t = np.asarray(temperature, dtype=np.float64)
    u = np.asarray(uniforms, dtype=np.float64)
    live = np.ones(len(t), bool) if active is None else np.asarray(active).astype(bool)
    bad = ~np.isfinite(t) | (t < 0) | ~(u >= 0) | ~(u < 1)
    return SAMPLING if np.any(live & bad) else None


# ---------------------------------------------------------------------------
# token-grouped LoRA
# ---------------------------------------------------------------------------

ADAPTER = "adapter"


def lora_apply(y, x, intervals, adapter_ids, lora_a, lora_b, scales):
    """Token t of question i with adapter a = adapter_ids[i] >= 0 gets
    y[t] + scales[a] * B_a (A_a x[t]), A_a = lora_a[a] [r, d_in], B_a = lora_b[a] [d_out, r];
    rows of questions without an adapter (-1) and of tokens in no question are unchanged.
    float64 in and out."""
    out = np.array(y, dtype=np.float64, copy=True)
    x = np.asarray(x, dtype=np.float64)
    for (s, e), a in zip(np.asarray(intervals).reshape(-1, 2), np.asarray(adapter_ids)):
        if a < 0 or e <= s:
            continue
        A = np.asarray(lora_a[a], dtype=np.float64)
        B = np.asarray(lora_b[a], dtype=np.float64)
        out[s:e] += float(scales[a]) * (x[s:e] @ A.T) @ B.T
    return out


def lora_router(y, x, intervals, adapter_ids, lora_a, lora_b, scales):
    """The same result in the routing form the article describes: every adapter's delta over
    the whole sequence, kept where a token's adapter id matches (a mask per adapter)."""
    out = np.array(y, dtype=np.float64, copy=True)
    x = np.asarray(x, dtype=np.float64)
    T = x.shape[0]
    token_adapter = np.full(T, -1)
    for (s, e), a in zip(np.asarray(intervals).reshape(-1, 2), np.asarray(adapter_ids)):
        token_adapter[s:e] = a
    for a in range(len(lora_a)):
        delta = float(scales[a]) * (x @ np.asarray(lora_a[a], np.float64).T) @ np.asarray(lora_b[a], np.float64).T
        out += (token_adapter == a)[:, None] * delta
    return out


def validate_lora(adapter_ids, n_adapters: int):
    """None, or ADAPTER when an adapter id lies outside [-1, n_adapters)."""
    a = np.asarray(adapter_ids, dtype=np.int64)
    return ADAPTER if np.any((a < -1) | (a >= n_adapters)) else None
