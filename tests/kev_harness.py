"""Test-side glue: seeded workloads -> device tensors -> libkev calls -> numpy.

Only marshalling lives here; the computation under test runs in libkev's
kernels and the expected values come from ``oracle/``.
"""
from __future__ import annotations

import numpy as np
import torch

import packed_question_isolated_gb300 as kev
import workloads as W

TOL_FP32_MAX = 1e-5
TOL_BF16_MAX = 2e-2
TOL_BF16_REL_L2 = 5e-3


def dev(arr: np.ndarray, dtype: str | None = None) -> torch.Tensor:
    """Stored numpy array -> device tensor (uint16 bf16 bits become torch.bfloat16)."""
    a = np.ascontiguousarray(arr)
    t = torch.from_numpy(a)
    if a.dtype == np.uint16:
        t = t.view(torch.bfloat16)
    return t.cuda()


def host(t: torch.Tensor) -> np.ndarray:
    """Device tensor -> stored numpy array (bf16 as uint16 bits)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.uint16).numpy()
    return t.numpy()


def f64(t_or_a, dtype: str) -> np.ndarray:
    a = host(t_or_a) if isinstance(t_or_a, torch.Tensor) else t_or_a
    return W.to_float64(a, dtype)


def tdtype(dtype: str):
    return torch.bfloat16 if dtype == "bf16" else torch.float32


def shape_of(w):
    return kev.make_shape(w.h_q, w.h_kv, w.d, w.dtype, w.scale)


def prefill_ws(w):
    nbytes = kev.kev_prefill_workspace_size(w.n_questions, w.total_tokens, shape_of(w))
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda"), nbytes


class PrefillRun:
    """Device buffers of one prefill call plus its result."""

    def __init__(self, w, slots: bool = True, sentinel_pool: bool = True, out_sentinel: bool = True,
                 intervals=None, slot_ids=None):
        self.w = w
        td = tdtype(w.dtype)
        self.q, self.k, self.v = dev(w.q), dev(w.k), dev(w.v)
        iv = w.intervals if intervals is None else intervals
        self.intervals = torch.from_numpy(np.ascontiguousarray(iv, dtype=np.int32)).cuda()
        sl = w.slot_ids if slot_ids is None else slot_ids
        self.slot_ids = torch.from_numpy(np.ascontiguousarray(sl, dtype=np.int32)).cuda() if slots else None
        T = w.total_tokens
        self.out = torch.empty((max(T, 1), w.h_q, w.d), dtype=td, device="cuda")
        if out_sentinel:
            self.out.fill_(float("nan"))
        if slots:
            shape = (w.n_slots, w.h_kv, w.cap, w.d)
            self.pool_k = torch.empty(shape, dtype=td, device="cuda")
            self.pool_v = torch.empty(shape, dtype=td, device="cuda")
            if sentinel_pool:
                self.pool_k.fill_(-7.0)
                self.pool_v.fill_(-9.0)
        else:
            self.pool_k = self.pool_v = None
        self.pool_k0 = self.pool_k.clone() if slots else None
        self.pool_v0 = self.pool_v.clone() if slots else None
        self.ws, self.ws_bytes = prefill_ws(w)
        self.status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        self.n_questions = len(iv)

    def run(self, check=True):
        w = self.w
        st = kev.kev_prefill_attn(self.q, self.k, self.v, w.total_tokens, self.intervals, self.n_questions,
                                  self.slot_ids, self.pool_k, self.pool_v, w.n_slots, w.cap, self.out,
                                  shape_of(w), self.ws, self.ws_bytes, self.status, check=check)
        return st

    def device_status(self) -> int:
        return kev.kev_read_status(self.status)


def compare(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = ""):
    """Assert the tolerance the float configurations are held to."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    diff = np.abs(got - ref)
    mx = float(diff.max()) if diff.size else 0.0
    if dtype == "fp32":
        assert mx <= TOL_FP32_MAX, f"{what}: max|d| {mx:.3e} > {TOL_FP32_MAX}"
    else:
        rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))
        assert mx <= TOL_BF16_MAX, f"{what}: max|d| {mx:.3e} > {TOL_BF16_MAX}"
        assert rel <= TOL_BF16_REL_L2, f"{what}: rel L2 {rel:.3e} > {TOL_BF16_REL_L2}"
    return mx


class DecodeRun:
    """Device buffers of one decode step."""

    def __init__(self, dtype, h_q, h_kv, d, pool_k, pool_v, slot_ids, lens, active, q_new, k_new, v_new,
                 cap, n_slots, scale=0.0):
        self.dtype = dtype
        self.shape = kev.make_shape(h_q, h_kv, d, dtype, scale)
        self.pool_k = pool_k if isinstance(pool_k, torch.Tensor) else dev(pool_k)
        self.pool_v = pool_v if isinstance(pool_v, torch.Tensor) else dev(pool_v)
        self.slot_ids = torch.from_numpy(np.ascontiguousarray(slot_ids, dtype=np.int32)).cuda()
        self.lens = torch.from_numpy(np.ascontiguousarray(lens, dtype=np.int32)).cuda()
        self.active = torch.from_numpy(np.ascontiguousarray(active, dtype=np.uint8)).cuda()
        self.q_new, self.k_new, self.v_new = dev(q_new), dev(k_new), dev(v_new)
        self.n = len(lens)
        self.cap, self.n_slots = cap, n_slots
        self.out = torch.full((self.n, h_q, d), float("nan"), dtype=tdtype(dtype), device="cuda")
        nbytes = kev.kev_decode_workspace_size(self.n, cap, self.shape)
        self.ws_bytes = nbytes
        self.ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device="cuda")
        self.status = torch.full((1,), -1, dtype=torch.int32, device="cuda")

    def run(self, check=True):
        return kev.kev_decode_attn(self.q_new, self.k_new, self.v_new, self.pool_k, self.pool_v, self.n_slots,
                                   self.cap, self.slot_ids, self.lens, self.active, self.n, self.out, self.shape,
                                   self.ws, self.ws_bytes, self.status, check=check)

    def device_status(self) -> int:
        return kev.kev_read_status(self.status)
