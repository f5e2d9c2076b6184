"""Thin ctypes binding of libkev (include/kev.h), same names as the C entry points.

Argument marshalling only: tensors become device pointers (``data_ptr()``),
the stream defaults to torch's current CUDA stream, ``kev_attn_shape`` is
built from its fields, and a non-OK status raises ``KevError``.  Every step of
the computation runs in the library's CUDA kernels; there is no Python or CPU
fallback, and importing this module fails if the library is not built.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkev.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libkev.so not found at {LIB_PATH}; build it first "
        "(python -m packed_question_isolated_gb300.build or __graft_entry__.build())")

_lib = ctypes.CDLL(LIB_PATH)

KEV_OK = 0
KEV_ERR_INVALID_ARG = 1
KEV_ERR_UNSUPPORTED = 2
KEV_ERR_INTERVALS = 3
KEV_ERR_SLOT = 4
KEV_ERR_SLOT_OVERFLOW = 5
KEV_ERR_TIMEOUT = 6
KEV_ERR_CUDA = 7
KEV_ERR_POSITION = 8
KEV_ERR_PREFIX = 9
KEV_ERR_SAMPLING = 10
KEV_ERR_ADAPTER = 11
KEV_BF16 = 0
KEV_FP32 = 1
KEV_PAGE = 128
KEV_MAX_PAGED_ENTRIES = 16384
KEV_MAX_QUESTIONS = 4096

STATUS_NAMES = {
    0: "KEV_OK", 1: "KEV_ERR_INVALID_ARG", 2: "KEV_ERR_UNSUPPORTED", 3: "KEV_ERR_INTERVALS",
    4: "KEV_ERR_SLOT", 5: "KEV_ERR_SLOT_OVERFLOW", 6: "KEV_ERR_TIMEOUT", 7: "KEV_ERR_CUDA",
    8: "KEV_ERR_POSITION", 9: "KEV_ERR_PREFIX", 10: "KEV_ERR_SAMPLING", 11: "KEV_ERR_ADAPTER",
}

# every symbol include/kev.h declares
EXPORTED = [
    "kev_prefill_workspace_size", "kev_build_segments", "kev_read_work_list", "kev_read_work_units",
    "kev_prefill_from_segments", "kev_prefill_attn", "kev_kv_write",
    "kev_decode_workspace_size", "kev_decode_attn", "kev_decode_advance",
    "kev_read_status", "kev_status_string", "kev_launch_count", "kev_decode_attn_static", "kev_decode_step",
    "kev_rope_table_size", "kev_rope_table", "kev_rope_prefill", "kev_prefill_attn_rope", "kev_rope_decode",
    "kev_decode_attn_rope", "kev_prefill_attn_paged", "kev_kv_write_paged", "kev_decode_attn_paged",
    "kev_assign_blocks", "kev_prefill_chunk", "kev_sample", "kev_lora_apply",
]


class kev_attn_shape(ctypes.Structure):
    _fields_ = [("h_q", ctypes.c_int32), ("h_kv", ctypes.c_int32), ("d_h", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("scale", ctypes.c_float)]


class KevError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {STATUS_NAMES.get(int(status), status)} "
                         f"({_lib.kev_status_string(int(status)).decode()})")


_P = ctypes.c_void_p
_I = ctypes.c_int32
_Z = ctypes.c_size_t
_S = ctypes.POINTER(kev_attn_shape)


def _sig(name, restype, *argtypes):
    f = getattr(_lib, name)
    f.restype = restype
    f.argtypes = list(argtypes)
    return f


_c = {
    "kev_prefill_workspace_size": _sig("kev_prefill_workspace_size", _Z, _I, _I, _S),
    "kev_build_segments": _sig("kev_build_segments", _I, _P, _I, _I, _P, _I, _I, _S, _P, _Z, _P, _P),
    "kev_read_work_list": _sig("kev_read_work_list", _I, _P, _Z, _P, _I, _P),
    "kev_read_work_units": _sig("kev_read_work_units", _I, _P, _Z, _P, _I, _P),
    "kev_prefill_from_segments": _sig("kev_prefill_from_segments", _I, _P, _P, _P, _I, _P, _I, _P, _P, _P,
                                      _I, _I, _P, _S, _P, _Z, _P, _P),
    "kev_prefill_attn": _sig("kev_prefill_attn", _I, _P, _P, _P, _I, _P, _I, _P, _P, _P, _I, _I, _P, _S,
                             _P, _Z, _P, _P),
    "kev_kv_write": _sig("kev_kv_write", _I, _P, _P, _I, _P, _I, _P, _P, _P, _I, _I, _S, _P, _Z, _P, _P),
    "kev_decode_workspace_size": _sig("kev_decode_workspace_size", _Z, _I, _I, _S),
    "kev_decode_attn": _sig("kev_decode_attn", _I, _P, _P, _P, _P, _P, _I, _I, _P, _P, _P, _I, _P, _S,
                            _P, _Z, _P, _P),
    "kev_decode_attn_static": _sig("kev_decode_attn_static", _I, _P, _P, _P, _P, _P, _I, _I, _P, _P, _P, _I,
                                   _P, _S, _P, _P),
    "kev_decode_advance": _sig("kev_decode_advance", _I, _P, _P, _I, _P),
    "kev_decode_step": _sig("kev_decode_step", _I, _P, _P, _P, _P, _P, _I, _I, _P, _P, _P, _I, _P, _S, _P, _Z, _P, _P),
    "kev_read_status": _sig("kev_read_status", _I, _P, _P),
    "kev_status_string": _sig("kev_status_string", ctypes.c_char_p, _I),
    "kev_launch_count": _sig("kev_launch_count", _I, _I),
    "kev_rope_table_size": _sig("kev_rope_table_size", _Z, _I, _I),
    "kev_rope_table": _sig("kev_rope_table", _I, _P, _I, _I, ctypes.c_double, _P),
    "kev_rope_prefill": _sig("kev_rope_prefill", _I, _P, _P, _P, _I, _P, _I, _P, _P, _P, _I, _I, _S, _P, _I,
                             _P, _Z, _P, _P),
    "kev_prefill_attn_rope": _sig("kev_prefill_attn_rope", _I, _P, _P, _P, _I, _P, _I, _P, _P, _P, _I, _I, _P,
                                  _S, _P, _I, _P, _Z, _P, _P),
    "kev_rope_decode": _sig("kev_rope_decode", _I, _P, _P, _P, _P, _I, _S, _P, _I, _P, _P),
    "kev_decode_attn_rope": _sig("kev_decode_attn_rope", _I, _P, _P, _P, _P, _P, _I, _I, _P, _P, _P, _I, _P,
                                 _S, _P, _I, _P, _Z, _P, _P),
    "kev_prefill_attn_paged": _sig("kev_prefill_attn_paged", _I, _P, _P, _P, _I, _P, _I, _P, _I, _P, _P, _I, _P,
                                   _S, _P, _Z, _P, _P),
    "kev_kv_write_paged": _sig("kev_kv_write_paged", _I, _P, _P, _I, _P, _I, _P, _I, _P, _P, _I, _S, _P, _Z, _P, _P),
    "kev_decode_attn_paged": _sig("kev_decode_attn_paged", _I, _P, _P, _P, _P, _P, _I, _P, _I, _P, _P, _I, _P, _S,
                                  _P, _Z, _P, _P),
    "kev_assign_blocks": _sig("kev_assign_blocks", _I, _P, _I, _P, _I, _P, _I, _I),
    "kev_lora_apply": _sig("kev_lora_apply", _I, _P, _P, _I, _I, _I, _P, _I, _P, _P, _P, _P, _I, _I, _P, _Z, _P,
                           _P),
    "kev_sample": _sig("kev_sample", _I, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P),
    "kev_prefill_chunk": _sig("kev_prefill_chunk", _I, _P, _P, _P, _I, _P, _I, _P, _P, _P, _P, _I, _I, _P, _S, _P,
                              _Z, _P, _P),
}


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_shape(h_q: int, h_kv: int, d_h: int, dtype="bf16", scale: float = 0.0) -> kev_attn_shape:
    if isinstance(dtype, str):
        dtype = {"bf16": KEV_BF16, "fp32": KEV_FP32}[dtype]
    return kev_attn_shape(int(h_q), int(h_kv), int(d_h), int(dtype), float(scale))


def _shape(shape) -> kev_attn_shape:
    if isinstance(shape, kev_attn_shape):
        return shape
    if isinstance(shape, dict):
        return make_shape(**shape)
    return make_shape(*shape)


def _check(status: int, where: str, check: bool) -> int:
    if check and status != KEV_OK:
        raise KevError(status, where)
    return status


def library_path() -> str:
    return LIB_PATH


def kev_status_string(status: int) -> str:
    return _c["kev_status_string"](int(status)).decode()


def kev_launch_count(entry_point: int) -> int:
    return int(_c["kev_launch_count"](int(entry_point)))


def kev_prefill_workspace_size(n_questions: int, total_tokens: int, shape) -> int:
    s = _shape(shape)
    return int(_c["kev_prefill_workspace_size"](int(n_questions), int(total_tokens), ctypes.byref(s)))


def kev_decode_workspace_size(n_questions: int, slot_cap: int, shape) -> int:
    s = _shape(shape)
    return int(_c["kev_decode_workspace_size"](int(n_questions), int(slot_cap), ctypes.byref(s)))


def kev_build_segments(intervals, n_questions, total_tokens, slot_ids, n_slots, slot_cap, shape, workspace,
                       workspace_bytes, dev_status=None, stream=None, check=True) -> int:
    s = _shape(shape)
    st = _c["kev_build_segments"](_ptr(intervals), int(n_questions), int(total_tokens), _ptr(slot_ids),
                                  int(n_slots), int(slot_cap), ctypes.byref(s), _ptr(workspace),
                                  int(workspace_bytes), _ptr(dev_status), _stream(stream))
    return _check(st, "kev_build_segments", check)


def kev_read_work_list(workspace, workspace_bytes, max_items: int, stream=None):
    """Returns the work list as (question, q_row_begin, q_rows, first_head | n_heads << 16) tuples."""
    buf = (ctypes.c_int32 * (4 * max(int(max_items), 1)))()
    n = int(_c["kev_read_work_list"](_ptr(workspace), int(workspace_bytes), buf, int(max_items),
                                     _stream(stream)))
    if n < 0:
        raise KevError(KEV_ERR_INVALID_ARG, "kev_read_work_list")
    m = min(n, int(max_items))
    return [tuple(buf[4 * j:4 * j + 4]) for j in range(m)], n


def kev_read_work_units(workspace, workspace_bytes, max_units: int, stream=None):
    """Returns the unit-form work list as (question, kv_head, nkv_a, nkv_b, a0, a1, b0, b1) tuples."""
    buf = (ctypes.c_int32 * (8 * max(int(max_units), 1)))()
    n = int(_c["kev_read_work_units"](_ptr(workspace), int(workspace_bytes), buf, int(max_units),
                                      _stream(stream)))
    if n < 0:
        raise KevError(KEV_ERR_INVALID_ARG, "kev_read_work_units")
    m = min(n, int(max_units))
    out = []
    for j in range(m):
        w = buf[8 * j:8 * j + 8]
        out.append((w[0], w[1], w[2] & 0xffff, w[2] >> 16, w[4], w[5], w[6], w[7]))
    return out, n


def kev_prefill_from_segments(q, k, v, total_tokens, intervals, n_questions, slot_ids, pool_k, pool_v, n_slots,
                              slot_cap, out, shape, workspace, workspace_bytes, dev_status=None, stream=None,
                              check=True) -> int:
    s = _shape(shape)
    st = _c["kev_prefill_from_segments"](_ptr(q), _ptr(k), _ptr(v), int(total_tokens), _ptr(intervals),
                                         int(n_questions), _ptr(slot_ids), _ptr(pool_k), _ptr(pool_v),
                                         int(n_slots), int(slot_cap), _ptr(out), ctypes.byref(s),
                                         _ptr(workspace), int(workspace_bytes), _ptr(dev_status),
                                         _stream(stream))
    return _check(st, "kev_prefill_from_segments", check)


def kev_prefill_attn(q, k, v, total_tokens, intervals, n_questions, slot_ids, pool_k, pool_v, n_slots, slot_cap,
                     out, shape, workspace, workspace_bytes, dev_status=None, stream=None, check=True) -> int:
    s = _shape(shape)
    st = _c["kev_prefill_attn"](_ptr(q), _ptr(k), _ptr(v), int(total_tokens), _ptr(intervals), int(n_questions),
                                _ptr(slot_ids), _ptr(pool_k), _ptr(pool_v), int(n_slots), int(slot_cap),
                                _ptr(out), ctypes.byref(s), _ptr(workspace), int(workspace_bytes),
                                _ptr(dev_status), _stream(stream))
    return _check(st, "kev_prefill_attn", check)


def kev_kv_write(k, v, total_tokens, intervals, n_questions, slot_ids, pool_k, pool_v, n_slots, slot_cap, shape,
                 workspace, workspace_bytes, dev_status=None, stream=None, check=True) -> int:
    s = _shape(shape)
    st = _c["kev_kv_write"](_ptr(k), _ptr(v), int(total_tokens), _ptr(intervals), int(n_questions),
                            _ptr(slot_ids), _ptr(pool_k), _ptr(pool_v), int(n_slots), int(slot_cap),
                            ctypes.byref(s), _ptr(workspace), int(workspace_bytes), _ptr(dev_status),
                            _stream(stream))
    return _check(st, "kev_kv_write", check)


def kev_decode_attn(q_new, k_new, v_new, pool_k, pool_v, n_slots, slot_cap, slot_ids, lens, active, n_questions,
                    out, shape, workspace, workspace_bytes, dev_status=None, stream=None, check=True) -> int:
    s = _shape(shape)
    st = _c["kev_decode_attn"](_ptr(q_new), _ptr(k_new), _ptr(v_new), _ptr(pool_k), _ptr(pool_v), int(n_slots),
                               int(slot_cap), _ptr(slot_ids), _ptr(lens), _ptr(active), int(n_questions),
                               _ptr(out), ctypes.byref(s), _ptr(workspace), int(workspace_bytes),
                               _ptr(dev_status), _stream(stream))
    return _check(st, "kev_decode_attn", check)


KEV_STATIC_SCRATCH_BYTES = 16 << 20


def kev_decode_attn_static(q_new, k_new, v_new, pool_k, pool_v, n_slots, slot_cap, slot_ids, lens, active,
                           n_questions, out, shape, dev_status=None, stream=None, check=True) -> int:
    """kev_decode_attn with the library's fixed scratch instead of a caller workspace (for
    callers that cannot allocate device memory); calls that overlap on the GPU race."""
    s = _shape(shape)
    st = _c["kev_decode_attn_static"](_ptr(q_new), _ptr(k_new), _ptr(v_new), _ptr(pool_k), _ptr(pool_v),
                                      int(n_slots), int(slot_cap), _ptr(slot_ids), _ptr(lens), _ptr(active),
                                      int(n_questions), _ptr(out), ctypes.byref(s), _ptr(dev_status),
                                      _stream(stream))
    return _check(st, "kev_decode_attn_static", check)


def kev_decode_step(q_new, k_new, v_new, pool_k, pool_v, n_slots, slot_cap, slot_ids, lens, active, n_questions,
                    out, shape, workspace, workspace_bytes, dev_status=None, stream=None, check=True) -> int:
    """kev_decode_attn followed by lens[i] += 1 for live i (folded into the merge kernel on the
    tensor-core path)."""
    s = _shape(shape)
    st = _c["kev_decode_step"](_ptr(q_new), _ptr(k_new), _ptr(v_new), _ptr(pool_k), _ptr(pool_v), int(n_slots),
                               int(slot_cap), _ptr(slot_ids), _ptr(lens), _ptr(active), int(n_questions), _ptr(out),
                               ctypes.byref(s), _ptr(workspace), int(workspace_bytes), _ptr(dev_status),
                               _stream(stream))
    return _check(st, "kev_decode_step", check)


def kev_decode_advance(lens, active, n, stream=None, check=True) -> int:
    st = _c["kev_decode_advance"](_ptr(lens), _ptr(active), int(n), _stream(stream))
    return _check(st, "kev_decode_advance", check)


def kev_read_status(dev_status, stream=None) -> int:
    return int(_c["kev_read_status"](_ptr(dev_status), _stream(stream)))


def kev_rope_table_size(max_pos: int, d_h: int) -> int:
    return int(_c["kev_rope_table_size"](int(max_pos), int(d_h)))


def kev_rope_table(table, max_pos, d_h, theta, stream=None, check=True) -> int:
    st = _c["kev_rope_table"](_ptr(table), int(max_pos), int(d_h), float(theta), _stream(stream))
    return _check(st, "kev_rope_table", check)


def kev_rope_prefill(q, k, v, total_tokens, intervals, n_questions, slot_ids, pool_k, pool_v, n_slots, slot_cap,
                     shape, rope_table, max_pos, workspace, workspace_bytes, dev_status=None, stream=None,
                     check=True) -> int:
    s = _shape(shape)
    st = _c["kev_rope_prefill"](_ptr(q), _ptr(k), _ptr(v), int(total_tokens), _ptr(intervals), int(n_questions),
                                _ptr(slot_ids), _ptr(pool_k), _ptr(pool_v), int(n_slots), int(slot_cap),
                                ctypes.byref(s), _ptr(rope_table), int(max_pos), _ptr(workspace),
                                int(workspace_bytes), _ptr(dev_status), _stream(stream))
    return _check(st, "kev_rope_prefill", check)


def kev_prefill_attn_rope(q, k, v, total_tokens, intervals, n_questions, slot_ids, pool_k, pool_v, n_slots,
                          slot_cap, out, shape, rope_table, max_pos, workspace, workspace_bytes, dev_status=None,
                          stream=None, check=True) -> int:
    s = _shape(shape)
    st = _c["kev_prefill_attn_rope"](_ptr(q), _ptr(k), _ptr(v), int(total_tokens), _ptr(intervals),
                                     int(n_questions), _ptr(slot_ids), _ptr(pool_k), _ptr(pool_v), int(n_slots),
                                     int(slot_cap), _ptr(out), ctypes.byref(s), _ptr(rope_table), int(max_pos),
                                     _ptr(workspace), int(workspace_bytes), _ptr(dev_status), _stream(stream))
    return _check(st, "kev_prefill_attn_rope", check)


def kev_rope_decode(q_new, k_new, lens, active, n_questions, shape, rope_table, max_pos, dev_status=None,
                    stream=None, check=True) -> int:
    s = _shape(shape)
    st = _c["kev_rope_decode"](_ptr(q_new), _ptr(k_new), _ptr(lens), _ptr(active), int(n_questions),
                               ctypes.byref(s), _ptr(rope_table), int(max_pos), _ptr(dev_status), _stream(stream))
    return _check(st, "kev_rope_decode", check)


def kev_decode_attn_rope(q_new, k_new, v_new, pool_k, pool_v, n_slots, slot_cap, slot_ids, lens, active,
                         n_questions, out, shape, rope_table, max_pos, workspace, workspace_bytes, dev_status=None,
                         stream=None, check=True) -> int:
    s = _shape(shape)
    st = _c["kev_decode_attn_rope"](_ptr(q_new), _ptr(k_new), _ptr(v_new), _ptr(pool_k), _ptr(pool_v),
                                    int(n_slots), int(slot_cap), _ptr(slot_ids), _ptr(lens), _ptr(active),
                                    int(n_questions), _ptr(out), ctypes.byref(s), _ptr(rope_table), int(max_pos),
                                    _ptr(workspace), int(workspace_bytes), _ptr(dev_status), _stream(stream))
    return _check(st, "kev_decode_attn_rope", check)


def kev_prefill_attn_paged(q, k, v, total_tokens, intervals, n_questions, block_table, max_blocks, pool_k, pool_v,
                           n_blocks, out, shape, workspace, workspace_bytes, dev_status=None, stream=None,
                           check=True) -> int:
    s = _shape(shape)
    st = _c["kev_prefill_attn_paged"](_ptr(q), _ptr(k), _ptr(v), int(total_tokens), _ptr(intervals),
                                      int(n_questions), _ptr(block_table), int(max_blocks), _ptr(pool_k),
                                      _ptr(pool_v), int(n_blocks), _ptr(out), ctypes.byref(s), _ptr(workspace),
                                      int(workspace_bytes), _ptr(dev_status), _stream(stream))
    return _check(st, "kev_prefill_attn_paged", check)


def kev_kv_write_paged(k, v, total_tokens, intervals, n_questions, block_table, max_blocks, pool_k, pool_v, n_blocks,
                       shape, workspace, workspace_bytes, dev_status=None, stream=None, check=True) -> int:
    s = _shape(shape)
    st = _c["kev_kv_write_paged"](_ptr(k), _ptr(v), int(total_tokens), _ptr(intervals), int(n_questions),
                                  _ptr(block_table), int(max_blocks), _ptr(pool_k), _ptr(pool_v), int(n_blocks),
                                  ctypes.byref(s), _ptr(workspace), int(workspace_bytes), _ptr(dev_status),
                                  _stream(stream))
    return _check(st, "kev_kv_write_paged", check)


def kev_decode_attn_paged(q_new, k_new, v_new, pool_k, pool_v, n_blocks, block_table, max_blocks, lens, active,
                          n_questions, out, shape, workspace, workspace_bytes, dev_status=None, stream=None,
                          check=True) -> int:
    s = _shape(shape)
    st = _c["kev_decode_attn_paged"](_ptr(q_new), _ptr(k_new), _ptr(v_new), _ptr(pool_k), _ptr(pool_v),
                                     int(n_blocks), _ptr(block_table), int(max_blocks), _ptr(lens), _ptr(active),
                                     int(n_questions), _ptr(out), ctypes.byref(s), _ptr(workspace),
                                     int(workspace_bytes), _ptr(dev_status), _stream(stream))
    return _check(st, "kev_decode_attn_paged", check)


def kev_assign_blocks(need, free_map, max_blocks: int, contiguous_first: bool = True):
    """Host block assignment (no CUDA call).  ``need``: ints per question; ``free_map``: numpy
    uint8/bool array (1 = free), updated in place on success.  Returns the table as a numpy
    int32 [n, max_blocks] array, or None when the free blocks do not suffice."""
    import numpy as np
    nd = np.ascontiguousarray(need, dtype=np.int32)
    fm = np.ascontiguousarray(free_map, dtype=np.uint8)
    table = np.empty((len(nd), int(max_blocks)), dtype=np.int32)
    r = _c["kev_assign_blocks"](nd.ctypes.data, len(nd), fm.ctypes.data, len(fm), table.ctypes.data,
                                int(max_blocks), int(bool(contiguous_first)))
    if r != 0:
        return None
    free_map[...] = fm.astype(np.asarray(free_map).dtype)
    return table


def kev_prefill_chunk(q, k, v, total_tokens, intervals, n_questions, prefix_lens, slot_ids, pool_k, pool_v, n_slots,
                      slot_cap, out, shape, workspace, workspace_bytes, dev_status=None, stream=None,
                      check=True) -> int:
    s = _shape(shape)
    st = _c["kev_prefill_chunk"](_ptr(q), _ptr(k), _ptr(v), int(total_tokens), _ptr(intervals), int(n_questions),
                                 _ptr(prefix_lens), _ptr(slot_ids), _ptr(pool_k), _ptr(pool_v), int(n_slots),
                                 int(slot_cap), _ptr(out), ctypes.byref(s), _ptr(workspace), int(workspace_bytes),
                                 _ptr(dev_status), _stream(stream))
    return _check(st, "kev_prefill_chunk", check)


def kev_sample(logits, n_questions, vocab, dtype, temperature, uniforms, active, tokens, dev_status=None, stream=None,
               check=True) -> int:
    if isinstance(dtype, str):
        dtype = {"bf16": KEV_BF16, "fp32": KEV_FP32}[dtype]
    st = _c["kev_sample"](_ptr(logits), int(n_questions), int(vocab), int(dtype), _ptr(temperature), _ptr(uniforms),
                          _ptr(active), _ptr(tokens), _ptr(dev_status), _stream(stream))
    return _check(st, "kev_sample", check)


def kev_lora_apply(x, y, total_tokens, d_in, d_out, intervals, n_questions, adapter_ids, lora_a, lora_b, scales,
                   n_adapters, rank, workspace, workspace_bytes, dev_status=None, stream=None, check=True) -> int:
    st = _c["kev_lora_apply"](_ptr(x), _ptr(y), int(total_tokens), int(d_in), int(d_out), _ptr(intervals),
                              int(n_questions), _ptr(adapter_ids), _ptr(lora_a), _ptr(lora_b), _ptr(scales),
                              int(n_adapters), int(rank), _ptr(workspace), int(workspace_bytes), _ptr(dev_status),
                              _stream(stream))
    return _check(st, "kev_lora_apply", check)
