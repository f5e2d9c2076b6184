"""CPU checks of the C ABI: the library loads, exports every declared symbol, and host-side
argument checks answer without a GPU (no compute call is made here)."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from packed_question_isolated_gb300 import build
    build.build()
    import packed_question_isolated_gb300 as kev
    return kev


def _declared():
    text = open(os.path.join(ROOT, "include", "kev.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kev_[a-z_]+)\s*\(", text)))


def test_header_constants_match_the_binding(lib):
    """Every integer #define and every kev_status / kev_dtype enumerator of kev.h has the same
    value in the Python binding (the binding copies them by hand)."""
    b = lib.binding
    text = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "kev.h")).read(), flags=re.S)
    consts = {}
    for name, val in re.findall(r"#define\s+(KEV_[A-Z0-9_]+)\s+([0-9]+)\s*$", text, flags=re.M):
        consts[name] = int(val)
    for name, val, shift in re.findall(r"#define\s+(KEV_[A-Z0-9_]+)\s+\(([0-9]+)u\s*<<\s*([0-9]+)\)", text):
        consts[name] = int(val) << int(shift)
    for name, val in re.findall(r"\b(KEV_[A-Z0-9_]+)\s*=\s*([0-9]+)", text):
        consts[name] = int(val)
    assert {"KEV_OK", "KEV_ERR_ADAPTER", "KEV_BF16", "KEV_PAGE", "KEV_MAX_QUESTIONS"} <= set(consts)
    for name, val in consts.items():
        assert getattr(b, name) == val, name


def test_workspace_sizes_at_the_int32_limit(lib):
    """Sizes for the largest token count and slot capacity an int32 holds: computed without
    overflow (monotone in T and cap, and at least the bytes of the work list they hold)."""
    big = 2 ** 31 - 1
    shape = lib.make_shape(4, 2, 128, "bf16")
    s_big = lib.kev_prefill_workspace_size(1, big, shape)
    s_less = lib.kev_prefill_workspace_size(1, big - 1000, shape)
    assert s_big >= s_less > 0
    assert s_big >= 16 * 4 * (big // 128)  # an int4 work item per (query tile, q-head)
    d_big = lib.kev_decode_workspace_size(8, big, shape)
    d_less = lib.kev_decode_workspace_size(8, big - 1000, shape)
    assert d_big >= d_less > 0


def test_every_declared_symbol_is_exported(lib):
    so = ctypes.CDLL(lib.library_path())
    declared = _declared()
    assert len(declared) >= 12
    for name in declared:
        assert hasattr(so, name), f"{name} declared in kev.h but not exported"
    assert set(declared) == set(lib.binding.EXPORTED)


def test_status_strings_and_launch_counts(lib):
    for code in range(12):
        assert lib.kev_status_string(code) != "unknown status"
    assert lib.kev_status_string(99) == "unknown status"
    assert lib.kev_launch_count(0) == 3 and lib.kev_launch_count(4) == 1 and lib.kev_launch_count(99) == -1
    assert [lib.kev_launch_count(i) for i in (6, 7, 8, 9, 10, 11, 12, 13, 14, 15)] == [1, 1, 1, 4, 3, 2, 3, 1, 1, 2]


def test_workspace_sizes(lib):
    s = lib.make_shape(28, 4, 128, "bf16")
    n, T = 8, 7921
    sz = lib.kev_prefill_workspace_size(n, T, s)
    max_tiles = (T + 127) // 128 + n
    assert sz >= max_tiles * 28 * 16 + max_tiles * 8 + (n + 1) * 4
    assert lib.kev_prefill_workspace_size(n, T, lib.make_shape(28, 5, 128)) == 0   # H_q % H_kv
    assert lib.kev_prefill_workspace_size(n, T, lib.make_shape(28, 4, 96)) == 0    # d_h
    # fp32 runs on the CUDA cores at any head dim that is a multiple of 16 up to 256
    for d in (16, 48, 96, 256):
        assert lib.kev_prefill_workspace_size(n, T, lib.make_shape(28, 4, d, "fp32")) > 0
        assert lib.kev_decode_workspace_size(n, 512, lib.make_shape(28, 4, d, "fp32")) > 0
    for d in (8, 100, 272):
        assert lib.kev_prefill_workspace_size(n, T, lib.make_shape(28, 4, d, "fp32")) == 0
    assert lib.kev_prefill_workspace_size(5000, T, s) == 0                          # too many questions
    d = lib.kev_decode_workspace_size(64, 2458, lib.make_shape(32, 8, 128))
    assert d >= 64 * 8 * 4 + 64 * 8 * ((2458 + 255) // 256) * 4 * 130 * 4


def test_host_argument_errors_without_gpu(lib):
    b = lib.binding
    s = lib.make_shape(4, 2, 64, "bf16")
    # null workspace / misaligned pointers / bad shape are refused before any CUDA call
    assert lib.kev_build_segments(None, 1, 10, None, 0, 0, s, None, 0, None, stream=0, check=False) == \
        b.KEV_ERR_INVALID_ARG
    assert lib.kev_prefill_attn(0x1000, 0x1000, 0x1000, 10, 0x1000, 1, None, None, None, 0, 0, 0x1000,
                                lib.make_shape(4, 3, 64), 0x1000, 1 << 20, None, stream=0, check=False) == \
        b.KEV_ERR_UNSUPPORTED
    assert lib.kev_prefill_attn(0x1000, 0x1000, 0x1000, 10, 0x1000, 1, None, None, None, 0, 0, 0x1000,
                                s, 0x1010, 1 << 20, None, stream=0, check=False) == b.KEV_ERR_INVALID_ARG
    assert lib.kev_decode_attn(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 1, 0, 0x1000, 0x1000, 0x1000, 1, 0x1000,
                               s, 0x1000, 1 << 20, None, stream=0, check=False) == b.KEV_ERR_INVALID_ARG
    assert lib.kev_decode_advance(None, None, -1, stream=0, check=False) == b.KEV_ERR_INVALID_ARG
    with pytest.raises(b.KevError):
        lib.kev_decode_advance(None, None, -1, stream=0)


def test_rope_table_size_and_host_errors_without_gpu(lib):
    b = lib.binding
    assert lib.kev_rope_table_size(4224, 128) == 4224 * 64 * 8
    assert lib.kev_rope_table_size(0, 128) == 0 and lib.kev_rope_table_size(16, 63) == 0
    s = lib.make_shape(4, 2, 64, "bf16")
    assert lib.kev_rope_table(None, 16, 64, 1e4, stream=0, check=False) == b.KEV_ERR_INVALID_ARG
    assert lib.kev_rope_table(0x1000, 16, 96, 1e4, stream=0, check=False) == b.KEV_ERR_UNSUPPORTED
    assert lib.kev_rope_table(0x1000, 16, 64, 1.0, stream=0, check=False) == b.KEV_ERR_INVALID_ARG
    assert lib.kev_rope_table(0x1008, 16, 64, 1e4, stream=0, check=False) == b.KEV_ERR_INVALID_ARG
    # RoPE pairs 16-byte chunks of a head's halves: head dims 64 and 128 only (fp32 attention
    # itself takes any multiple of 16 up to 256)
    s96 = lib.make_shape(4, 2, 96, "fp32")
    assert lib.kev_rope_prefill(0x1000, 0x1000, 0x1000, 10, 0x1000, 1, None, None, None, 0, 0, s96, 0x1000, 16,
                                0x1000, 1 << 20, None, stream=0, check=False) == b.KEV_ERR_UNSUPPORTED
    assert lib.kev_prefill_attn_rope(0x1000, 0x1000, 0x1000, 10, 0x1000, 1, None, None, None, 0, 0, 0x1000, s96,
                                     0x1000, 16, 0x1000, 1 << 20, None, stream=0, check=False) == b.KEV_ERR_UNSUPPORTED
    assert lib.kev_rope_decode(0x1000, 0x1000, 0x1000, 0x1000, 1, s96, 0x1000, 16, None, stream=0,
                               check=False) == b.KEV_ERR_UNSUPPORTED
    # no table / misaligned table / bad max_pos are refused before any CUDA call
    assert lib.kev_rope_prefill(0x1000, 0x1000, 0x1000, 10, 0x1000, 1, None, None, None, 0, 0, s, None, 16,
                                0x1000, 1 << 20, None, stream=0, check=False) == b.KEV_ERR_INVALID_ARG
    assert lib.kev_rope_decode(0x1000, 0x1000, 0x1000, 0x1000, 1, s, 0x1008, 16, None, stream=0,
                               check=False) == b.KEV_ERR_INVALID_ARG
    assert lib.kev_rope_decode(0x1000, 0x1000, 0x1000, 0x1000, 1, s, 0x1000, 0, None, stream=0,
                               check=False) == b.KEV_ERR_INVALID_ARG
    # the decode-side table must cover the slot
    assert lib.kev_decode_attn_rope(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 1, 64, 0x1000, 0x1000, 0x1000, 1,
                                    0x1000, s, 0x1000, 32, 0x1000, 1 << 20, None, stream=0, check=False) == \
        b.KEV_ERR_INVALID_ARG


def test_assign_blocks_matches_the_oracle(lib):
    """Host logic, no GPU: the library's contiguous-first block assignment against the oracle's."""
    from oracle import kev_oracle as O
    free = np.array([1, 1, 0, 1, 1, 1, 0, 1], np.uint8)
    assert lib.kev_assign_blocks([2, 2, 2], free, 3).tolist() == [[0, 1, -1], [3, 4, -1], [5, 7, -1]]
    assert not free.any()
    rng = np.random.default_rng(1)
    for it in range(300):
        fr = rng.random(64) < 0.6
        need = rng.integers(0, 6, 8)
        cf = bool(it % 2)
        ref = O.assign_blocks(need, fr, 5, contiguous_first=cf)
        fm = fr.astype(np.uint8)
        got = lib.kev_assign_blocks(need, fm, 5, contiguous_first=cf)
        if ref is None:
            assert got is None and (fm.astype(bool) == fr).all()  # nothing taken on failure
        else:
            np.testing.assert_array_equal(got, ref[0])
            np.testing.assert_array_equal(fm.astype(bool), ref[1])


def test_paged_host_errors_without_gpu(lib):
    b = lib.binding
    s = lib.make_shape(4, 2, 128, "bf16")
    # no table, a misaligned table, too many entries, a decode shape off the tensor cores
    assert lib.kev_prefill_attn_paged(0x1000, 0x1000, 0x1000, 10, 0x1000, 1, None, 4, 0x1000, 0x1000, 8, 0x1000, s,
                                      0x1000, 1 << 20, None, stream=0, check=False) == b.KEV_ERR_INVALID_ARG
    assert lib.kev_kv_write_paged(0x1000, 0x1000, 10, 0x1000, 1, 0x1002, 4, 0x1000, 0x1000, 8, s, 0x1000, 1 << 20,
                                  None, stream=0, check=False) == b.KEV_ERR_INVALID_ARG
    assert lib.kev_decode_attn_paged(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 8, 0x1000, 20000, 0x1000, 0x1000, 1,
                                     0x1000, s, 0x1000, 1 << 20, None, stream=0, check=False) == b.KEV_ERR_UNSUPPORTED
    assert lib.kev_decode_attn_paged(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 8, 0x1000, 4, 0x1000, 0x1000, 1,
                                     0x1000, lib.make_shape(4, 2, 64, "bf16"), 0x1000, 1 << 20, None, stream=0,
                                     check=False) == b.KEV_ERR_UNSUPPORTED


def test_chunk_host_errors_without_gpu(lib):
    b = lib.binding
    s = lib.make_shape(4, 2, 128, "bf16")
    args = (0x1000, 0x1000, 0x1000, 10, 0x1000, 1, 0x1000, 0x1000, 0x1000, 0x1000, 4)
    # slot capacity not a multiple of 128, fp32, no prefix array, no slots
    assert lib.kev_prefill_chunk(*args, 2458, 0x1000, s, 0x1000, 1 << 20, None, stream=0, check=False) == \
        b.KEV_ERR_UNSUPPORTED
    assert lib.kev_prefill_chunk(*args, 2560, 0x1000, lib.make_shape(4, 2, 128, "fp32"), 0x1000, 1 << 20, None,
                                 stream=0, check=False) == b.KEV_ERR_UNSUPPORTED
    assert lib.kev_prefill_chunk(0x1000, 0x1000, 0x1000, 10, 0x1000, 1, None, 0x1000, 0x1000, 0x1000, 4, 2560,
                                 0x1000, s, 0x1000, 1 << 20, None, stream=0, check=False) == b.KEV_ERR_INVALID_ARG
    assert lib.kev_prefill_chunk(0x1000, 0x1000, 0x1000, 10, 0x1000, 1, 0x1000, None, 0x1000, 0x1000, 4, 2560,
                                 0x1000, s, 0x1000, 1 << 20, None, stream=0, check=False) == b.KEV_ERR_INVALID_ARG


def test_sample_host_errors_without_gpu(lib):
    b = lib.binding
    args = (0x1000, 0x1000, 0x1000, 0x1000)
    assert lib.kev_sample(0x1000, 2, 0, "bf16", *args, None, stream=0, check=False) == b.KEV_ERR_INVALID_ARG
    assert lib.kev_sample(0x1000, 2, 100, "bf16", *args, None, stream=0, check=False) == b.KEV_ERR_UNSUPPORTED
    assert lib.kev_sample(0x1000, 2, 128, 7, *args, None, stream=0, check=False) == b.KEV_ERR_UNSUPPORTED
    assert lib.kev_sample(0x1008, 2, 128, "bf16", *args, None, stream=0, check=False) == b.KEV_ERR_INVALID_ARG
    assert lib.kev_sample(None, 0, 128, "bf16", None, None, None, None, None, stream=0, check=False) == b.KEV_OK
    # more questions than a call takes (the library's limit, the same for every entry point)
    assert lib.kev_sample(0x1000, b.KEV_MAX_QUESTIONS + 1, 128, "bf16", *args, None, stream=0, check=False) == \
        b.KEV_ERR_UNSUPPORTED


def test_lora_host_errors_without_gpu(lib):
    b = lib.binding
    args = (0x1000, 0x1000, 0x1000, 0x1000, 3)  # adapter ids, lora_a, lora_b, scales, n_adapters
    # rank, d_in, d_out outside what the kernel takes; a misaligned workspace
    assert lib.kev_lora_apply(0x1000, 0x1000, 10, 256, 256, 0x1000, 1, *args, 8, 0x1000, 1 << 20, None, stream=0,
                              check=False) == b.KEV_ERR_UNSUPPORTED
    assert lib.kev_lora_apply(0x1000, 0x1000, 10, 240, 256, 0x1000, 1, *args, 16, 0x1000, 1 << 20, None, stream=0,
                              check=False) == b.KEV_ERR_UNSUPPORTED
    assert lib.kev_lora_apply(0x1000, 0x1000, 10, 256, 248, 0x1000, 1, *args, 16, 0x1000, 1 << 20, None, stream=0,
                              check=False) == b.KEV_ERR_UNSUPPORTED
    assert lib.kev_lora_apply(0x1000, 0x1000, 10, 256, 256, 0x1000, 1, *args, 16, 0x1010, 1 << 20, None, stream=0,
                              check=False) == b.KEV_ERR_INVALID_ARG
