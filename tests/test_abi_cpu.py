"""The C-ABI library builds, loads and exports what include/sink_attn.h
declares; host-side validation rejects bad arguments before any launch.
CPU only: no call here reaches a kernel."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sink_attn.h")


@pytest.fixture(scope="module")
def lib():
    import gqa_attention_sinks_head_gb300 as sa
    sa.build()
    sa.load()
    return sa


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    for n in ["sa_decode", "sa_decode_partial", "sa_merge_states", "sa_prefill", "sa_decode_workspace_size",
              "sa_decode_num_splits", "sa_device_status", "sa_status_string", "sa_last_error", "sa_version"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(lib._LIB_PATH)
    for n in declared_functions():
        assert hasattr(raw, n), n
    assert set(lib.EXPORTS) == set(declared_functions())


def test_version_and_status_strings(lib):
    L = lib.load()
    assert L.sa_version() == 10000
    for i, name in enumerate(["SA_OK", "SA_ERR_INVALID_ARG", "SA_ERR_UNSUPPORTED", "SA_ERR_WORKSPACE",
                              "SA_ERR_CUDA", "SA_ERR_TIMEOUT"]):
        assert L.sa_status_string(i).decode() == name


def _desc(lib, **over):
    d = lib.KVDesc()
    d.k = 4096
    d.v = 8192
    d.dtype = 0
    d.num_pages = 10
    d.num_kv_heads = 8
    d.head_dim = 64
    d.page_size = 16
    d.page_table_stride = 64
    d.stride_page = 8 * 16 * 64
    d.stride_head = 16 * 64
    d.stride_token = 64
    d.page_table = 1024
    d.k_scale = 1.0
    d.v_scale = 1.0
    for k, v in over.items():
        setattr(d, k, v)
    return d


def _decode(lib, d, **kw):
    L = lib.load()
    a = dict(q=4096, seqlens=512, batch=2, hq=64, maxlen=1000, sinks=None, window=0, scale=0.125, out=8192,
             lse=None, ws=None, wsb=0, splits=1)
    a.update(kw)
    return L.sa_decode(a["q"], ctypes.byref(d), a["seqlens"], a["batch"], a["hq"], a["maxlen"], a["sinks"],
                       a["window"], a["scale"], a["out"], a["lse"], a["ws"], a["wsb"], a["splits"], None)


@pytest.mark.parametrize("over,kw,expect", [
    ({}, dict(hq=60), 1),                                  # Hq not a multiple of Hkv
    ({"head_dim": 128}, {}, 2),                            # only head_dim 64
    ({"page_size": 8}, {}, 2),                             # page size not a multiple of 16
    ({"dtype": 7}, {}, 1),                                 # bad dtype
    ({"k": 0}, {}, 1),                                     # NULL cache
    ({"k": 4100}, {}, 2),                                  # misaligned cache
    ({"stride_token": 60}, {}, 2),                         # stride not 16-byte aligned
    ({"page_table_stride": 10}, {}, 1),                    # table rows too short for max_kv_len
    ({}, dict(window=-1), 1),
    ({}, dict(batch=-1), 1),
    ({}, dict(scale=float("inf")), 1),
    ({}, dict(hq=128), 2),                                 # 16 query heads per kv head
    ({}, dict(splits=-2), 1),
    ({}, dict(splits=4, ws=None, wsb=0), 3),               # split without workspace
    ({"page_table": None, "num_pages": 1}, {}, 1),         # contiguous needs a page per sequence
    ({"dtype": 1, "k_scale": float("nan")}, {}, 1),
])
def test_decode_argument_validation(lib, over, kw, expect):
    d = _desc(lib, **over)
    assert _decode(lib, d, **kw) == expect
    assert lib.load().sa_last_error().decode() != ""


def test_batch_zero_is_a_noop(lib):
    assert _decode(lib, _desc(lib), batch=0, q=None, seqlens=None, out=None) == 0


def test_merge_validation(lib):
    L = lib.load()
    assert L.sa_merge_states(4096, 4096, 0, 4, 8, 64, None, 4096, None, None) == 1
    assert L.sa_merge_states(4096, 4096, 2, 4, 8, 62, None, 4096, None, None) == 2
    assert L.sa_merge_states(4096, 4096, 2, 0, 8, 64, None, 4096, None, None) == 0


def test_workspace_size(lib):
    assert lib.sa_decode_workspace_size(4, 64, 8, 64, 1000, 0, 1) == 0
    s = lib.sa_decode_workspace_size(4, 64, 8, 64, 1000, 0, 3)
    assert s >= 3 * 4 * 64 * 65 * 4
    assert s % 256 == 0


def test_split_heuristic_is_deterministic_and_bounded(lib):
    for args in [(64, 8, 8192, 0), (128, 8, 32768, 0), (1, 8, 256, 0), (256, 8, 8192, 128), (1, 1, 1, 0)]:
        s = lib.sa_decode_num_splits(*args)
        assert 1 <= s <= 256
        assert s == lib.sa_decode_num_splits(*args)
    assert lib.sa_decode_num_splits(256, 8, 8192, 128) <= 2   # a 128-key window needs no split
    assert lib.sa_decode_num_splits(1, 8, 32768, 0) > 8        # one long sequence is spread out


def _decode_multi(lib, d, q_len, **kw):
    L = lib.load()
    a = dict(q=4096, seqlens=512, batch=2, hq=64, maxlen=1000, sinks=None, window=0, scale=0.125, out=8192,
             lse=None, ws=None, wsb=0, splits=1)
    a.update(kw)
    return L.sa_decode_multi(a["q"], q_len, ctypes.byref(d), a["seqlens"], a["batch"], a["hq"], a["maxlen"],
                             a["sinks"], a["window"], a["scale"], a["out"], a["lse"], a["ws"], a["wsb"], a["splits"],
                             None)


@pytest.mark.parametrize("q_len,expect", [(0, 2), (-1, 2), (9, 2), (64, 2)])
def test_decode_multi_token_count(lib, q_len, expect):
    assert _decode_multi(lib, _desc(lib), q_len) == expect
    assert "q_len" in lib.load().sa_last_error().decode()


def test_decode_multi_validation_matches_decode(lib):
    # the shared checks run first: a bad cache is refused whatever q_len is
    assert _decode_multi(lib, _desc(lib, head_dim=128), 4) == 2
    assert _decode_multi(lib, _desc(lib), 4, splits=4, ws=None, wsb=0) == 3
    assert _decode_multi(lib, _desc(lib), 4, batch=0, q=None, seqlens=None, out=None) == 0


def test_multi_token_split_count(lib):
    """sa_decode_multi_num_splits: the one-token count for q_len 1 and for FP8
    caches; for q_len >= 2 on bf16 the tensor-core kernel (two blocks per SM)
    takes no more chunks; the automatic workspace covers either choice."""
    L = lib.load()
    for B, Hkv, Lmax, w in [(64, 8, 8192, 0), (1, 8, 32768, 0), (4, 8, 4096, 0), (256, 8, 8192, 128), (1, 1, 1, 0)]:
        one = L.sa_decode_num_splits(B, Hkv, Lmax, w)
        assert L.sa_decode_multi_num_splits(B, 1, Hkv, Lmax, w, lib.SA_KV_BF16) == one
        for q_len in (2, 4, 8):
            assert L.sa_decode_multi_num_splits(B, q_len, Hkv, Lmax, w, lib.SA_KV_FP8_E4M3) == one
            s = L.sa_decode_multi_num_splits(B, q_len, Hkv, Lmax, w, lib.SA_KV_BF16)
            assert 1 <= s <= one
            auto = L.sa_decode_multi_workspace_size(B, q_len, 64, Hkv, 64, Lmax, w, 0)
            assert auto == L.sa_decode_multi_workspace_size(B, q_len, 64, Hkv, 64, Lmax, w, max(s, one))
    assert L.sa_decode_multi_num_splits(1, 4, 8, 32768, 0, lib.SA_KV_BF16) > 4  # one long sequence is spread out


def test_decode_multi_workspace_size(lib):
    assert lib.sa_decode_multi_workspace_size(4, 3, 64, 8, 64, 1000, 0, 1) == 0
    s = lib.sa_decode_multi_workspace_size(4, 3, 64, 8, 64, 1000, 0, 5)
    assert s == lib.sa_decode_workspace_size(12, 64, 8, 64, 1000, 0, 5)  # rows = batch * q_len


def test_prefill_q8_needs_an_fp8_cache(lib):
    L = lib.load()
    d = _desc(lib)  # bf16 cache
    rc = L.sa_prefill_q8(4096, 0.1, 4096, 10, ctypes.byref(d), 4096, 2, 64, 5, 100, None, 0, 0.125, 4096, None, None)
    assert rc == 2 and "FP8" in L.sa_last_error().decode()
    d = _desc(lib, dtype=1)
    rc = L.sa_prefill_q8(4096, float("nan"), 4096, 10, ctypes.byref(d), 4096, 2, 64, 5, 100, None, 0, 0.125, 4096,
                         None, None)
    assert rc == 1
