"""fp64 CPU oracle for sink attention (grouped-query attention with per-head
attention sinks).

TEST INFRASTRUCTURE ONLY: imported by tests/, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``, never by the library.  The
arithmetic lives in ``sa_oracle.c`` (plain C, fp64, two-pass definition); this
module compiles it with gcc, loads it with ctypes and marshals numpy arrays.

The query-position conventions are part of the definition and live here:
  * decode: the query of sequence b sits at position L_b - 1 (its own key and
    value are already in the cache);
  * prefill: queries are bottom-right aligned, query i of a sequence holding
    L_q queries and L_kv keys sits at position L_kv - L_q + i.
Sources: "GPT-OSS on day 0" (Perplexity), sections "Attention: GQA with
attention sinks" and "GPT-OSS kernels / Sink Attention"; NVIDIA gpt-oss launch
article, introduction (full context alternating with a 128-token window).

Every function here is pinned by tests/test_oracle_pins.py against things other
than itself: a pure-Python brute force, the SDPA identity with one extra key,
closed forms, the limiting cases of the sink, the all-codes E4M3 table of
torch, and split invariance.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libsaoracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile sa_oracle.c into oracle/_build/libsaoracle.so (gcc, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    base = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)  # no OpenMP: one thread
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _KV(ctypes.Structure):
    _fields_ = [
        ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("dtype", ctypes.c_int32),
        ("num_pages", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
        ("stride_page", ctypes.c_int64), ("stride_head", ctypes.c_int64),
        ("stride_token", ctypes.c_int64), ("page_table", ctypes.c_void_p),
        ("page_table_stride", ctypes.c_int32), ("k_scale", ctypes.c_double),
        ("v_scale", ctypes.c_double),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # SA_ORACLE_LIB: load a different build of sa_oracle.c (the mutation
            # tests point it at copies with planted mistakes)
            lib = ctypes.CDLL(os.environ.get("SA_ORACLE_LIB") or build())
            P = ctypes.c_void_p
            lib.sao_attend.restype = ctypes.c_int
            lib.sao_attend.argtypes = [P, ctypes.c_int32, ctypes.c_int32, P, P, ctypes.POINTER(_KV), P,
                                       P, ctypes.c_int32, ctypes.c_double, P, P, ctypes.c_int64, P, P]
            lib.sao_attend_q8.restype = ctypes.c_int
            lib.sao_attend_q8.argtypes = [P, ctypes.c_double] + lib.sao_attend.argtypes[1:]
            lib.sao_attend_range.restype = ctypes.c_int
            lib.sao_attend_range.argtypes = lib.sao_attend.argtypes[:13] + [ctypes.c_int32, ctypes.c_int32,
                                                                             P, P]
            lib.sao_attend_split.restype = ctypes.c_int
            lib.sao_attend_split.argtypes = [P, ctypes.c_int32, ctypes.c_int32, P, P, ctypes.POINTER(_KV),
                                             P, P, ctypes.c_int32, ctypes.c_double, P, P, ctypes.c_int64,
                                             ctypes.c_int32, ctypes.c_int32, P, P, P, P]
            lib.sao_merge.restype = None
            lib.sao_merge.argtypes = [P, P, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                      P, P, P]
            lib.sao_bf16_array.argtypes = [P, ctypes.c_int64, P]
            lib.sao_e4m3_array.argtypes = [P, ctypes.c_int64, P]
            lib.sao_num_threads.restype = ctypes.c_int
            lib.sao_set_num_threads.restype = None
            lib.sao_set_num_threads.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().sao_num_threads())


def set_num_threads(n: int) -> None:
    """Threads of the oracle's next parallel loops (for timing; the results do not depend on it)."""
    _load().sao_set_num_threads(int(n))


# ---------------------------------------------------------------- marshalling
def _np(x, dtype=None):
    """numpy view of a CPU torch tensor or array; bf16 -> uint16 bits, fp8 -> uint8 codes."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                x = x.view(torch.int16).numpy().view(np.uint16)
            elif x.dtype in (torch.float8_e4m3fn,):
                x = x.view(torch.uint8).numpy()
            else:
                x = x.numpy()
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if dtype is not None and x.dtype != dtype:
        x = x.astype(dtype)
    return x


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _kv_struct(kv: dict, keep: list) -> _KV:
    k = _np(kv["k"])
    v = _np(kv["v"])
    if kv.get("dtype", "bf16") == "bf16":
        k = k.view(np.uint16)
        v = v.view(np.uint16)
        dt = 0
    else:
        k = k.view(np.uint8)
        v = v.view(np.uint8)
        dt = 1
    table = kv.get("page_table")
    table = None if table is None else _np(table, np.int32)
    keep += [k, v, table]
    s = _KV()
    s.k = k.ctypes.data
    s.v = v.ctypes.data
    s.dtype = dt
    s.num_pages = int(kv["num_pages"])
    s.num_kv_heads = int(kv["num_kv_heads"])
    s.head_dim = int(kv["head_dim"])
    s.page_size = int(kv["page_size"])
    s.stride_page = int(kv["stride_page"])
    s.stride_head = int(kv["stride_head"])
    s.stride_token = int(kv["stride_token"])
    s.page_table = None if table is None else table.ctypes.data
    s.page_table_stride = int(kv.get("page_table_stride", 0 if table is None else table.shape[-1]))
    s.k_scale = float(kv.get("k_scale", 1.0))
    s.v_scale = float(kv.get("v_scale", 1.0))
    return s


# ------------------------------------------------------------ query positions
def decode_rows(seqlens):
    """Decode: row b belongs to sequence b and sits at position L_b - 1."""
    L = _np(seqlens, np.int32)
    return np.arange(L.shape[0], dtype=np.int32), (L - 1).astype(np.int32)


def prefill_rows(cu_seqlens_q, seqlens_kv):
    """Prefill: rows cu[b] .. cu[b+1]-1 belong to sequence b; row cu[b]+i sits
    at position L_kv,b - L_q,b + i (bottom-right aligned)."""
    cu = _np(cu_seqlens_q, np.int64)
    Lkv = _np(seqlens_kv, np.int64)
    n = int(cu[-1])
    seq = np.empty(n, np.int32)
    pos = np.empty(n, np.int32)
    for b in range(cu.shape[0] - 1):
        lq = int(cu[b + 1] - cu[b])
        seq[cu[b]:cu[b + 1]] = b
        pos[cu[b]:cu[b + 1]] = Lkv[b] - lq + np.arange(lq)
    return seq, pos


# ------------------------------------------------------------------ the math
def attend(q, row_seq, row_pos, kv: dict, seqlens, sinks, window: int, sm_scale: float,
           sel_rows=None, sel_heads=None, split=None, key_range=None, q_scale=None):
    """out [n_sel, D] and lse [n_sel] (fp64) for the selected (row, head) pairs.

    q: bf16 [n_rows, Hq, D], or E4M3 codes (uint8) when q_scale is given
    (element = code * q_scale); kv: dict with k, v, dtype ('bf16' | 'e4m3'),
    num_pages, num_kv_heads, head_dim, page_size, strides (elements),
    page_table ([B, max_pages] int32 or None), k_scale, v_scale.
    sel_rows/sel_heads default to every (row, head).  split=(num_chunks, chunk)
    evaluates the chunked form (sink-free partials merged with the sink once).
    key_range=(lo, hi) restricts the keys to [lo, hi): with sinks=None that is
    the sink-free partial state of one chunk.
    """
    lib = _load()
    keep = []
    qa = _np(q).view(np.uint8 if q_scale is not None else np.uint16)
    n_rows, Hq, D = qa.shape
    row_seq = _np(row_seq, np.int32)
    row_pos = _np(row_pos, np.int32)
    seqlens = _np(seqlens, np.int32)
    sinks_a = None if sinks is None else _np(sinks, np.float32)
    if sel_rows is None:
        rr, hh = np.meshgrid(np.arange(n_rows, dtype=np.int32), np.arange(Hq, dtype=np.int32), indexing="ij")
        sel_rows, sel_heads = rr.reshape(-1), hh.reshape(-1)
    sel_rows = _np(sel_rows, np.int32)
    sel_heads = _np(sel_heads, np.int32)
    n_sel = sel_rows.shape[0]
    kvs = _kv_struct(kv, keep)
    out = np.zeros((n_sel, D), np.float64)
    lse = np.zeros((n_sel,), np.float64)
    if q_scale is not None:
        if key_range is not None or split is not None:
            raise ValueError("an E4M3 query is supported by the plain definition only")
        rc = lib.sao_attend_q8(_ptr(qa), float(q_scale), n_rows, Hq, _ptr(row_seq), _ptr(row_pos),
                               ctypes.byref(kvs), _ptr(seqlens), _ptr(sinks_a), int(window), float(sm_scale),
                               _ptr(sel_rows), _ptr(sel_heads), n_sel, _ptr(out), _ptr(lse))
    elif key_range is not None:
        rc = lib.sao_attend_range(_ptr(qa), n_rows, Hq, _ptr(row_seq), _ptr(row_pos), ctypes.byref(kvs),
                                  _ptr(seqlens), _ptr(sinks_a), int(window), float(sm_scale),
                                  _ptr(sel_rows), _ptr(sel_heads), n_sel, int(key_range[0]),
                                  int(key_range[1]), _ptr(out), _ptr(lse))
    elif split is None:
        rc = lib.sao_attend(_ptr(qa), n_rows, Hq, _ptr(row_seq), _ptr(row_pos), ctypes.byref(kvs),
                            _ptr(seqlens), _ptr(sinks_a), int(window), float(sm_scale),
                            _ptr(sel_rows), _ptr(sel_heads), n_sel, _ptr(out), _ptr(lse))
    else:
        nc, chunk = split
        po = np.zeros((nc, n_sel, D), np.float64)
        pl = np.zeros((nc, n_sel), np.float64)
        rc = lib.sao_attend_split(_ptr(qa), n_rows, Hq, _ptr(row_seq), _ptr(row_pos), ctypes.byref(kvs),
                                  _ptr(seqlens), _ptr(sinks_a), int(window), float(sm_scale),
                                  _ptr(sel_rows), _ptr(sel_heads), n_sel, int(nc), int(chunk),
                                  _ptr(po), _ptr(pl), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle: page table points outside the page pool (rc=%d)" % rc)
    return out, lse


def merge(o_part, lse_part, sinks=None):
    """Merge partial states: o_part [S, N, H, D], lse_part [S, N, H] -> out [N, H, D], lse [N, H]."""
    lib = _load()
    o = _np(o_part, np.float64)
    l = _np(lse_part, np.float64)
    S, N, H, D = o.shape
    sk = None if sinks is None else _np(sinks, np.float32)
    out = np.zeros((N, H, D), np.float64)
    lse = np.zeros((N, H), np.float64)
    lib.sao_merge(_ptr(o), _ptr(l), S, N, H, D, _ptr(sk), _ptr(out), _ptr(lse))
    return out, lse


def bf16_to_f64(bits) -> np.ndarray:
    b = _np(bits).view(np.uint16).reshape(-1)
    out = np.zeros(b.shape[0], np.float64)
    _load().sao_bf16_array(_ptr(b), b.shape[0], _ptr(out))
    return out


def e4m3_to_f64(codes) -> np.ndarray:
    c = _np(codes).view(np.uint8).reshape(-1)
    out = np.zeros(c.shape[0], np.float64)
    _load().sao_e4m3_array(_ptr(c), c.shape[0], _ptr(out))
    return out
