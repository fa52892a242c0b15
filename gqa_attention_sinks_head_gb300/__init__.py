"""Python binding of libsinkattn: GQA attention with per-head attention sinks
on GB300 (sm_103a).

The functions carry the C ABI's names (include/sink_attn.h) and only marshal
arguments: torch CUDA tensors go in as raw device pointers, the current torch
stream is passed as the CUDA stream, and a nonzero status raises SinkAttnError
with the library's message.  Every step of the computation runs in the CUDA
kernels of libsinkattn.so; there is no fallback.  If the library is missing
the calls raise.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "SinkAttnError", "KVDesc", "load", "build", "sa_decode", "sa_decode_partial", "sa_merge_states",
    "sa_prefill", "sa_decode_static_workspace", "sa_decode_num_splits", "sa_decode_workspace_size", "sa_device_status", "sa_version",
    "sa_decode_multi", "sa_decode_multi_workspace_size", "sa_decode_multi_num_splits", "SA_MAX_DECODE_TOKENS",
    "sa_rope_yarn_table",
    "sa_rope_append", "sa_prefill_q8", "sa_selftest_wait_timeout",
    "SA_KV_BF16", "SA_KV_FP8_E4M3", "kv_desc",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libsinkattn.so")

SA_OK, SA_ERR_INVALID_ARG, SA_ERR_UNSUPPORTED, SA_ERR_WORKSPACE, SA_ERR_CUDA, SA_ERR_TIMEOUT = range(6)
SA_KV_BF16, SA_KV_FP8_E4M3 = 0, 1
SA_DEVICE_SEQLEN_RANGE, SA_DEVICE_BAD_PAGE, SA_DEVICE_TIMEOUT, SA_DEVICE_BAD_QLEN = 1, 2, 4, 8

EXPORTS = ["sa_decode", "sa_decode_num_splits", "sa_decode_workspace_size", "sa_decode_partial",
           "sa_merge_states", "sa_prefill", "sa_device_status", "sa_status_string", "sa_last_error",
           "sa_version", "sa_decode_static_workspace", "sa_decode_multi", "sa_decode_multi_workspace_size",
           "sa_decode_multi_num_splits", "sa_rope_yarn_table", "sa_rope_append", "sa_prefill_q8",
           "sa_selftest_wait_timeout"]
SA_MAX_DECODE_TOKENS = 8
SA_STATIC_WORKSPACE_BYTES = 16 << 20


class SinkAttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (_STATUS_NAMES.get(status, status), message))
        self.status = status


_STATUS_NAMES = {0: "SA_OK", 1: "SA_ERR_INVALID_ARG", 2: "SA_ERR_UNSUPPORTED", 3: "SA_ERR_WORKSPACE",
                 4: "SA_ERR_CUDA", 5: "SA_ERR_TIMEOUT"}


class KVDesc(ctypes.Structure):
    """sa_kv_desc_t."""
    _fields_ = [
        ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("dtype", ctypes.c_int32),
        ("num_pages", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32), ("page_table_stride", ctypes.c_int32),
        ("stride_page", ctypes.c_int64), ("stride_head", ctypes.c_int64), ("stride_token", ctypes.c_int64),
        ("page_table", ctypes.c_void_p), ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float),
    ]


_lib = None


def build(force: bool = False) -> str:
    from . import _build
    return _build.build(force=force)


def load(path: str | None = None):
    """Load libsinkattn.so (built in-tree by build()); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError("libsinkattn.so is not built (%s): call gqa_attention_sinks_head_gb300.build()" % path)
    lib = ctypes.CDLL(path)
    P, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    KP = ctypes.POINTER(KVDesc)
    lib.sa_decode.argtypes = [P, KP, P, i32, i32, i32, P, i32, f32, P, P, P, sz, i32, P]
    lib.sa_decode_static_workspace.argtypes = [P, KP, P, i32, i32, i32, P, i32, f32, P, P, i32, P]
    lib.sa_decode_multi.argtypes = [P, i32, KP, P, i32, i32, i32, P, i32, f32, P, P, P, sz, i32, P]
    lib.sa_decode_multi_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32]
    lib.sa_decode_multi_workspace_size.restype = sz
    lib.sa_decode_multi_num_splits.argtypes = [i32, i32, i32, i32, i32, i32]
    lib.sa_decode_multi_num_splits.restype = i32
    dbl = ctypes.c_double
    lib.sa_rope_yarn_table.argtypes = [P, i32, i32, dbl, dbl, i32, dbl, dbl]
    lib.sa_rope_append.argtypes = [P, P, P, i32, i32, P, P, P, i32, KP, i32, P, f32, P]
    lib.sa_prefill_q8.argtypes = [P, f32, P, i32, KP, P, i32, i32, i32, i32, P, i32, f32, P, P, P]
    lib.sa_selftest_wait_timeout.argtypes = [P]
    lib.sa_decode_partial.argtypes = [P, KP, P, i32, i32, i32, i32, f32, i32, P, P, P]
    lib.sa_merge_states.argtypes = [P, P, i32, i32, i32, i32, P, P, P, P]
    lib.sa_prefill.argtypes = [P, P, i32, KP, P, i32, i32, i32, i32, P, i32, f32, P, P, P]
    lib.sa_decode_num_splits.argtypes = [i32, i32, i32, i32]
    lib.sa_decode_num_splits.restype = i32
    lib.sa_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    lib.sa_decode_workspace_size.restype = sz
    lib.sa_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
    lib.sa_status_string.argtypes = [ctypes.c_int]
    lib.sa_status_string.restype = ctypes.c_char_p
    lib.sa_last_error.restype = ctypes.c_char_p
    lib.sa_version.restype = ctypes.c_int
    for fn in ("sa_decode", "sa_decode_static_workspace", "sa_decode_partial", "sa_merge_states", "sa_prefill",
               "sa_device_status", "sa_decode_multi", "sa_rope_yarn_table", "sa_rope_append", "sa_prefill_q8",
               "sa_selftest_wait_timeout"):
        getattr(lib, fn).restype = ctypes.c_int
    _lib = lib
    return lib


def _check(status: int):
    if status != SA_OK:
        raise SinkAttnError(status, _lib.sa_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def kv_desc(kv) -> tuple[KVDesc, list]:
    """sa_kv_desc_t for a workloads.KVCache-like object (or its as_dict())."""
    d = kv.as_dict() if hasattr(kv, "as_dict") else kv
    s = KVDesc()
    s.k = d["k"].data_ptr()
    s.v = d["v"].data_ptr()
    s.dtype = SA_KV_BF16 if d["dtype"] == "bf16" else SA_KV_FP8_E4M3
    s.num_pages = int(d["num_pages"])
    s.num_kv_heads = int(d["num_kv_heads"])
    s.head_dim = int(d["head_dim"])
    s.page_size = int(d["page_size"])
    s.page_table_stride = int(d.get("page_table_stride") or 0)
    s.stride_page = int(d["stride_page"])
    s.stride_head = int(d["stride_head"])
    s.stride_token = int(d["stride_token"])
    pt = d.get("page_table")
    s.page_table = None if pt is None else pt.data_ptr()
    s.k_scale = float(d.get("k_scale", 1.0))
    s.v_scale = float(d.get("v_scale", 1.0))
    return s, [d["k"], d["v"], pt]


def sa_version() -> int:
    return int(load().sa_version())


def sa_decode_num_splits(batch, num_kv_heads, max_kv_len, window) -> int:
    return int(load().sa_decode_num_splits(batch, num_kv_heads, max_kv_len, window))


def sa_decode_workspace_size(batch, num_qo_heads, num_kv_heads, head_dim, max_kv_len, window, num_splits=0) -> int:
    return int(load().sa_decode_workspace_size(batch, num_qo_heads, num_kv_heads, head_dim, max_kv_len, window,
                                               num_splits))


def sa_decode(q, kv, seqlens, sinks, window, sm_scale, out, lse=None, *, max_kv_len, workspace=None,
              num_splits=0, stream=None):
    """sa_decode on torch CUDA tensors; writes `out` (and `lse`) in place."""
    lib = load()
    desc, keep = kv_desc(kv)
    B, Hq, _ = q.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.sa_decode(_ptr(q), ctypes.byref(desc), _ptr(seqlens), B, Hq, int(max_kv_len), _ptr(sinks),
                         int(window), float(sm_scale), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
                         int(num_splits), _stream(stream)))
    return out, lse


def sa_decode_multi(q, q_len, kv, seqlens, sinks, window, sm_scale, out, lse=None, *, max_kv_len, workspace=None,
                    num_splits=0, stream=None):
    """sa_decode_multi on torch CUDA tensors: q, out [batch * q_len, Hq, 64],
    token k of sequence b in row b * q_len + k; writes `out` (and `lse`)."""
    lib = load()
    desc, keep = kv_desc(kv)
    R, Hq, _ = q.shape
    B = seqlens.shape[0]
    if R != B * int(q_len):
        raise ValueError("q has %d rows, expected batch * q_len = %d" % (R, B * int(q_len)))
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.sa_decode_multi(_ptr(q), int(q_len), ctypes.byref(desc), _ptr(seqlens), B, Hq, int(max_kv_len),
                               _ptr(sinks), int(window), float(sm_scale), _ptr(out), _ptr(lse), _ptr(workspace),
                               ws_bytes, int(num_splits), _stream(stream)))
    return out, lse


def sa_decode_multi_num_splits(batch, q_len, num_kv_heads, max_kv_len, window, kv_dtype="bf16") -> int:
    """Chunk count of sa_decode_multi with num_splits = 0 (kv_dtype: "bf16" or "e4m3")."""
    code = SA_KV_BF16 if kv_dtype == "bf16" else SA_KV_FP8_E4M3
    return int(load().sa_decode_multi_num_splits(int(batch), int(q_len), int(num_kv_heads), int(max_kv_len),
                                                 int(window), code))


def sa_decode_multi_workspace_size(batch, q_len, num_qo_heads, num_kv_heads, head_dim, max_kv_len, window,
                                   num_splits=0):
    return int(load().sa_decode_multi_workspace_size(int(batch), int(q_len), int(num_qo_heads), int(num_kv_heads),
                                                     int(head_dim), int(max_kv_len), int(window), int(num_splits)))


def sa_rope_yarn_table(max_position, *, theta, factor, original_max_position, beta_fast, beta_slow, head_dim=64):
    """The rotary table of sa_rope_append as a CPU float32 tensor [max_position, 64]
    (fill on the host; move it to the device yourself)."""
    import torch
    t = torch.empty(int(max_position), int(head_dim), dtype=torch.float32)
    _check(load().sa_rope_yarn_table(ctypes.c_void_p(t.data_ptr()), int(max_position), int(head_dim),
                                     float(theta), float(factor), int(original_max_position), float(beta_fast),
                                     float(beta_slow)))
    return t


def sa_rope_append(q, k, v, seq_ids, positions, table, kv, batch, q_out, q_out_scale=0.0, stream=None):
    """sa_rope_append on torch CUDA tensors: writes q_out (bf16, or E4M3 codes
    of q / q_out_scale when q_out_scale > 0) and the cache of kv."""
    lib = load()
    desc, keep = kv_desc(kv)
    T, Hq, _ = q.shape
    _check(lib.sa_rope_append(_ptr(q), _ptr(k), _ptr(v), T, Hq, _ptr(seq_ids), _ptr(positions), _ptr(table),
                              int(table.shape[0]), ctypes.byref(desc), int(batch), _ptr(q_out), float(q_out_scale),
                              _stream(stream)))
    return q_out


def sa_decode_static_workspace(q, kv, seqlens, sinks, window, sm_scale, out, lse=None, *, max_kv_len,
                               num_splits=0, stream=None):
    """sa_decode with the split scratch in the library's own static device
    array (for callers that cannot allocate); see include/sink_attn.h."""
    lib = load()
    desc, keep = kv_desc(kv)
    B, Hq, _ = q.shape
    _check(lib.sa_decode_static_workspace(_ptr(q), ctypes.byref(desc), _ptr(seqlens), B, Hq, int(max_kv_len),
                                          _ptr(sinks), int(window), float(sm_scale), _ptr(out), _ptr(lse),
                                          int(num_splits), _stream(stream)))
    return out, lse


def sa_decode_partial(q, kv, seqlens, window, sm_scale, num_splits, o_part, lse_part, *, max_kv_len, stream=None):
    lib = load()
    desc, keep = kv_desc(kv)
    B, Hq, _ = q.shape
    _check(lib.sa_decode_partial(_ptr(q), ctypes.byref(desc), _ptr(seqlens), B, Hq, int(max_kv_len), int(window),
                                 float(sm_scale), int(num_splits), _ptr(o_part), _ptr(lse_part), _stream(stream)))
    return o_part, lse_part


def sa_merge_states(o_part, lse_part, sinks, out, lse_out=None, stream=None):
    lib = load()
    S, N, H, D = o_part.shape
    _check(lib.sa_merge_states(_ptr(o_part), _ptr(lse_part), S, N, H, D, _ptr(sinks), _ptr(out), _ptr(lse_out),
                               _stream(stream)))
    return out, lse_out


def sa_prefill(q, cu_seqlens_q, kv, seqlens_kv, sinks, window, sm_scale, out, lse=None, *, max_q_len, max_kv_len,
               stream=None):
    lib = load()
    desc, keep = kv_desc(kv)
    B = int(seqlens_kv.shape[0])
    Hq = int(q.shape[1])
    _check(lib.sa_prefill(_ptr(q), _ptr(cu_seqlens_q), int(q.shape[0]), ctypes.byref(desc), _ptr(seqlens_kv), B,
                          Hq, int(max_q_len),
                          int(max_kv_len), _ptr(sinks), int(window), float(sm_scale), _ptr(out), _ptr(lse),
                          _stream(stream)))
    return out, lse


def sa_prefill_q8(q_codes, q_scale, cu_seqlens_q, kv, seqlens_kv, sinks, window, sm_scale, out, lse=None, *,
                  max_q_len, max_kv_len, stream=None):
    """sa_prefill with E4M3 query codes (uint8 [total_q, Hq, 64], value = code * q_scale)."""
    lib = load()
    desc, keep = kv_desc(kv)
    B = int(seqlens_kv.shape[0])
    Hq = int(q_codes.shape[1])
    _check(lib.sa_prefill_q8(_ptr(q_codes), float(q_scale), _ptr(cu_seqlens_q), int(q_codes.shape[0]),
                             ctypes.byref(desc), _ptr(seqlens_kv), B, Hq, int(max_q_len), int(max_kv_len),
                             _ptr(sinks), int(window), float(sm_scale), _ptr(out), _ptr(lse), _stream(stream)))
    return out, lse


def sa_selftest_wait_timeout(stream=None):
    """Queue the bounded-wait self-test (about 1 s on the device); read the
    result with sa_device_status()."""
    _check(load().sa_selftest_wait_timeout(_stream(stream)))


def sa_device_status(stream=None) -> int:
    lib = load()
    v = ctypes.c_uint32(0)
    _check(lib.sa_device_status(_stream(stream), ctypes.byref(v)))
    return int(v.value)
