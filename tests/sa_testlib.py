"""Shared helpers of the GPU parity tests: run the library, run the oracle on
the same bytes, compare with the tolerance of the contract.

Tolerance (bf16 outputs, fp32 lse): |out - ref| <= 1e-2 + 1e-2 * |ref|
elementwise, |lse - ref| <= 1e-3; no NaN anywhere; -inf lse only where the
reference is -inf.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import workloads as W

OUT_ATOL = 1e-2
OUT_RTOL = 1e-2
LSE_ATOL = 1e-3


def check_close(out, lse, ref_out, ref_lse, what=""):
    o = out.detach().float().cpu().double().numpy()
    r = np.asarray(ref_out, np.float64).reshape(o.shape)
    assert not np.isnan(o).any(), "%s: NaN in output (%d)" % (what, int(np.isnan(o).sum()))
    err = np.abs(o - r)
    bound = OUT_ATOL + OUT_RTOL * np.abs(r)
    bad = err > bound
    assert not bad.any(), "%s: %d/%d outputs out of tolerance, worst err %.3g at %s (ref %.4g)" % (
        what, int(bad.sum()), bad.size, float(err.max()), np.unravel_index(int(np.argmax(err - bound)), o.shape),
        float(r.reshape(-1)[int(np.argmax((err - bound).reshape(-1)))]))
    if lse is not None:
        l = lse.detach().cpu().double().numpy().reshape(-1)
        rl = np.asarray(ref_lse, np.float64).reshape(-1)
        assert not np.isnan(l).any(), "%s: NaN in lse" % what
        inf_r = np.isneginf(rl)
        assert (np.isneginf(l) == inf_r).all(), "%s: -inf lse mismatch" % what
        d = np.abs(l[~inf_r] - rl[~inf_r])
        assert d.size == 0 or d.max() <= LSE_ATOL, "%s: lse err %.3g" % (what, float(d.max()))


def decode_gpu(sa, case_gpu, num_splits=0, with_lse=True, max_kv_len=None):
    B, Hq, D = case_gpu.q.shape
    if max_kv_len is None:
        max_kv_len = int(case_gpu.seqlens.max().item()) if B > 0 else 0
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda") if with_lse else None
    kv = case_gpu.kv
    ws_bytes = sa.sa_decode_workspace_size(B, Hq, kv.num_kv_heads, D, max_kv_len, case_gpu.window, num_splits)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    sa.sa_decode(case_gpu.q, kv, case_gpu.seqlens, case_gpu.sinks, case_gpu.window, case_gpu.sm_scale, out, lse,
                 max_kv_len=max_kv_len, workspace=ws, num_splits=num_splits)
    torch.cuda.synchronize()
    return out, lse


def oracle_decode(oracle, case_cpu, sel_rows=None):
    """Reference for decode rows (all, or the selected sequences' rows)."""
    rows = oracle.decode_rows(case_cpu.seqlens)
    B, Hq, D = case_cpu.q.shape
    if sel_rows is None:
        out, lse = oracle.attend(case_cpu.q, rows[0], rows[1], case_cpu.kv.as_dict(), case_cpu.seqlens,
                                 case_cpu.sinks, case_cpu.window, case_cpu.sm_scale)
        return out.reshape(B, Hq, D), lse.reshape(B, Hq)
    sr = np.repeat(np.asarray(sel_rows, np.int32), Hq)
    sh = np.tile(np.arange(Hq, dtype=np.int32), len(sel_rows))
    out, lse = oracle.attend(case_cpu.q, rows[0], rows[1], case_cpu.kv.as_dict(), case_cpu.seqlens,
                             case_cpu.sinks, case_cpu.window, case_cpu.sm_scale, sr, sh)
    return out.reshape(len(sel_rows), Hq, D), lse.reshape(len(sel_rows), Hq)


def compact_decode_case(case, seq_ids) -> W.Case:
    return W.subset(case, seq_ids)


def prefill_gpu(sa, case_gpu, with_lse=True):
    T, Hq, D = case_gpu.q.shape
    out = torch.full((T, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((T, Hq), float("nan"), dtype=torch.float32, device="cuda") if with_lse else None
    cu = case_gpu.cu_seqlens_q
    qlens = (cu[1:] - cu[:-1]).cpu()
    sa.sa_prefill(case_gpu.q, cu, case_gpu.kv, case_gpu.seqlens, case_gpu.sinks, case_gpu.window,
                  case_gpu.sm_scale, out, lse, max_q_len=int(qlens.max()) if len(qlens) else 0,
                  max_kv_len=int(case_gpu.seqlens.max()) if len(qlens) else 0)
    torch.cuda.synchronize()
    return out, lse


def oracle_prefill(oracle, case_cpu, sel_rows=None):
    rows = oracle.prefill_rows(case_cpu.cu_seqlens_q, case_cpu.seqlens)
    T, Hq, D = case_cpu.q.shape
    if sel_rows is None:
        sel_rows = np.arange(T, dtype=np.int32)
    sel_rows = np.asarray(sel_rows, np.int32)
    sr = np.repeat(sel_rows, Hq)
    sh = np.tile(np.arange(Hq, dtype=np.int32), len(sel_rows))
    out, lse = oracle.attend(case_cpu.q, rows[0], rows[1], case_cpu.kv.as_dict(), case_cpu.seqlens,
                             case_cpu.sinks, case_cpu.window, case_cpu.sm_scale, sr, sh)
    return out.reshape(len(sel_rows), Hq, D), lse.reshape(len(sel_rows), Hq)
