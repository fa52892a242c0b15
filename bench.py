#!/usr/bin/env python3
"""Benchmark of the sink-attention hot path on GB300.

Default workload (N=1): decode of 64 sequences with KV lengths uniform in
[1024, 8192] over a paged bf16 cache (16-token pages, permuted table), 64 query
/ 8 kv heads, head_dim 64, sinks ~ U(-2, 6); one step = the full-context call
followed by the 128-token-window call on the same cache (the alternating
layers of gpt-oss).  Metric: algorithmic HBM bytes / time, in GB/s.
--config 1..5 selects the other workloads (3 = prefill, TFLOP/s).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference] [--config C]

Under torchrun (N > 1) every rank runs the same per-GPU workload on its own
GPU (independent replicas; weak scaling), the timed region is bracketed by a
barrier and a synchronize on both sides, and rank 0 prints the max over ranks.
`--impl reference` times the fp64 CPU oracle on a bounded sample of the same
workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sink-attn decode HBM GB/s (% peak); prefill TFLOP/s (% bf16 tensor peak)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
DEFAULT_STEPS = {1: 2000, 2: 2000, 3: 50, 4: 100, 5: 500, 6: 50, 7: 50, 8: 1000, 9: 2000, 10: 50}


# ------------------------------------------------------------------ helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def source_sha(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key, workload):
    """dram bytes per launch from the committed ncu summary, if it was taken on
    the current source of that kernel; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(kernel_key, {}).get(workload)
    if not e:
        return None
    if e.get("source_sha") != source_sha(e.get("sources", [])):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples around the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device_index):
        self.samples = []
        self.proc = None
        self.t0 = self.t1 = None
        ident = None
        try:
            import torch
            u = getattr(torch.cuda.get_device_properties(device_index), "uuid", None)
            if u is not None:
                ident = "GPU-" + str(u)
        except Exception:
            pass
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits", "-lms", "100"]
        if ident:
            cmd += ["-i", ident]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def begin(self):
        self.t0 = time.time()

    def end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.proc = None

    def summary(self, t0=None, t1=None):
        """Median SM clock, max clock and throttle reasons of the samples taken
        inside [t0, t1] (the timed region), or of all samples if none fell in it."""
        t0 = self.t0 if t0 is None else t0
        t1 = self.t1 if t1 is None else t1
        inside = [s for t, s in self.samples if t0 is not None and t0 - 0.15 <= t <= t1 + 0.15]
        rows = inside or [s for _, s in self.samples]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if len(r) > 1 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if len(r) > 2 and r[2].replace(".", "").isdigit()]
        reasons = set()
        for r in rows:
            for i, name in enumerate(self.NAMES):
                if len(r) > 5 + i and r[5 + i].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows), "in_timed_region": bool(inside)}


# ------------------------------------------------------------ distributed
def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend)
    return dist


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def dist_max(value: float, world: int) -> float:
    """Max of a host float over ranks (the slowest rank sets the job time)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


L2_FLUSH_BYTES = 256 << 20  # about twice the GB300's 129 MB L2


def timed_loop(torch, stream, one, steps, warmup, flush=None):
    """Median device time (ms) of one() over `steps` iterations after
    `warmup`, each bracketed by CUDA events on `stream`; flush() (if any) runs
    before each iteration, outside its events."""
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            one()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for e0, e1 in evs:
            if flush is not None:
                flush()
            e0.record(stream)
            one()
            e1.record(stream)
        torch.cuda.synchronize()
    return statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)


def timed_pipelined(torch, stream, ins, outs, calls, steps, warmup):
    """Device time (ms) per step of a loop that overlaps each step's host
    transfers with its neighbours' work, as a serving loop does: ins[b] /
    outs[b] (b = step % 2) are Packed input / result buffers, and calls(b)
    queues the step's library calls on `stream`, reading ins[b] and writing
    outs[b].  Step k's inputs go up on an upload stream once step k - 2 no
    longer reads that buffer; its results come back on a download stream once
    they are written, while step k + 1 computes.  Every step still moves all
    of its bytes.  Events on `stream` at the two ends of the K steps (the
    last download included) time them; the result is their mean."""
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    in_free = [torch.cuda.Event() for _ in range(2)]
    in_ready = [torch.cuda.Event() for _ in range(2)]
    out_ready = [torch.cuda.Event() for _ in range(2)]
    out_free = [torch.cuda.Event() for _ in range(2)]

    def run(n):
        for k in range(n):
            b = k % 2
            up.wait_event(in_free[b])
            with torch.cuda.stream(up):
                ins[b].h2d()
            in_ready[b].record(up)
            stream.wait_event(in_ready[b])
            stream.wait_event(out_free[b])
            calls(b)
            in_free[b].record(stream)
            out_ready[b].record(stream)
            down.wait_event(out_ready[b])
            with torch.cuda.stream(down):
                outs[b].d2h()
            out_free[b].record(down)

    with torch.cuda.stream(stream):
        for e in in_free + out_free:  # every wait below refers to a recorded event
            e.record(stream)
        run(warmup)
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        up.wait_event(t0)
        down.wait_event(t0)
        run(steps)
        stream.wait_event(out_free[(steps - 1) % 2])
        t1.record(stream)
        torch.cuda.synchronize()
    return t0.elapsed_time(t1) / steps


class Packed:
    """Tensors of one step laid out back to back (256-byte aligned) in one
    device buffer with a pinned host mirror, so that one copy moves them all:
    h2d() before the step's calls for its inputs, d2h() after them for its
    results.  `dev` / `host` are views shaped like the given tensors, which
    fill both sides at construction."""

    def __init__(self, torch, tensors):
        offs, end = [], 0
        for t in tensors:
            offs.append(end)
            end = (end + t.numel() * t.element_size() + 255) // 256 * 256
        self.nbytes = offs[-1] + tensors[-1].numel() * tensors[-1].element_size()  # bytes one copy moves
        self._dev = torch.empty(max(end, 256), dtype=torch.uint8, device="cuda")
        self._host = torch.empty(max(end, 256), dtype=torch.uint8, pin_memory=True)
        self.dev, self.host = [], []
        for t, o in zip(tensors, offs):
            n = t.numel() * t.element_size()
            dv = self._dev[o:o + n].view(t.dtype).view(t.shape)
            hv = self._host[o:o + n].view(t.dtype).view(t.shape)
            dv.copy_(t)
            hv.copy_(t.cpu())
            self.dev.append(dv)
            self.host.append(hv)

    def h2d(self):
        self._dev[:self.nbytes].copy_(self._host[:self.nbytes], non_blocking=True)

    def d2h(self):
        self._host[:self.nbytes].copy_(self._dev[:self.nbytes], non_blocking=True)


# --------------------------------------------------------------- workloads
def decode_bytes(seqlens, window, hkv, hq, dim, elem_bytes, with_lse=True):
    """Algorithmic HBM bytes of one decode call: every visible K and V element
    once per kv head, plus q in and out (bf16) and lse (fp32)."""
    keys = sum(min(int(L), window) if window > 0 else int(L) for L in seqlens)
    b = len(seqlens)
    return keys * hkv * dim * 2 * elem_bytes + 2 * b * hq * dim * 2 + (4 * b * hq if with_lse else 0)


def multi_bytes(seqlens, window, q_len, hkv, hq, dim, elem_bytes):
    """Algorithmic HBM bytes of one multi-token decode call: every key visible
    to any of a sequence's q_len tokens once per kv head, plus q, out, lse."""
    keys = sum(min(int(L), window + q_len - 1) if window > 0 else int(L) for L in seqlens)
    rows = len(seqlens) * q_len
    return keys * hkv * dim * 2 * elem_bytes + 2 * rows * hq * dim * 2 + 4 * rows * hq


def prefill_flops(q_lens, kv_lens, window, hq, dim):
    """4 * Hq * D * sum over queries of the visible keys (QK and PV)."""
    tot = 0
    for lq, lk in zip(q_lens, kv_lens):
        for i in range(lq):
            p = lk - lq + i
            n = p + 1 if window <= 0 else min(window, p + 1)
            tot += n
    return 4 * hq * dim * tot


def windows_of(cfg):
    return {1: [0], 2: [0, 128], 3: [0, 128], 4: [0], 5: [0, 128, 0, 128], 6: [0, 128], 7: [0, 128], 8: [0, 128], 9: [0], 10: [0, 128]}[cfg]


PREFILL_CONFIGS = (3, 6, 7, 10)
MULTI_CONFIGS = (8,)
ROPE_CONFIGS = (9,)


def workload_name(cfg):
    return {
        1: "decode B=1 L=256 contiguous bf16, 64q/8kv heads, D=64, w=0",
        2: "decode B=64 L~U[1024,8192] paged P=16 bf16, 64q/8kv heads, D=64, step = w=0 call + w=128 call",
        3: "prefill T=8192 causal contiguous bf16, 64q/8kv heads, D=64, step = w=0 call + w=128 call",
        4: "decode B=128 L=32768 paged P=16 bf16 split-KV, 64q/8kv heads, D=64, w=0",
        5: "decode B=256 L=8192 paged P=16 fp8-e4m3, 64q/8kv heads, D=64, step = w=0,128,0,128",
        6: "chunked prefill B=8, 1024 new queries each on a paged P=16 bf16 context L_kv~U[2048,16384], "
           "64q/8kv heads, D=64, step = w=0 call + w=128 call",
        7: "chunked prefill B=8, 1024 new queries each on a paged P=16 fp8-e4m3 context L_kv~U[2048,16384], "
           "64q/8kv heads, D=64, step = w=0 call + w=128 call",
        8: "multi-token decode B=64, 4 new tokens each, L~U[1024,8192] paged P=16 bf16, 64q/8kv heads, D=64, "
           "step = w=0 call + w=128 call",
        9: "YaRN RoPE of q/k + paged bf16 cache write for 8192 new tokens (one sequence), 64q/8kv heads, D=64",
        10: "workload 7 with E4M3 queries (sa_prefill_q8: FP8 tensor cores for Q K^T), step = w=0 call + "
            "w=128 call",
    }[cfg]


class DecodeBench:
    """One step = the decode calls of the workload on one resident cache.
    With sa=None (the reference arm) only the inputs are built: the same
    seeded bytes, drawn on the same device, and no library call is made."""

    def __init__(self, sa, cfg, device, batch=None):
        import torch
        import workloads as W
        self.sa, self.cfg, self.torch = sa, cfg, torch
        gen_dev = device if cfg in (2, 4, 5) else "cpu"
        self.case = W.make_config(cfg, window=0, device=gen_dev, batch=batch).to(device)
        if batch is not None:
            self.label = "%s; first %d sequences" % (workload_name(cfg), len(self.case.seqlens))
        self.sample_units = len(self.case.seqlens)
        c = self.case
        self.B, self.Hq, self.D = c.q.shape
        self.Hkv = c.kv.num_kv_heads
        self.maxlen = int(c.seqlens.max())
        self.seqlens = [int(x) for x in c.seqlens.cpu()]
        self.elem = 1 if c.kv.dtype == "e4m3" else 2
        self.calls = []
        for w in windows_of(cfg):
            if sa is None:
                self.calls.append(dict(window=w, S=1, bytes=decode_bytes(self.seqlens, w, self.Hkv, self.Hq, self.D,
                                                                         self.elem)))
                continue
            S = sa.sa_decode_num_splits(self.B, self.Hkv, self.maxlen, w)
            out = torch.empty(self.B, self.Hq, self.D, dtype=torch.bfloat16, device=device)
            lse = torch.empty(self.B, self.Hq, dtype=torch.float32, device=device)
            o_part = l_part = ws = None
            if S > 1:
                o_part = torch.empty(S, self.B, self.Hq, self.D, dtype=torch.float32, device=device)
                l_part = torch.empty(S, self.B, self.Hq, dtype=torch.float32, device=device)
                nbytes = sa.sa_decode_workspace_size(self.B, self.Hq, self.Hkv, self.D, self.maxlen, w, S)
                ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
            self.calls.append(dict(window=w, S=S, out=out, lse=lse, o_part=o_part, l_part=l_part, ws=ws,
                                   bytes=decode_bytes(self.seqlens, w, self.Hkv, self.Hq, self.D, self.elem)))
        self.step_bytes = sum(cl["bytes"] for cl in self.calls)
        self.kernels_per_step = sum(2 if cl["S"] > 1 else 1 for cl in self.calls)
        self.unit = "GB/s"
        self.dtype_name = "bf16" if self.elem == 2 else "fp8-e4m3 kv, bf16 q/out"
        self.e2e_api = ("sa_decode with pinned host q/seqlens/page table in, out/lse back; KV cache resident; "
                        "double-buffered (a step's copies overlap its neighbours' calls, steps back to back) "
                        "unless the step needs an L2 flush")

    def amount(self):
        return self.step_bytes / 1e9

    def resident_bytes(self):
        """Bytes of the step's inputs in HBM: the cache the largest call reads."""
        return max(cl["bytes"] for cl in self.calls)

    def run_call(self, cl, stream, ev=None):
        """Per call: [ev0] decode kernel [ev1] merge kernel.  For S > 1 this is
        sa_decode_partial + sa_merge_states, the two launches sa_decode makes."""
        sa, c = self.sa, self.case
        if ev is not None:
            ev[0].record(stream)
        if cl["S"] > 1:
            sa.sa_decode_partial(c.q, c.kv, c.seqlens, cl["window"], c.sm_scale, cl["S"], cl["o_part"],
                                 cl["l_part"], max_kv_len=self.maxlen, stream=stream)
            if ev is not None:
                ev[1].record(stream)
            sa.sa_merge_states(cl["o_part"], cl["l_part"], c.sinks, cl["out"], cl["lse"], stream=stream)
        else:
            sa.sa_decode(c.q, c.kv, c.seqlens, c.sinks, cl["window"], c.sm_scale, cl["out"], cl["lse"],
                         max_kv_len=self.maxlen, num_splits=1, stream=stream)
            if ev is not None:
                ev[1].record(stream)

    def step(self, stream, evs=None):
        for i, cl in enumerate(self.calls):
            self.run_call(cl, stream, None if evs is None else evs[i])

    def dominant(self):
        return 0, "decode_kernel", self.calls[0]["bytes"]

    def segment_names(self):
        names = []
        for cl in self.calls:
            if cl["S"] > 1:
                names += ["decode w=%d (%d chunks)" % (cl["window"], cl["S"]), "merge w=%d" % cl["window"]]
            else:
                names.append("decode w=%d" % cl["window"])
        return names

    def notes(self, seg_ms, peaks):
        """Calls too small to stream at HBM rate are reported in microseconds."""
        out, j = {}, 0
        for cl in self.calls:
            n = 2 if cl["S"] > 1 else 1
            ms = sum(seg_ms[j:j + n])
            j += n
            if cl["bytes"] < 64e6:
                out["decode w=%d" % cl["window"]] = {
                    "us": round(ms * 1e3, 2), "GB/s": round(cl["bytes"] / 1e6 / ms, 1),
                    "bound": "latency (one wave of short blocks; launch and one HBM round trip dominate)"}
        return out

    def segments(self, stream):
        """The step as launch segments: decode kernel, then its merge when split."""
        sa, c = self.sa, self.case
        segs = []
        for cl in self.calls:
            if cl["S"] > 1:
                segs.append(lambda cl=cl: sa.sa_decode_partial(c.q, c.kv, c.seqlens, cl["window"], c.sm_scale, cl["S"],
                                                               cl["o_part"], cl["l_part"], max_kv_len=self.maxlen,
                                                               stream=stream))
                segs.append(lambda cl=cl: sa.sa_merge_states(cl["o_part"], cl["l_part"], c.sinks, cl["out"],
                                                             cl["lse"], stream=stream))
            else:
                segs.append(lambda cl=cl: sa.sa_decode(c.q, c.kv, c.seqlens, c.sinks, cl["window"], c.sm_scale,
                                                       cl["out"], cl["lse"], max_kv_len=self.maxlen, num_splits=1,
                                                       stream=stream))
        return segs

    # ---- end to end through sa_decode with host buffers
    def e2e(self, stream, steps, warmup, flush=None):
        """Per step: one copy of q, the sequence lengths and the page table in,
        the calls, one copy of every call's out and lse back.  Double-buffered
        (timed_pipelined) unless the step needs an L2 flush: then one step at
        a time, its copies and calls in order on one stream."""
        import dataclasses
        torch = self.torch
        c = self.case
        paged = c.kv.page_table is not None
        nbuf = 1 if flush is not None else 2
        ins = [Packed(torch, [c.q, c.seqlens] + ([c.kv.page_table] if paged else [])) for _ in range(nbuf)]
        outs = [Packed(torch, [t for cl in self.calls for t in (cl["out"], cl["lse"])]) for _ in range(nbuf)]
        kvs = [dataclasses.replace(c.kv, page_table=inp.dev[2]) if paged else c.kv for inp in ins]

        def calls(b):
            for i, cl in enumerate(self.calls):
                self.sa.sa_decode(ins[b].dev[0], kvs[b], ins[b].dev[1], c.sinks, cl["window"], c.sm_scale,
                                  outs[b].dev[2 * i], outs[b].dev[2 * i + 1], max_kv_len=self.maxlen,
                                  workspace=cl["ws"], num_splits=cl["S"], stream=stream)

        if flush is None:
            ms = timed_pipelined(torch, stream, ins, outs, calls, steps, warmup)
        else:
            def one():
                ins[0].h2d()
                calls(0)
                outs[0].d2h()

            ms = timed_loop(torch, stream, one, steps, warmup, flush)
        return ms, ins[0].nbytes, outs[0].nbytes

    # ---- oracle on a bounded sample
    def oracle_sample(self, budget_s, max_seqs=None):
        """(seconds per sample, bytes of the sample, description)."""
        import oracle
        import workloads as W
        oracle.build()
        c = self.case
        n = self.B if max_seqs is None else max(1, min(self.B, max_seqs))
        ids = list(range(n))
        sub = W.subset(c, ids)
        rows = oracle.decode_rows(sub.seqlens)
        t0 = time.time()
        nbytes = 0
        for cl in self.calls:
            oracle.attend(sub.q, rows[0], rows[1], sub.kv.as_dict(), sub.seqlens, sub.sinks, cl["window"],
                          sub.sm_scale)
            nbytes += decode_bytes([int(x) for x in sub.seqlens], cl["window"], self.Hkv, self.Hq, self.D,
                                   self.elem)
        dt = time.time() - t0
        desc = "%d of %d sequences x %d heads, every call of the step (windows %s)" % (
            n, self.B, self.Hq, [cl["window"] for cl in self.calls])
        return dt, nbytes, desc


class MultiDecodeBench:
    """One step = the multi-token decode calls of the workload (w=0, w=128) on
    one resident cache; each call is one sa_decode_multi (decode kernel, plus
    the merge kernel when split), timed as a whole."""

    def __init__(self, sa, cfg, device):
        import torch
        import workloads as W
        self.sa, self.cfg, self.torch = sa, cfg, torch
        self.case = W.make_config(cfg, window=0, device=device)
        c = self.case
        self.R, self.Hq, self.D = c.q.shape
        self.Hkv = c.kv.num_kv_heads
        self.seqlens = [int(x) for x in c.seqlens.cpu()]
        self.B = len(self.seqlens)
        self.sample_units = self.B
        self.q_len = self.R // self.B
        self.maxlen = max(self.seqlens)
        self.elem = 1 if c.kv.dtype == "e4m3" else 2
        self.calls = []
        for w in windows_of(cfg):
            if sa is None:  # the reference arm: inputs only
                self.calls.append(dict(window=w, S=1, bytes=multi_bytes(self.seqlens, w, self.q_len, self.Hkv,
                                                                        self.Hq, self.D, self.elem)))
                continue
            S = sa.sa_decode_multi_num_splits(self.B, self.q_len, self.Hkv, self.maxlen, w, c.kv.dtype)
            nbytes = sa.sa_decode_multi_workspace_size(self.B, self.q_len, self.Hq, self.Hkv, self.D, self.maxlen,
                                                       w, S)
            self.calls.append(dict(
                window=w, S=S, ws=torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device),
                out=torch.empty(self.R, self.Hq, self.D, dtype=torch.bfloat16, device=device),
                lse=torch.empty(self.R, self.Hq, dtype=torch.float32, device=device),
                bytes=multi_bytes(self.seqlens, w, self.q_len, self.Hkv, self.Hq, self.D, self.elem)))
        self.step_bytes = sum(cl["bytes"] for cl in self.calls)
        self.kernels_per_step = sum(2 if cl["S"] > 1 else 1 for cl in self.calls)
        self.unit = "GB/s"
        self.dtype_name = "bf16" if self.elem == 2 else "fp8-e4m3 kv, bf16 q/out"
        self.e2e_api = ("sa_decode_multi with pinned host q/seqlens/page table in, out/lse back; "
                        "KV cache resident; double-buffered (a step's copies overlap its neighbours' calls, "
                        "steps back to back)")

    def amount(self):
        return self.step_bytes / 1e9

    def resident_bytes(self):
        return max(cl["bytes"] for cl in self.calls)

    def run_call(self, cl, stream, ev=None):
        c = self.case
        if ev is not None:
            ev[0].record(stream)
        self.sa.sa_decode_multi(c.q, self.q_len, c.kv, c.seqlens, c.sinks, cl["window"], c.sm_scale, cl["out"],
                                cl["lse"], max_kv_len=self.maxlen, workspace=cl["ws"], num_splits=cl["S"],
                                stream=stream)
        if ev is not None:
            ev[1].record(stream)

    def step(self, stream, evs=None):
        for i, cl in enumerate(self.calls):
            self.run_call(cl, stream, None if evs is None else evs[i])

    def dominant(self):
        # q_len >= 2 on a bf16 cache runs the tcgen05 kernel (an FP8 cache the
        # one-token kernel's multi-token build); a split call adds the merge
        name = "decode_mt_kernel" if self.elem == 2 and self.q_len > 1 else "decode_kernel"
        return 0, name + (" (with its merge)" if self.calls[0]["S"] > 1 else ""), self.calls[0]["bytes"]

    def segment_names(self):
        return ["decode q_len=%d w=%d (%d chunks)" % (self.q_len, cl["window"], cl["S"]) for cl in self.calls]

    def notes(self, seg_ms, peaks):
        return {"decode q_len=%d w=%d" % (self.q_len, cl["window"]): {
                    "us": round(ms * 1e3, 2), "GB/s": round(cl["bytes"] / 1e6 / ms, 1),
                    "bound": "latency (one wave of short blocks)"}
                for cl, ms in zip(self.calls, seg_ms) if cl["bytes"] < 64e6}

    def segments(self, stream):
        """The step as launch segments: one per call."""
        return [lambda cl=cl: self.run_call(cl, stream) for cl in self.calls]

    def e2e(self, stream, steps, warmup, flush=None):
        """Per step: one copy of q, the sequence lengths and the page table in,
        the calls, one copy of every call's out and lse back."""
        import dataclasses
        torch = self.torch
        c = self.case
        nbuf = 1 if flush is not None else 2
        ins = [Packed(torch, [c.q, c.seqlens, c.kv.page_table]) for _ in range(nbuf)]
        outs = [Packed(torch, [t for cl in self.calls for t in (cl["out"], cl["lse"])]) for _ in range(nbuf)]
        kvs = [dataclasses.replace(c.kv, page_table=inp.dev[2]) for inp in ins]

        def calls(b):
            for i, cl in enumerate(self.calls):
                self.sa.sa_decode_multi(ins[b].dev[0], self.q_len, kvs[b], ins[b].dev[1], c.sinks, cl["window"],
                                        c.sm_scale, outs[b].dev[2 * i], outs[b].dev[2 * i + 1],
                                        max_kv_len=self.maxlen, workspace=cl["ws"], num_splits=cl["S"],
                                        stream=stream)

        if flush is None:
            ms = timed_pipelined(torch, stream, ins, outs, calls, steps, warmup)
        else:
            def one():
                ins[0].h2d()
                calls(0)
                outs[0].d2h()

            ms = timed_loop(torch, stream, one, steps, warmup, flush)
        return ms, ins[0].nbytes, outs[0].nbytes

    def oracle_sample(self, budget_s, max_seqs=None):
        """Every token row of the first n sequences, all heads, every call."""
        import numpy as np
        import oracle
        oracle.build()
        c = self.case
        cpu = c.to("cpu")
        n = self.B if max_seqs is None else max(1, min(self.B, max_seqs))
        rows = oracle.prefill_rows(cpu.cu_seqlens_q, cpu.seqlens)
        sel = np.arange(n * self.q_len, dtype=np.int32)
        sr = np.repeat(sel, self.Hq)
        sh = np.tile(np.arange(self.Hq, dtype=np.int32), len(sel))
        t0 = time.time()
        nbytes = 0
        for cl in self.calls:
            oracle.attend(cpu.q, rows[0], rows[1], cpu.kv.as_dict(), cpu.seqlens, cpu.sinks, cl["window"],
                          cpu.sm_scale, sr, sh)
            nbytes += multi_bytes(self.seqlens[:n], cl["window"], self.q_len, self.Hkv, self.Hq, self.D, self.elem)
        dt = time.time() - t0
        return dt, nbytes, "%d of %d sequences x %d tokens x %d heads, every call of the step" % (
            n, self.B, self.q_len, self.Hq)


class RopeBench:
    """One step = one sa_rope_append over 8192 new tokens of one sequence
    (q/k/v of a prefill chunk) into a paged bf16 cache."""

    T = 8192

    def __init__(self, sa, cfg, device):
        import torch
        import workloads as W
        self.sa, self.cfg, self.torch = sa, cfg, torch
        g = torch.Generator(device="cpu").manual_seed(1009)
        self.Hq, self.Hkv, self.D = 64, 8, 64
        T = self.T
        self.kv = W.make_kv([T], self.Hkv, self.D, 16, paged=True, poison_pages=64, seed=1009, device=device,
                            layout="HND")
        self.q = torch.randn(T, self.Hq, self.D, generator=g).to(torch.bfloat16).to(device)
        self.k = torch.randn(T, self.Hkv, self.D, generator=g).to(torch.bfloat16).to(device)
        self.v = torch.randn(T, self.Hkv, self.D, generator=g).to(torch.bfloat16).to(device)
        self.seq = torch.zeros(T, dtype=torch.int32, device=device)
        self.pos = torch.arange(T, dtype=torch.int32, device=device)
        self.yarn = dict(theta=150000.0, factor=32.0, original_max_position=4096, beta_fast=32.0, beta_slow=1.0)
        self.table = sa.sa_rope_yarn_table(T, **self.yarn).to(device)
        self.q_out = torch.empty_like(self.q)
        self.calls = [dict(window=0, S=1)]
        # read q, k, v, positions, sequence ids and the table rows; write q_out and the cache rows
        self.step_bytes = (2 * T * (self.Hq + 2 * self.Hkv) * self.D * 2 + 8 * T + T * self.D * 4)
        self.calls[0]["bytes"] = self.step_bytes
        self.kernels_per_step = 1
        self.unit = "GB/s"
        self.elem = 2
        self.B = 1
        self.sample_units = T // 32
        self.maxlen = T
        self.dtype_name = "bf16 (fp32 rotation)"
        self.e2e_api = "sa_rope_append with pinned host q/k/v/positions in, rotated q back; cache resident"
        self.oracle_cores = 1  # the rotary oracle is single-threaded numpy

    def amount(self):
        return self.step_bytes / 1e9

    def resident_bytes(self):
        return sum(t.numel() * t.element_size() for t in (self.q, self.k, self.v))

    def run_call(self, cl, stream, ev=None):
        if ev is not None:
            ev[0].record(stream)
        self.sa.sa_rope_append(self.q, self.k, self.v, self.seq, self.pos, self.table, self.kv, 1, self.q_out,
                               stream=stream)
        if ev is not None:
            ev[1].record(stream)

    def step(self, stream, evs=None):
        self.run_call(self.calls[0], stream, None if evs is None else evs[0])

    def dominant(self):
        return 0, "rope_append_kernel", self.step_bytes

    def segment_names(self):
        return ["rope_append"]

    def segments(self, stream):
        """The step as launch segments: one per call."""
        return [lambda cl=cl: self.run_call(cl, stream) for cl in self.calls]

    def e2e(self, stream, steps, warmup, flush=None):
        """Per step: one copy of q, k, v and the positions in, the call, the
        rotated q back; the cache stays resident."""
        torch = self.torch
        inp = Packed(torch, [self.q, self.k, self.v, self.pos])
        q, k, v, pos = inp.dev
        hout = torch.empty(self.q_out.shape, dtype=torch.bfloat16, pin_memory=True)

        def one():
            inp.h2d()
            self.sa.sa_rope_append(q, k, v, self.seq, pos, self.table, self.kv, 1, self.q_out, stream=stream)
            hout.copy_(self.q_out, non_blocking=True)

        ms = timed_loop(torch, stream, one, steps, warmup, flush)
        return ms, inp.nbytes, hout.numel() * 2

    def oracle_sample(self, budget_s, max_seqs=None):
        """The oracle's rotation + cache write of the first n tokens."""
        import copy
        import numpy as np
        from oracle import rope as R
        n = 256 if max_seqs is None else max(1, min(self.T, 32 * max_seqs))
        kc = self.kv.k.cpu().view(self.torch.int16).numpy().view(np.uint16).copy()
        vc = self.kv.v.cpu().view(self.torch.int16).numpy().view(np.uint16).copy()
        d = self.kv.as_dict()
        cache = dict(k=kc, v=vc, dtype="bf16", page_table=self.kv.page_table.cpu().numpy(),
                     page_size=self.kv.page_size, stride_page=d["stride_page"], stride_head=d["stride_head"],
                     stride_token=d["stride_token"], k_scale=1.0, v_scale=1.0)
        q = self.q[:n].double().cpu().numpy()
        k = self.k[:n].double().cpu().numpy()
        v = self.v[:n].double().cpu().numpy()
        seq = self.seq[:n].cpu().numpy()
        pos = self.pos[:n].cpu().numpy()
        t0 = time.time()
        R.rope_append(q, k, v, seq, pos, self.yarn, cache)
        dt = time.time() - t0
        nbytes = self.step_bytes * n / self.T
        return dt, nbytes, "%d of %d tokens, every head" % (n, self.T)


def make_bench(sa, cfg, device, batch=None):
    if batch is not None and cfg in (2, 4, 5):
        return DecodeBench(sa, cfg, device, batch=batch)
    if cfg in ROPE_CONFIGS:
        return RopeBench(sa, cfg, device)
    if cfg in PREFILL_CONFIGS:
        return PrefillBench(sa, cfg, device)
    if cfg in MULTI_CONFIGS:
        return MultiDecodeBench(sa, cfg, device)
    return DecodeBench(sa, cfg, device)


class PrefillBench:
    """One step = the prefill calls of the workload (full context, then window
    128), or the calls of the given windows only.  With sa=None (the reference
    arm) only the inputs are built."""

    def __init__(self, sa, cfg, device, windows=None, case=None):
        import torch
        import workloads as W
        self.sa, self.cfg, self.torch = sa, cfg, torch
        self.q8 = cfg == 10
        self.case = case if case is not None else W.make_config(7 if self.q8 else cfg, window=0, device=device)
        c = self.case
        self.T, self.Hq, self.D = c.q.shape
        if self.q8:  # per-tensor E4M3 codes of q (scale = amax / 448, nearest-even cast)
            self.q_scale = float(c.q.float().abs().max()) / 448.0
            self.q_codes = (c.q.float() / self.q_scale).to(torch.float8_e4m3fn).view(torch.uint8)
        self.Hkv = c.kv.num_kv_heads
        cu = c.cu_seqlens_q.cpu()
        self.q_lens = [int(x) for x in (cu[1:] - cu[:-1])]
        self.kv_lens = [int(x) for x in c.seqlens.cpu()]
        self.sample_units = self.T
        self.calls = []
        for w in (windows_of(cfg) if windows is None else windows):
            out = lse = None
            if sa is not None:
                out = torch.empty(self.T, self.Hq, self.D, dtype=torch.bfloat16, device=device)
                lse = torch.empty(self.T, self.Hq, dtype=torch.float32, device=device)
            self.calls.append(dict(window=w, out=out, lse=lse,
                                   flops=prefill_flops(self.q_lens, self.kv_lens, w, self.Hq, self.D)))
        self.step_flops = sum(cl["flops"] for cl in self.calls)
        self.kernels_per_step = len(self.calls)
        self.unit = "TFLOP/s"
        self.elem = 1 if c.kv.dtype == "e4m3" else 2
        self.dtype_name = "bf16" if self.elem == 2 else "fp8-e4m3 kv (widened to f16 for the products), bf16 q/out"
        self.fp8_qk_share = 0.0
        if self.q8:
            self.dtype_name = "fp8-e4m3 q and k (kind::f8f6f4 Q K^T), v widened to f16 for P V, bf16 out"
            self.fp8_qk_share = 0.5  # Q K^T and P V have equal flops
        self.e2e_api = "sa_prefill with pinned host q, k, v in, out/lse of every call back"
        self.label = None
        if windows is not None:  # a sub-step of the workload: name its calls
            base = workload_name(cfg).split(", step =")[0]
            self.label = "%s, call%s %s" % (base, "s" if len(windows) > 1 else "",
                                            " + ".join("w=%d" % w for w in windows))
        self.B = len(self.q_lens)
        self.maxlen = max(self.kv_lens)
        if self.streamed_e2e():
            self.e2e_api = ("sa_prefill from pinned host q, k, v, streamed in 4 query chunks (chunk i's rows in on a "
                            "copy stream, its calls for those queries against keys up to its last position, its "
                            "out/lse back on a third stream)")
        # algorithmic bytes of a call: q in, out and lse back, and the K/V rows
        # some query of the call sees (a window call is bound by these, not by flops)
        qe = 1 if self.q8 else 2
        for cl in self.calls:
            w = cl["window"]
            keys = sum(min(L, lq + w - 1) if w > 0 else L for lq, L in zip(self.q_lens, self.kv_lens))
            cl["bytes"] = (sum(self.q_lens) * self.Hq * (self.D * qe + self.D * 2 + 4)
                           + keys * self.Hkv * self.D * 2 * self.elem)

    def amount(self):
        return self.step_flops / 1e12

    def resident_bytes(self):
        """q (or its codes) and the cache."""
        c = self.case
        q = self.q_codes if self.q8 else c.q
        return q.numel() * q.element_size() + (c.kv.k.numel() + c.kv.v.numel()) * c.kv.k.element_size()

    def run_call(self, cl, stream, ev=None, q=None, kv=None, out=None, lse=None):
        c = self.case
        kv = c.kv if kv is None else kv
        out = cl["out"] if out is None else out
        lse = cl["lse"] if lse is None else lse
        if ev is not None:
            ev[0].record(stream)
        if self.q8:
            self.sa.sa_prefill_q8(self.q_codes if q is None else q, self.q_scale, c.cu_seqlens_q, kv, c.seqlens,
                                  c.sinks, cl["window"], c.sm_scale, out, lse, max_q_len=max(self.q_lens),
                                  max_kv_len=self.maxlen, stream=stream)
        else:
            self.sa.sa_prefill(c.q if q is None else q, c.cu_seqlens_q, kv, c.seqlens, c.sinks, cl["window"],
                               c.sm_scale, out, lse, max_q_len=max(self.q_lens), max_kv_len=self.maxlen,
                               stream=stream)
        if ev is not None:
            ev[1].record(stream)

    def step(self, stream, evs=None):
        for i, cl in enumerate(self.calls):
            self.run_call(cl, stream, None if evs is None else evs[i])

    def dominant(self):
        return 0, "prefill_kernel", self.calls[0]["flops"]

    def bound_of(self, i):
        """The roofline that bounds call i: a full-context call is a dense
        contraction (tensor), a window-128 call does about 111 flop per HBM
        byte, below the ridge (hbm)."""
        cl = self.calls[i]
        return "tensor" if cl["flops"] / cl["bytes"] > 300 else "hbm"

    def segment_names(self):
        return ["prefill w=%d" % cl["window"] for cl in self.calls]

    def notes(self, seg_ms, peaks):
        """Window calls against their HBM roofline as well as in TFLOP/s."""
        out = {}
        hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        for cl, ms in zip(self.calls, seg_ms):
            if cl["window"] > 0:
                gbs = cl["bytes"] / 1e6 / ms
                out["prefill w=%d" % cl["window"]] = {
                    "us": round(ms * 1e3, 1), "TFLOP/s": round(cl["flops"] / 1e9 / ms, 1),
                    "algorithmic_bytes": cl["bytes"], "GB/s": round(gbs, 1), "frac_of_hbm": round(gbs / hbm, 4),
                    "hbm_floor_us": round(cl["bytes"] / hbm / 1e3, 1)}
        return out

    def segments(self, stream):
        """The step as launch segments: one per call."""
        return [lambda cl=cl: self.run_call(cl, stream) for cl in self.calls]

    def e2e(self, stream, steps, warmup, flush=None):
        """Per step: one copy of q (or its codes), k and v in, the calls, one
        copy of every call's out and lse back.  A single contiguous sequence
        streams instead (e2e_streamed)."""
        import dataclasses
        torch = self.torch
        c = self.case
        if self.streamed_e2e():
            return self.e2e_streamed(stream, steps, warmup, flush)
        inp = Packed(torch, [self.q_codes if self.q8 else c.q, c.kv.k, c.kv.v])
        q = inp.dev[0]
        kv = dataclasses.replace(c.kv, k=inp.dev[1], v=inp.dev[2])
        res = Packed(torch, [t for cl in self.calls for t in (cl["out"], cl["lse"])])

        def one():
            inp.h2d()
            for i, cl in enumerate(self.calls):
                self.run_call(cl, stream, q=q, kv=kv, out=res.dev[2 * i], lse=res.dev[2 * i + 1])
            res.d2h()

        ms = timed_loop(torch, stream, one, steps, warmup, flush)
        return ms, inp.nbytes, res.nbytes

    def streamed_e2e(self):
        c = self.case
        return self.B == 1 and c.kv.page_table is None and c.kv.layout == "NHD" and not self.q8 and self.T % 4 == 0

    def e2e_streamed(self, stream, steps, warmup, flush=None, chunks=4):
        """One sequence from pinned host memory, in `chunks` query chunks: the
        rows of chunk i (its q, and the k and v of its positions) go in on a
        copy stream; on the compute stream each call runs for the chunk's
        queries against the keys up to its last position (chunked prefill:
        the same rows, positions and flops as the whole call); the chunk's out
        and lse come back on a third stream.  Later chunks' copies overlap
        earlier chunks' calls.  Every input byte goes in and every result byte
        comes back once per step."""
        import dataclasses
        torch = self.torch
        c = self.case
        T, Tc = self.T, self.T // chunks
        k, v = c.kv.k, c.kv.v  # [1, page, Hkv, D]: token-major rows of one sequence
        hq = c.q.cpu().pin_memory()
        hk, hv = k.cpu().pin_memory(), v.cpu().pin_memory()
        dq, dk, dv = torch.empty_like(c.q), torch.empty_like(k), torch.empty_like(v)
        kv = dataclasses.replace(c.kv, k=dk, v=dv)
        res = [(torch.empty_like(cl["out"]), torch.empty_like(cl["lse"])) for cl in self.calls]
        hres = [(torch.empty(o.shape, dtype=o.dtype, pin_memory=True), torch.empty(l.shape, dtype=l.dtype, pin_memory=True))
                for o, l in res]
        cu = torch.tensor([0, Tc], dtype=torch.int32, device="cuda")
        kv_len = [torch.tensor([(i + 1) * Tc], dtype=torch.int32, device="cuda") for i in range(chunks)]
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

        def one():
            start = torch.cuda.Event()
            start.record(stream)
            s_in.wait_event(start)
            s_out.wait_event(start)
            landed = []
            with torch.cuda.stream(s_in):
                for i in range(chunks):
                    r = slice(i * Tc, (i + 1) * Tc)
                    dq[r].copy_(hq[r], non_blocking=True)
                    dk[0, r].copy_(hk[0, r], non_blocking=True)
                    dv[0, r].copy_(hv[0, r], non_blocking=True)
                    e = torch.cuda.Event()
                    e.record(s_in)
                    landed.append(e)
            done = []
            for i in range(chunks):
                r = slice(i * Tc, (i + 1) * Tc)
                stream.wait_event(landed[i])
                for cl, (o, l) in zip(self.calls, res):
                    self.sa.sa_prefill(dq[r], cu, kv, kv_len[i], c.sinks, cl["window"], c.sm_scale, o[r], l[r],
                                       max_q_len=Tc, max_kv_len=(i + 1) * Tc, stream=stream)
                e = torch.cuda.Event()
                e.record(stream)
                done.append(e)
            with torch.cuda.stream(s_out):
                for i in range(chunks):
                    r = slice(i * Tc, (i + 1) * Tc)
                    s_out.wait_event(done[i])
                    for (o, l), (ho, hl) in zip(res, hres):
                        ho[r].copy_(o[r], non_blocking=True)
                        hl[r].copy_(l[r], non_blocking=True)
            end = torch.cuda.Event()
            end.record(s_out)
            stream.wait_event(end)

        ms = timed_loop(torch, stream, one, steps, warmup, flush)
        h2d = (c.q.numel() + 2 * T * self.Hkv * self.D) * 2
        d2h = sum(o.numel() * o.element_size() + l.numel() * l.element_size() for o, l in res)
        return ms, h2d, d2h

    def oracle_sample(self, budget_s, max_seqs=None):
        """Rows of the sequence, all heads: the first, then every k-th."""
        import numpy as np
        import oracle
        oracle.build()
        if getattr(self, "_cpu_case", None) is None:
            self._cpu_case = self.case.to("cpu")
        cpu = self._cpu_case
        rows = oracle.prefill_rows(cpu.cu_seqlens_q, cpu.seqlens)
        n = 64 if max_seqs is None else max(1, min(self.T, max_seqs))
        sel = np.linspace(0, self.T - 1, n).astype(np.int32)
        t0 = time.time()
        flops = 0
        for cl in self.calls:
            sr = np.repeat(sel, self.Hq)
            sh = np.tile(np.arange(self.Hq, dtype=np.int32), len(sel))
            if self.q8:
                oracle.attend(self.q_codes.cpu(), rows[0], rows[1], cpu.kv.as_dict(), cpu.seqlens, cpu.sinks,
                              cl["window"], cpu.sm_scale, sr, sh, q_scale=self.q_scale)
            else:
                oracle.attend(cpu.q, rows[0], rows[1], cpu.kv.as_dict(), cpu.seqlens, cpu.sinks, cl["window"],
                              cpu.sm_scale, sr, sh)
            for r in sel:
                p = int(rows[1][r])
                nk = p + 1 if cl["window"] <= 0 else min(cl["window"], p + 1)
                flops += 4 * self.Hq * self.D * nk
        dt = time.time() - t0
        return dt, flops, "%d of %d query rows x %d heads, every call (windows %s)" % (
            len(sel), self.T, self.Hq, [cl["window"] for cl in self.calls])


# ------------------------------------------------------------------- main
def cpu_baseline(wl, budget_s):
    """The oracle, as it stands, on a bounded sample of the workload: the
    sample grows (doubling from one unit: a sequence, a query row, 32 tokens)
    until one sample takes a tenth of the budget, then repeats until the
    budget is spent.  Returns (amount in the workload's unit, seconds,
    description)."""
    import oracle
    n, dt, amount, reps, desc = 1, 0.0, 0.0, 0, ""
    while True:
        d1, a1, desc = wl.oracle_sample(budget_s, max_seqs=n)
        dt, amount, reps = dt + d1, amount + a1, reps + 1
        if d1 >= budget_s / 10 or n >= wl.sample_units or dt >= budget_s:
            break
        n = min(2 * n, wl.sample_units)
    while dt < budget_s and reps < 1000:
        d1, a1, desc = wl.oracle_sample(budget_s, max_seqs=n)
        dt, amount, reps = dt + d1, amount + a1, reps + 1
    scale = 1e9 if wl.unit == "GB/s" else 1e12
    return {"value": round(amount / scale / dt, 6), "unit": wl.unit,
            "cores": getattr(wl, "oracle_cores", 0) or oracle.num_threads(), "kind": "oracle",
            "sample": "%s; timed %d times" % (desc, reps), "seconds": round(dt, 2)}


def workload_config(cfg, wl, world):
    """The workload the line is quoted on (identical in both arms)."""
    return {"workload": getattr(wl, "label", None) or workload_name(cfg), "global_batch": wl.B * world,
            "seq_len_max": wl.maxlen,
            "parallelism": "replicas" if world > 1 else "single GPU"}


def measure(wl, cfg, args, world, rank, stream, sampler, steps, cpu_budget_s):
    """Times one workload on this GPU and returns its record.

    Two passes of K steps after W warm-up steps.  The first times whole steps
    with CUDA events on the launching stream at step boundaries only (no event
    between a step's launches): the step time is the median over the K steps
    (the mean is given beside it), and `value` = the step's algorithmic work /
    that time.  The second repeats the steps with an event after every launch
    segment: the dominant kernel's average launch time and the per-segment
    breakdown.  Inputs under twice the L2 size are evicted before every step,
    outside the events."""
    import torch
    peaks, peak_src = load_peaks()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            wl.step(stream)
    torch.cuda.synchronize()
    # Inputs smaller than twice the L2 (129 MB) are evicted before every step
    # by a 256 MB write outside the step's events, followed by a 256 MB read
    # of a second buffer: the read evicts the write's dirty lines, so their
    # write-back to DRAM happens before the step and not inside it.
    flush_buf = flush = None
    if wl.resident_bytes() < L2_FLUSH_BYTES:
        flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        flush_rd = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device="cuda")

        def flush():
            flush_buf.zero_()
            flush_rd.sum()
    ci, kname, kwork = wl.dominant()
    segs = wl.segments(stream)
    runs = list(segs)
    if args.graph:
        runs = []
        for fn in segs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn()
            runs.append(g.replay)
        torch.cuda.synchronize()
    step_evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(runs) + 1)] for _ in range(steps)]
    dist_barrier(world)
    torch.cuda.synchronize()
    t_begin = time.time()
    with torch.cuda.stream(stream):  # the timed region: K steps
        for i in range(steps):
            if flush is not None:
                flush()
            step_evs[i][0].record(stream)
            for run in runs:
                run()
            step_evs[i][1].record(stream)
    torch.cuda.synchronize()
    t_end = time.time()
    dist_barrier(world)
    with torch.cuda.stream(stream):  # the segment breakdown: K more steps
        for i in range(steps):
            if flush is not None:
                flush()
            evs[i][0].record(stream)
            for j, run in enumerate(runs):
                run()
                evs[i][j + 1].record(stream)
    torch.cuda.synchronize()
    dist_barrier(world)
    step_ms = [e[0].elapsed_time(e[1]) for e in step_evs]
    ms = dist_max(statistics.median(step_ms), world)
    ms_mean = dist_max(statistics.fmean(step_ms), world)
    seg_ms = [statistics.fmean(e[j].elapsed_time(e[j + 1]) for e in evs) for j in range(len(runs))]
    k_ms = statistics.fmean(e[ci].elapsed_time(e[ci + 1]) for e in evs)

    bound = wl.bound_of(0) if hasattr(wl, "bound_of") else ("hbm" if wl.unit == "GB/s" else "tensor")
    if bound == "hbm":
        kbytes = kwork if wl.unit == "GB/s" else wl.calls[0]["bytes"]
        achieved = kbytes / 1e9 / (k_ms / 1e3)
        peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        nominal, runit, peak_name = 8000.0, "GB/s", "hbm_gbs"
        work_key, work = "algorithmic_bytes_per_launch", kbytes
    else:
        achieved = kwork / 1e12 / (k_ms / 1e3)
        # one isolated launch of under a millisecond behind an L2 flush, not a
        # seconds-long loop: the burst figure
        peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        nominal, runit, peak_name = 2250.0, "TFLOP/s", "bf16_tflops (burst)"
        work_key, work = "algorithmic_flops_per_launch", kwork
        # Q K^T on E4M3 runs at FP8 rate (2x the 16-bit rate, the nominal 4.5 / 2.25
        # PFLOP/s ratio), P V at the 16-bit rate; half the flops each: the peak of
        # that mix is F / (F/2 / 2P + F/2 / P) = 4/3 P
        mix = getattr(wl, "fp8_qk_share", 0.0)
        if mix:
            scale = 1.0 / (mix / 2.0 + (1.0 - mix))
            peak, nominal = peak * scale, nominal * scale
            peak_name += ", scaled for FP8 Q K^T (%.0f %% of the flops at 2x rate)" % (100 * mix)
    traffic = ncu_traffic(kname, "config%d" % cfg)

    e2e_ms, h2d, d2h = wl.e2e(stream, max(3, min(steps, 200)), 3, flush)
    rec = {
        "value": round(wl.amount() * world / (ms / 1e3), 2), "unit": wl.unit, "steps": steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 6), "ms_per_step_mean": round(ms_mean, 6),
        "dtype": wl.dtype_name, "config": workload_config(cfg, wl, world),
        "method": {"splits": [cl.get("S", 1) for cl in wl.calls],
                   "l2": ("flushed before every step (256 MB write, then a 256 MB read of another buffer so "
                          "that no dirty line is left to write back; outside the step's events)"
                          if flush_buf is not None else
                          "inputs larger than twice the L2 (%.2f GB per step); no flush" % (wl.resident_bytes() / 1e9)),
                   "launch": "each launch segment of the step captured as a CUDA graph and replayed"
                             if args.graph else "eager",
                   "timing": "CUDA events around each step on its stream, none between a step's launches; "
                             "ms_per_step and value from the median of the K steps (mean beside it). A second "
                             "pass of K steps with an event after every launch segment times the dominant kernel "
                             "(avg_launch_ms, a mean) and the segments."},
        "roofline": {"bound": bound, "achieved": round(achieved, 1), "peak": peak, "unit": runit,
                     "frac": round(achieved / peak, 4), "traffic": traffic, "kernel": kname, work_key: work,
                     "avg_launch_ms": round(k_ms, 6), "peak_source": "%s %s" % (peak_src, peak_name),
                     "frac_of_nominal": round(achieved / nominal, 4)},
        "clocks": sampler.summary(t_begin, t_end) if sampler else None,
        "e2e": {"value": round(wl.amount() * world / (e2e_ms / 1e3), 2), "unit": wl.unit,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "api": wl.e2e_api},
        "gpu_launches": steps * wl.kernels_per_step,  # the library's kernels in the timed region (the flush is torch's)
        "segments": [{"name": n, "ms": round(t, 6)} for n, t in
                     zip(getattr(wl, "segment_names", lambda: ["segment %d" % j for j in range(len(seg_ms))])(),
                         seg_ms)],
    }
    if hasattr(wl, "notes"):
        notes = wl.notes(seg_ms, peaks)
        if notes:
            rec["notes"] = notes
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rec["cpu_baseline"] = cpu_baseline(wl, cpu_budget_s)
        if cfg == 1:  # the smallest workload: the oracle on one thread as well
            import oracle
            cores = oracle.num_threads()
            oracle.set_num_threads(1)
            try:
                rec["cpu_baseline"]["single_thread_value"] = cpu_baseline(wl, 3.0)["value"]
            finally:
                oracle.set_num_threads(cores)
    return rec


HEADLINE = 4  # decode B=128, L=32768: the largest single-GPU decode workload


def run_native(args, world, rank, local):
    import torch
    import gqa_attention_sinks_head_gb300 as sa
    sa.build()
    sa.load()
    torch.cuda.set_device(local)
    dist_init(world, "nccl")
    stream = torch.cuda.Stream()
    sampler = ClockSampler(local) if rank == 0 else None
    if args.config is not None:  # one workload
        cfg = args.config
        steps = args.steps if args.steps is not None else DEFAULT_STEPS[cfg]
        rec = measure(make_bench(sa, cfg, "cuda", args.batch), cfg, args, world, rank, stream, sampler, steps, 10.0)
        subs = {}
    else:
        # The default line: decode B=128, L=32768 (split-KV) as the headline;
        # then, as sub-records with their own roofline, cpu_baseline and e2e,
        # the B=64 ragged decode step (full context and window 128) and each
        # call of the T=8192 prefill.
        def steps_of(cfg):
            return args.steps if args.steps is not None else DEFAULT_STEPS[cfg]
        wl = make_bench(sa, HEADLINE, "cuda")
        rec = measure(wl, HEADLINE, args, world, rank, stream, sampler, steps_of(HEADLINE), 10.0)
        del wl
        torch.cuda.empty_cache()
        subs = {}
        wl = make_bench(sa, 2, "cuda")
        subs["decode_ragged"] = measure(wl, 2, args, world, rank, stream, sampler, steps_of(2), 6.0)
        del wl
        torch.cuda.empty_cache()
        import workloads as W
        case = W.make_config(3, window=0, device="cuda")
        calls = []
        for w in (0, 128):
            wl = PrefillBench(sa, 3, "cuda", windows=[w], case=case)
            r = measure(wl, 3, args, world, rank, stream, sampler, steps_of(3), 6.0)
            r["window"] = w
            calls.append(r)
            del wl
        subs["prefill"] = {"workload": workload_name(3), "calls": calls}
    if sampler:
        sampler.stop()
    if rank == 0:
        line = {"metric": METRIC, "value": rec["value"], "unit": rec["unit"], "n_gpus": world,
                "steps": rec["steps"], "warmup": rec["warmup"], "ms_per_step": rec["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": rec["dtype"],
                "data": "synthetic (seeded; N(0,1) q/k/v, sinks U(-2,6)); no weights or datasets"}
        line.update({k: v for k, v in rec.items() if k not in line})
        line.update(subs)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args, world, rank, local):
    """The oracle, as it stands, timed on the host cores on the native arm's
    headline workload (the same seeded bytes, drawn with torch on the same
    device); each step is a bounded sample of it.  The CUDA library is not
    loaded."""
    if rank != 0:
        return
    import torch
    import oracle
    cfg = HEADLINE if args.config is None else args.config
    oracle.build()
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    wl = make_bench(None, cfg, dev)
    total_budget = float(args.budget_s)
    steps = args.steps if args.steps is not None else DEFAULT_STEPS[cfg]
    warmup = args.warmup
    # size the per-step sample from a one-unit pilot
    dt1, _, _ = wl.oracle_sample(5.0, max_seqs=1)
    per_step = total_budget / max(1, steps + warmup)
    n = max(1, min(wl.sample_units, int(per_step / max(dt1, 1e-6))))
    for _ in range(warmup):
        wl.oracle_sample(per_step, max_seqs=n)
    t0 = time.time()
    amount = 0
    desc = ""
    for _ in range(steps):
        _, a, desc = wl.oracle_sample(per_step, max_seqs=n)
        amount += a
    dt = time.time() - t0
    value = amount / (1e9 if wl.unit == "GB/s" else 1e12) / dt
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": wl.unit, "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": round(dt / steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded), same bytes as the native arm",
        "config": workload_config(cfg, wl, 1),
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 4), "unit": wl.unit,
                         "cores": getattr(wl, "oracle_cores", 0) or oracle.num_threads(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(value, 4), "unit": wl.unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--config", type=int, default=None, choices=[1, 2, 3, 4, 5, 6, 7, 8, 9, 10],
                    help="one workload only (default: the headline decode B=128 L=32768 with the B=64 ragged "
                         "decode and the T=8192 prefill calls as sub-records)")
    ap.add_argument("--batch", type=int, default=None,
                    help="with --config 2, 4 or 5: only the first N sequences (a smaller case, e.g. for a profiler)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="capture each launch segment of the step as a CUDA graph and replay it")
    ap.add_argument("--budget-s", type=float, default=120.0,
                    help="reference arm: host seconds the whole --steps/--warmup run may take")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)
    world, rank, local = dist_info()
    if args.impl == "reference":
        run_reference(args, world, rank, local)
    else:
        run_native(args, world, rank, local)


if __name__ == "__main__":
    main()
