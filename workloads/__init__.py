"""Seeded synthetic inputs for sink attention.

This module only draws numbers and lays them out; it holds none of the
attention arithmetic.  Both the CUDA path (tests, bench) and the fp64 oracle
read the tensors it returns, so that the two sides see identical bytes.

Shapes and distributions follow the gpt-oss attention layer: 64 query heads,
8 kv heads (GQA 8:1), head_dim 64, bf16 Q/K/V ~ N(0, 1), fp32 sinks ~ U(-2, 6),
softmax scale 1/8, paged KV with 16-token pages and a randomly permuted page
table, and an FP8-E4M3 cache quantised with one fp32 scale per tensor
(scale = amax / 448, codes = round-to-nearest-even saturating cast).

NaN poison: every page that no sequence references, every table entry past a
sequence's last page (it points at a poison page), and every slot at or past
L_b in a sequence's last page is filled with NaN (bf16 NaN, or E4M3 code 0x7F),
so that any out-of-range read shows up as a NaN in the output.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

E4M3_MAX = 448.0
E4M3_NAN_CODE = 0x7F
_CHUNK = 1 << 24


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _fill_normal(out: torch.Tensor, g: torch.Generator) -> torch.Tensor:
    """Fill `out` (any float dtype) with N(0, 1) draws, in chunks of fp32."""
    flat = out.view(-1)
    for s in range(0, flat.numel(), _CHUNK):
        n = min(_CHUNK, flat.numel() - s)
        flat[s:s + n] = torch.randn(n, generator=g, device=out.device, dtype=torch.float32).to(out.dtype)
    return out


def _quantise_e4m3(out_codes: torch.Tensor, seed: int, device) -> float:
    """Draw N(0,1) into `out_codes` (uint8 E4M3 codes) with a per-tensor scale.

    Two passes over the same seeded stream: the first finds amax, the second
    quantises x / scale with torch's saturating round-to-nearest cast."""
    flat = out_codes.view(-1)
    g = _gen(seed, device)
    amax = 0.0
    for s in range(0, flat.numel(), _CHUNK):
        n = min(_CHUNK, flat.numel() - s)
        x = torch.randn(n, generator=g, device=device, dtype=torch.float32)
        amax = max(amax, float(x.abs().max()))
    scale = amax / E4M3_MAX if amax > 0 else 1.0
    g = _gen(seed, device)
    for s in range(0, flat.numel(), _CHUNK):
        n = min(_CHUNK, flat.numel() - s)
        x = torch.randn(n, generator=g, device=device, dtype=torch.float32)
        flat[s:s + n] = (x / scale).to(torch.float8_e4m3fn).view(torch.uint8)
    return float(scale)


@dataclass
class KVCache:
    """A paged (or contiguous) KV cache plus the metadata both sides read."""
    k: torch.Tensor                  # [num_pages, Hkv, P, D] bf16, or uint8 E4M3 codes
    v: torch.Tensor
    dtype: str                       # "bf16" | "e4m3"
    page_table: torch.Tensor | None  # [B, max_pages] int32, or None (sequence b uses page b)
    page_size: int
    k_scale: float = 1.0
    v_scale: float = 1.0
    layout: str = "HND"              # HND: [page, head, token, dim]; NHD: [page, token, head, dim]

    @property
    def num_pages(self) -> int:
        return int(self.k.shape[0])

    @property
    def num_kv_heads(self) -> int:
        return int(self.k.shape[1] if self.layout == "HND" else self.k.shape[2])

    @property
    def head_dim(self) -> int:
        return int(self.k.shape[3])

    def strides(self):
        """(stride_page, stride_head, stride_token) in elements."""
        s = self.k.stride()
        if self.layout == "HND":
            return s[0], s[1], s[2]
        return s[0], s[2], s[1]

    def as_dict(self) -> dict:
        sp, sh, st = self.strides()
        return dict(k=self.k, v=self.v, dtype=self.dtype, num_pages=self.num_pages,
                    num_kv_heads=self.num_kv_heads, head_dim=self.head_dim,
                    page_size=self.page_size, stride_page=sp, stride_head=sh, stride_token=st,
                    page_table=self.page_table,
                    page_table_stride=0 if self.page_table is None else int(self.page_table.shape[1]),
                    k_scale=self.k_scale, v_scale=self.v_scale)

    def to(self, device) -> "KVCache":
        return KVCache(self.k.to(device), self.v.to(device), self.dtype,
                       None if self.page_table is None else self.page_table.to(device),
                       self.page_size, self.k_scale, self.v_scale, self.layout)


@dataclass
class Case:
    """One attention call's inputs (decode: one query row per sequence)."""
    q: torch.Tensor                  # [rows, Hq, D] bf16
    kv: KVCache
    seqlens: torch.Tensor            # [B] int32: keys held by each sequence
    sinks: torch.Tensor | None       # [Hq] fp32
    window: int
    sm_scale: float
    cu_seqlens_q: torch.Tensor | None = None  # prefill: [B+1] int32
    name: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.seqlens.shape[0])

    def to(self, device) -> "Case":
        return Case(self.q.to(device), self.kv.to(device), self.seqlens.to(device),
                    None if self.sinks is None else self.sinks.to(device), self.window,
                    self.sm_scale, None if self.cu_seqlens_q is None else self.cu_seqlens_q.to(device),
                    self.name, dict(self.meta))


def _nan_like(dtype_name: str):
    return float("nan") if dtype_name == "bf16" else E4M3_NAN_CODE


def make_kv(seqlens, num_kv_heads: int, head_dim: int, page_size: int, *, paged: bool = True,
            kv_dtype: str = "bf16", poison_pages: int = 0, seed: int = 0, device="cpu",
            layout: str = "HND", poison: bool = True) -> KVCache:
    """Paged KV cache for sequences of the given lengths.

    paged=True: pages of `page_size` tokens, assigned to sequences through a
    random permutation of the pool (sum ceil(L_b/P) pages + `poison_pages`
    unreferenced NaN pages).  paged=False: one page per sequence holding
    `page_size` >= max L_b tokens and no table."""
    L = [int(x) for x in seqlens]
    B = len(L)
    P = int(page_size)
    npages_seq = [max(1, math.ceil(l / P)) for l in L] if paged else [1] * B
    if not paged:
        assert P >= max(L + [1])
    n_live = sum(npages_seq)
    num_pages = n_live + (int(poison_pages) if paged else 0)
    if layout == "HND":
        shape = (num_pages, num_kv_heads, P, head_dim)
    else:
        shape = (num_pages, P, num_kv_heads, head_dim)
    store = torch.bfloat16 if kv_dtype == "bf16" else torch.uint8
    k = torch.empty(shape, dtype=store, device=device)
    v = torch.empty(shape, dtype=store, device=device)
    if kv_dtype == "bf16":
        g = _gen(seed, device)
        _fill_normal(k, g)
        _fill_normal(v, g)
        k_scale = v_scale = 1.0
    else:
        k_scale = _quantise_e4m3(k, seed, device)
        v_scale = _quantise_e4m3(v, seed + 7919, device)

    table = None
    if paged:
        g = _gen(seed + 1, "cpu")
        perm = torch.randperm(num_pages, generator=g).to(torch.int32)
        live = perm[:n_live]
        dead = perm[n_live:]
        max_pages = max(npages_seq)
        fill = int(dead[0]) if dead.numel() > 0 else 0
        table = torch.full((B, max_pages), fill, dtype=torch.int32)
        o = 0
        for b in range(B):
            table[b, :npages_seq[b]] = live[o:o + npages_seq[b]]
            o += npages_seq[b]
        if poison and dead.numel() > 0:
            k[dead.to(device).long()] = _nan_like(kv_dtype)
            v[dead.to(device).long()] = _nan_like(kv_dtype)
        table = table.to(device)
    if poison:
        for b in range(B):
            tail = L[b] % P if paged else L[b]
            if paged and tail == 0:
                continue
            last = int(table[b, npages_seq[b] - 1]) if paged else b
            if layout == "HND":
                k[last, :, tail:] = _nan_like(kv_dtype)
                v[last, :, tail:] = _nan_like(kv_dtype)
            else:
                k[last, tail:] = _nan_like(kv_dtype)
                v[last, tail:] = _nan_like(kv_dtype)
    return KVCache(k, v, kv_dtype, table, P, k_scale, v_scale, layout)


def make_decode_case(seqlens, *, num_qo_heads=64, num_kv_heads=8, head_dim=64, page_size=16,
                     paged=True, kv_dtype="bf16", window=0, sm_scale=0.125, sinks=True,
                     poison_pages=0, seed=0, device="cpu", layout="HND", name="",
                     poison=True) -> Case:
    L = torch.as_tensor([int(x) for x in seqlens], dtype=torch.int32)
    B = L.shape[0]
    kv = make_kv(L.tolist(), num_kv_heads, head_dim, page_size, paged=paged, kv_dtype=kv_dtype,
                 poison_pages=poison_pages, seed=seed + 11, device=device, layout=layout,
                 poison=poison)
    g = _gen(seed + 3, device)
    q = _fill_normal(torch.empty((B, num_qo_heads, head_dim), dtype=torch.bfloat16, device=device), g)
    s = None
    if sinks:
        s = torch.empty(num_qo_heads, dtype=torch.float32, device=device).uniform_(-2.0, 6.0, generator=g)
    return Case(q, kv, L.to(device), s, int(window), float(sm_scale), None, name)


def make_prefill_case(q_lens, kv_lens, *, num_qo_heads=64, num_kv_heads=8, head_dim=64,
                      page_size=None, paged=False, window=0, sm_scale=0.125, sinks=True,
                      poison_pages=0, seed=0, device="cpu", layout="NHD", kv_dtype="bf16", name="") -> Case:
    """Ragged prefill: sequence b has q_lens[b] queries (the last ones of its
    kv_lens[b] keys).  Contiguous NHD K/V by default: one page per sequence."""
    ql = [int(x) for x in q_lens]
    kl = [int(x) for x in kv_lens]
    assert all(a <= b for a, b in zip(ql, kl))
    if page_size is None:
        page_size = max(kl + [1]) if not paged else 16
        if not paged:
            page_size = ((page_size + 127) // 128) * 128
    kv = make_kv(kl, num_kv_heads, head_dim, page_size, paged=paged, kv_dtype=kv_dtype,
                 poison_pages=poison_pages, seed=seed + 11, device=device, layout=layout)
    g = _gen(seed + 3, device)
    T = sum(ql)
    q = _fill_normal(torch.empty((T, num_qo_heads, head_dim), dtype=torch.bfloat16, device=device), g)
    s = None
    if sinks:
        s = torch.empty(num_qo_heads, dtype=torch.float32, device=device).uniform_(-2.0, 6.0, generator=g)
    cu = torch.zeros(len(ql) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.as_tensor(ql, dtype=torch.int32), 0)
    return Case(q, kv, torch.as_tensor(kl, dtype=torch.int32, device=device), s, int(window),
                float(sm_scale), cu.to(device), name)


# ------------------------------------------------------------------- configs
CONFIG_SEED = 1000


def config_seqlens(cfg: int):
    if cfg == 1:
        return [256]
    if cfg == 2:
        g = _gen(CONFIG_SEED + 2, "cpu")
        return torch.randint(1024, 8192 + 1, (64,), generator=g).tolist()
    if cfg == 4:
        return [32768] * 128
    if cfg == 5:
        return [8192] * 256
    if cfg == 6:
        g = _gen(CONFIG_SEED + 6, "cpu")
        return torch.randint(2048, 16384 + 1, (8,), generator=g).tolist()
    raise ValueError(cfg)


def make_config(cfg: int, *, window: int = 0, device="cpu", batch: int | None = None) -> Case:
    """The five gpt-oss-shaped workloads (64 q / 8 kv heads, head_dim 64).

    1: decode, B=1, L=256, contiguous bf16, full causal.
    2: decode, B=64, L_b ~ U[1024, 8192], paged bf16 (P=16, permuted table,
       64 poison pages); window 0 or 128.
    3: prefill, one 8192-token sequence, contiguous bf16 NHD; window 0 or 128.
    4: decode, B=128, L=32768, paged bf16 (262,144 pages), split-KV.
    5: decode, B=256, L=8192, paged FP8-E4M3 (per-tensor scales); window 0 or 128.
    6: chunked prefill, B=8: each sequence appends 1024 queries to its paged
       context, L_kv ~ U[2048, 16384] (P=16, permuted table, HND, 64 poison
       pages), bottom-right causal; window 0 or 128.
    7: workload 6 on an FP8-E4M3 cache (per-tensor scales).
    8: multi-token decode: the cache of workload 2 (B=64, L_b ~ U[1024, 8192],
       paged bf16) with 4 new query tokens per sequence at L_b - 4 .. L_b - 1.

    batch: decode workloads (2, 4, 5) only, keep the first `batch` sequences
    (a smaller case of the same shape, e.g. for a profiler capture).
    """
    seed = CONFIG_SEED + cfg
    if batch is not None and cfg in (2, 4, 5):
        kl = config_seqlens(cfg)[:max(1, int(batch))]
        return make_decode_case(kl, page_size=16, paged=True, window=window, poison_pages=64 if cfg == 2 else 0,
                                kv_dtype="e4m3" if cfg == 5 else "bf16", seed=seed, device=device,
                                name="config %d, first %d sequences w=%d" % (cfg, len(kl), window))
    if cfg == 1:
        return make_decode_case([256], page_size=256, paged=False, window=window, seed=seed,
                                device=device, name="decode B=1 L=256 contiguous bf16")
    if cfg == 2:
        return make_decode_case(config_seqlens(2), page_size=16, paged=True, window=window,
                                poison_pages=64, seed=seed, device=device,
                                name="decode B=64 L~U[1024,8192] paged P=16 bf16 w=%d" % window)
    if cfg == 3:
        return make_prefill_case([8192], [8192], window=window, seed=seed, device=device,
                                 name="prefill T=8192 contiguous bf16 w=%d" % window)
    if cfg == 4:
        return make_decode_case(config_seqlens(4), page_size=16, paged=True, window=window, seed=seed,
                                device=device,
                                name="decode B=128 L=32768 paged P=16 bf16 split-KV")
    if cfg == 5:
        return make_decode_case(config_seqlens(5), page_size=16, paged=True, kv_dtype="e4m3",
                                window=window, seed=seed, device=device,
                                name="decode B=256 L=8192 paged P=16 fp8-e4m3 w=%d" % window)
    if cfg in (6, 7):
        kl = config_seqlens(6)
        dt = "bf16" if cfg == 6 else "e4m3"
        return make_prefill_case([1024] * len(kl), kl, paged=True, page_size=16, layout="HND", window=window,
                                 poison_pages=64, seed=seed, device=device, kv_dtype=dt,
                                 name="chunked prefill B=8 Lq=1024 L_kv~U[2048,16384] paged P=16 %s w=%d"
                                 % (dt, window))
    if cfg == 8:
        kl = config_seqlens(2)
        return make_prefill_case([4] * len(kl), kl, paged=True, page_size=16, layout="HND", window=window,
                                 poison_pages=64, seed=seed, device=device,
                                 name="multi-token decode B=64 q_len=4 L~U[1024,8192] paged P=16 bf16 w=%d" % window)
    raise ValueError(cfg)


def subset(case: Case, seq_ids) -> Case:
    """CPU copy of the listed sequences only (decode cases): their pages are
    gathered into a small pool and the table renumbered.  Lets the oracle read
    a sample of a workload whose cache is too large to copy whole."""
    kv = case.kv
    seq_ids = [int(s) for s in seq_ids]
    L = case.seqlens.cpu()[seq_ids]
    P = kv.page_size
    if kv.page_table is None:
        pages = torch.as_tensor(seq_ids, dtype=torch.long)
        k = kv.k[pages.to(kv.k.device)].cpu()
        v = kv.v[pages.to(kv.v.device)].cpu()
        nkv = KVCache(k, v, kv.dtype, None, P, kv.k_scale, kv.v_scale, kv.layout)
    else:
        npg = [(int(l) + P - 1) // P for l in L]
        table_cpu = kv.page_table.cpu()
        rows = [table_cpu[s, :n].long() for s, n in zip(seq_ids, npg)]
        allp = torch.cat(rows) if rows else torch.zeros(0, dtype=torch.long)
        allp_dev = allp.to(kv.k.device)
        k = kv.k[allp_dev].cpu()
        v = kv.v[allp_dev].cpu()
        if k.shape[0] == 0:  # keep one page so the pool is never empty
            k, v = kv.k[:1].cpu(), kv.v[:1].cpu()
        table = torch.zeros(len(seq_ids), max(npg + [1]), dtype=torch.int32)
        o = 0
        for i, n in enumerate(npg):
            table[i, :n] = torch.arange(o, o + n, dtype=torch.int32)
            o += n
        nkv = KVCache(k, v, kv.dtype, table, P, kv.k_scale, kv.v_scale, kv.layout)
    return Case(case.q.cpu()[seq_ids], nkv, L.to(torch.int32),
                None if case.sinks is None else case.sinks.cpu(), case.window, case.sm_scale,
                name=case.name + " (sequences %s)" % seq_ids[:8])
