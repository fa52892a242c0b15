"""Bit-exact mask and index probes for prefill and multi-token decode.

One key carries score 40 against 0 for every other key: a query row's output
is that key's value row bit for bit exactly when the key is visible to the
row (causal: key <= position; window w: key > position - w), and differs
from it otherwise.  Value rows encode (sequence, key), so a wrong page, slot
or row shows too.  Targets sweep tile edges (64 keys), page edges (16 keys),
the causal diagonal and the window edge for every query row."""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

P = 16


def probe_case(q_lens, kv_lens, window, layout, seed):
    case = W.make_prefill_case(q_lens, kv_lens, num_qo_heads=8, num_kv_heads=8, paged=True, page_size=P,
                               layout=layout, window=window, sinks=False, poison_pages=4, seed=seed)
    kv = case.kv
    hnd = layout == "HND"
    for b, L in enumerate(kv_lens):
        for t in range(L):
            pg, sl = int(kv.page_table[b, t // P]), t % P
            d = torch.arange(64, dtype=torch.float32)
            row = 1 + (d % 7)
            row[0], row[1], row[2] = 1 + (t & 255), 1 + (t >> 8), 1 + b
            # pseudo-random small integers: a mean of other rows cannot match them all
            row[3], row[4], row[5] = 1 + (t * 37 + b) % 101, 1 + (t * 53 + 7 * b) % 97, 1 + (t * 29 + 3) % 89
            if hnd:
                kv.k[pg, :, sl] = 0
                kv.v[pg, :, sl] = row.to(torch.bfloat16)
            else:
                kv.k[pg, sl] = 0
                kv.v[pg, sl] = row.to(torch.bfloat16)
    case.q.zero_()
    case.q[:, :, 0] = 16.0
    return case


def set_key(case_gpu, b, t, value, hnd):
    pg, sl = int(case_gpu.kv.page_table[b, t // P]), t % P
    if hnd:
        case_gpu.kv.k[pg, :, sl, 0] = value
        return case_gpu.kv.v[pg, 0, sl]
    case_gpu.kv.k[pg, sl, :, 0] = value
    return case_gpu.kv.v[pg, sl, 0]


def run_probe(sa, q_lens, kv_lens, window, layout, call):
    case = probe_case(q_lens, kv_lens, window, layout, seed=120)
    g = case.to("cuda")
    hnd = layout == "HND"
    cu = np.concatenate([[0], np.cumsum(q_lens)])
    targets = set()
    for L, Lq in zip(kv_lens, q_lens):
        off = L - Lq
        for base in (0, off, L - 1):
            for dt in (-129, -128, -127, -65, -64, -63, -17, -16, -15, -1, 0, 1, 15, 16, 17, 63, 64, 65, 127, 128):
                if 0 <= base + dt < L:
                    targets.add(base + dt)
    for t in sorted(targets):
        vrows = {}
        for b, L in enumerate(kv_lens):
            if t < L:
                vrows[b] = set_key(g, b, t, 20.0, hnd).clone()  # score 16 * 20 / 8 = 40
        out = call(g)
        for b, (L, Lq) in enumerate(zip(kv_lens, q_lens)):
            if b not in vrows:
                continue
            off = L - Lq
            rows = out[cu[b]:cu[b + 1], 0]
            for i in range(Lq):
                p = off + i
                visible = t <= p and (window == 0 or t > p - window)
                same = torch.equal(rows[i], vrows[b])
                assert same == visible, (b, t, i, p, visible)
        for b, L in enumerate(kv_lens):
            if t < L:
                set_key(g, b, t, 0.0, hnd)
    assert sa.sa_device_status() == 0


@pytest.mark.parametrize("window", [0, 128, 37])
@pytest.mark.parametrize("layout", ["HND", "NHD"])
def test_prefill_masks_bit_exact(sa, window, layout):
    q_lens, kv_lens = [300, 70], [300, 333]  # a full prefill and a chunk at the end of a longer context

    def call(g):
        T = int(sum(q_lens))
        out = torch.empty(T, 8, 64, dtype=torch.bfloat16, device="cuda")
        sa.sa_prefill(g.q, g.cu_seqlens_q, g.kv, g.seqlens, None, window, g.sm_scale, out, None,
                      max_q_len=max(q_lens), max_kv_len=max(kv_lens))
        torch.cuda.synchronize()
        return out

    run_probe(sa, q_lens, kv_lens, window, layout, call)


@pytest.mark.parametrize("window", [0, 128, 3])
@pytest.mark.parametrize("q_len", [2, 4, 7])
def test_multi_token_decode_masks_bit_exact(sa, window, q_len):
    kv_lens = [q_len + 1, 300, 1029]
    q_lens = [q_len] * len(kv_lens)

    def call(g):
        out = torch.empty(q_len * len(kv_lens), 8, 64, dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(max(sa.sa_decode_multi_workspace_size(3, q_len, 8, 8, 64, 1029, window, 3), 16),
                         dtype=torch.uint8, device="cuda")
        sa.sa_decode_multi(g.q, q_len, g.kv, g.seqlens, None, window, g.sm_scale, out, None, max_kv_len=1029,
                           workspace=ws, num_splits=3)
        torch.cuda.synchronize()
        return out

    run_probe(sa, q_lens, kv_lens, window, "HND", call)
