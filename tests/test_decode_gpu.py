"""GPU parity of sa_decode / sa_decode_partial / sa_merge_states against the
fp64 oracle, on small seeded cases that span several tiles, pages and ragged
tails (the NaN-poisoned pages and slots of the generator catch any read
outside a sequence), plus bit-exact page-table / mask probes."""
import math

import numpy as np
import pytest
import torch

import workloads as W
from sa_testlib import check_close, compact_decode_case, decode_gpu, oracle_decode

pytestmark = pytest.mark.gpu

LENS = [0, 1, 15, 16, 17, 100, 127, 128, 129, 255, 300, 1000, 1037]


def run_case(sa, oracle, case, splits=0, what=""):
    out, lse = decode_gpu(sa, case.to("cuda"), num_splits=splits)
    ref_o, ref_l = oracle_decode(oracle, case)
    check_close(out, lse, ref_o, ref_l, what)
    assert sa.sa_device_status() == 0
    return out, lse


@pytest.mark.parametrize("window", [0, 128, 1, 37])
@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_ragged_paged(sa, oracle, window, kv_dtype):
    case = W.make_decode_case(LENS, page_size=16, window=window, kv_dtype=kv_dtype, poison_pages=7, seed=100)
    run_case(sa, oracle, case, what="paged %s w=%d" % (kv_dtype, window))


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 64])
@pytest.mark.parametrize("window", [0, 128])
def test_split_counts_agree(sa, oracle, splits, window):
    case = W.make_decode_case([1, 40, 333, 1000, 2049], page_size=16, window=window, poison_pages=3, seed=101)
    run_case(sa, oracle, case, splits=splits, what="splits=%d w=%d" % (splits, window))


@pytest.mark.parametrize("page_size", [32, 64, 256])
@pytest.mark.parametrize("layout", ["HND", "NHD"])
def test_page_sizes_and_layouts(sa, oracle, page_size, layout):
    case = W.make_decode_case([5, 300, 700], page_size=page_size, layout=layout, poison_pages=2, seed=102)
    run_case(sa, oracle, case, what="P=%d %s" % (page_size, layout))


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_contiguous_no_table(sa, oracle, kv_dtype):
    case = W.make_decode_case([256, 3, 64], page_size=256, paged=False, kv_dtype=kv_dtype, seed=103)
    run_case(sa, oracle, case, what="contiguous " + kv_dtype)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 4), (12, 2), (64, 8), (7, 1)])
def test_group_sizes(sa, oracle, hq, hkv):
    case = W.make_decode_case([17, 290], num_qo_heads=hq, num_kv_heads=hkv, page_size=16, seed=104)
    run_case(sa, oracle, case, what="Hq=%d Hkv=%d" % (hq, hkv))


def test_no_sinks(sa, oracle):
    case = W.make_decode_case([0, 33, 500], page_size=16, sinks=False, seed=105)
    out, lse = run_case(sa, oracle, case, what="no sink")
    assert torch.all(out[0].float() == 0) and torch.all(torch.isneginf(lse[0]))


def test_empty_sequences_give_sink_only(sa, oracle):
    case = W.make_decode_case([0, 0], page_size=16, seed=106)
    out, lse = run_case(sa, oracle, case, what="empty")
    assert torch.all(out.float() == 0)
    assert torch.allclose(lse.cpu(), case.sinks[None].expand(2, -1), atol=1e-6)


def test_huge_sink_and_extreme_scores(sa, oracle):
    case = W.make_decode_case([50, 400], page_size=16, seed=107)
    case.sinks = torch.full((64,), 1e4, dtype=torch.float32)
    run_case(sa, oracle, case, what="sink 1e4")
    case = W.make_decode_case([50, 400], page_size=16, seed=108, sm_scale=2.0)  # peaked softmax
    run_case(sa, oracle, case, what="scale 2")


def test_partial_then_merge_equals_decode(sa, oracle):
    case = W.make_decode_case([3, 200, 1500], page_size=16, window=0, seed=109).to("cuda")
    B, Hq, D = case.q.shape
    S, maxlen = 5, 1500
    o_part = torch.empty(S, B, Hq, D, device="cuda")
    l_part = torch.empty(S, B, Hq, device="cuda")
    sa.sa_decode_partial(case.q, case.kv, case.seqlens, 0, case.sm_scale, S, o_part, l_part, max_kv_len=maxlen)
    out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, Hq, device="cuda")
    sa.sa_merge_states(o_part, l_part, case.sinks, out, lse)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle_decode(oracle, case.to("cpu"))
    check_close(out, lse, ref_o, ref_l, "partial+merge")
    # each partial is the sink-free state of its chunk: keys [chunk*s, chunk*(s+1))
    rows = oracle.decode_rows(case.seqlens.cpu())
    tiles = (maxlen + 15) // 16
    chunk = 16 * ((tiles + S - 1) // S)
    kv_cpu = case.kv.to("cpu").as_dict()
    for s in range(S):
        ro, rl = oracle.attend(case.q.cpu(), rows[0], rows[1], kv_cpu, case.seqlens.cpu(), None, 0,
                               case.sm_scale, key_range=(chunk * s, chunk * (s + 1)))
        check_close(o_part[s], l_part[s], ro.reshape(B, Hq, D), rl.reshape(B, Hq), "partial chunk %d" % s)


def test_merge_kernel_against_oracle(sa, oracle):
    g = torch.Generator().manual_seed(5)
    S, N, H, D = 9, 33, 64, 64
    o = torch.randn(S, N, H, D, generator=g)
    l = torch.randn(S, N, H, generator=g) * 5
    l[2] = -math.inf
    l[:, 0, 0] = -math.inf  # a row with nothing but the sink
    sinks = torch.empty(H).uniform_(-2, 6, generator=g)
    for sk in (sinks, None):
        out = torch.empty(N, H, D, dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(N, H, device="cuda")
        sa.sa_merge_states(o.cuda(), l.cuda(), None if sk is None else sk.cuda(), out, lse)
        torch.cuda.synchronize()
        ref_o, ref_l = oracle.merge(o.double(), l.double(), sk)
        check_close(out, lse, ref_o, ref_l, "merge sinks=%s" % (sk is not None))


@pytest.mark.parametrize("window", [0, 128])
def test_bit_exact_index_and_mask_probe(sa, window):
    """One key carries score 40 against 0 for all others: the output must be
    that key's value row bit for bit when the key is visible, and must not be
    when it is not.  Targets sweep page starts/ends, the window edge and the
    last key; value rows encode (sequence, key) so a wrong page or slot shows."""
    L = [300, 517]
    case = W.make_decode_case(L, num_qo_heads=8, num_kv_heads=8, page_size=16, window=window, sinks=False,
                              poison_pages=4, seed=110)
    kv = case.kv
    P = 16
    for b, Lb in enumerate(L):
        for t in range(Lb):
            pg, sl = int(kv.page_table[b, t // P]), t % P
            kv.k[pg, :, sl] = 0
            d = torch.arange(64, dtype=torch.float32)
            row = 1 + (d % 7)
            row[0], row[1], row[2] = 1 + (t & 255), 1 + (t >> 8), 1 + b
            kv.v[pg, :, sl] = row.to(torch.bfloat16)
    case.q.zero_()
    case.q[:, :, 0] = 16.0
    targets = {0, 15, 16, 17, 31, 32}
    for Lb in L:
        targets |= {Lb - 1, Lb - 16, Lb - 17, Lb - 127, Lb - 128, Lb - 129}
    cuda_case = case.to("cuda")
    for t in sorted(targets):
        for b, Lb in enumerate(L):
            if not 0 <= t < Lb:
                continue
            pg, sl = int(kv.page_table[b, t // P]), t % P
            cuda_case.kv.k[pg, :, sl, 0] = 20.0  # score 16*20/8 = 40
        out, lse = decode_gpu(sa, cuda_case, num_splits=0)
        for b, Lb in enumerate(L):
            if not 0 <= t < Lb:
                continue
            pg, sl = int(kv.page_table[b, t // P]), t % P
            vrow = cuda_case.kv.v[pg, 0, sl]
            visible = window == 0 or t > Lb - 1 - window
            same = torch.equal(out[b, 0], vrow)
            assert same == visible, (b, t, visible)
            cuda_case.kv.k[pg, :, sl, 0] = 0.0


def test_device_status_flags(sa):
    case = W.make_decode_case([40, 70], page_size=16, seed=111).to("cuda")
    out, lse = decode_gpu(sa, case, num_splits=1, max_kv_len=50)   # seqlen 70 > max_kv_len
    assert sa.sa_device_status() & sa.SA_DEVICE_SEQLEN_RANGE
    bad = case.kv.page_table.clone()
    bad[1, 0] = case.kv.num_pages + 5                              # a page outside the pool
    kv = W.KVCache(case.kv.k, case.kv.v, "bf16", bad, 16)
    c2 = W.Case(case.q, kv, case.seqlens, case.sinks, 0, case.sm_scale)
    decode_gpu(sa, c2, num_splits=1)
    assert sa.sa_device_status() & sa.SA_DEVICE_BAD_PAGE
    assert sa.sa_device_status() == 0  # cleared by the read


def test_cuda_graph_capture_and_replay(sa, oracle):
    case = W.make_decode_case([100, 900, 2000], page_size=16, seed=112)
    cg = case.to("cuda")
    B, Hq, D = cg.q.shape
    out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, Hq, device="cuda")
    S = 4
    ws = torch.empty(sa.sa_decode_workspace_size(B, Hq, 8, D, 2000, 0, S), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        sa.sa_decode(cg.q, cg.kv, cg.seqlens, cg.sinks, 0, cg.sm_scale, out, lse, max_kv_len=2000, workspace=ws,
                     num_splits=S)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        sa.sa_decode(cg.q, cg.kv, cg.seqlens, cg.sinks, 0, cg.sm_scale, out, lse, max_kv_len=2000, workspace=ws,
                     num_splits=S)
    out.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    ref_o, ref_l = oracle_decode(oracle, case)
    check_close(out, lse, ref_o, ref_l, "graph replay")


def test_batch_zero(sa):
    q = torch.empty(0, 64, 64, dtype=torch.bfloat16, device="cuda")
    case = W.make_decode_case([5], page_size=16, seed=1).to("cuda")
    out = torch.empty(0, 64, 64, dtype=torch.bfloat16, device="cuda")
    sa.sa_decode(q, case.kv, case.seqlens[:0], case.sinks, 0, 0.125, out, None, max_kv_len=0)


