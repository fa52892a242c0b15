"""GPU parity of sa_decode_multi (q_len new tokens per sequence, token k at
position L - q_len + k) against the fp64 oracle, which evaluates the same rows
as a bottom-right-aligned ragged prefill: every output of every row."""
import numpy as np
import pytest
import torch

import workloads as W
from sa_testlib import check_close, oracle_prefill

pytestmark = pytest.mark.gpu


def multi_gpu(sa, case_gpu, q_len, num_splits=0):
    R, Hq, D = case_gpu.q.shape
    B = case_gpu.seqlens.shape[0]
    max_kv = int(case_gpu.seqlens.max().item())
    kv = case_gpu.kv
    out = torch.full((R, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((R, Hq), float("nan"), dtype=torch.float32, device="cuda")
    ws_bytes = sa.sa_decode_multi_workspace_size(B, q_len, Hq, kv.num_kv_heads, D, max_kv, case_gpu.window,
                                                 num_splits)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    sa.sa_decode_multi(case_gpu.q, q_len, kv, case_gpu.seqlens, case_gpu.sinks, case_gpu.window, case_gpu.sm_scale,
                       out, lse, max_kv_len=max_kv, workspace=ws, num_splits=num_splits)
    torch.cuda.synchronize()
    return out, lse


def case_of(q_len, kv_lens, seed, **kw):
    kw.setdefault("paged", True)
    kw.setdefault("page_size", 16)
    kw.setdefault("layout", "HND")
    return W.make_prefill_case([q_len] * len(kv_lens), kv_lens, seed=seed, **kw)


def run(sa, oracle, case, q_len, what, num_splits=0):
    out, lse = multi_gpu(sa, case.to("cuda"), q_len, num_splits)
    ref_o, ref_l = oracle_prefill(oracle, case)
    check_close(out, lse, ref_o, ref_l, what)
    assert sa.sa_device_status() == 0


LENS = [8, 9, 17, 100, 301, 1000, 2049]


@pytest.mark.parametrize("q_len", [1, 2, 3, 4, 5, 7, 8])
@pytest.mark.parametrize("window", [0, 128])
@pytest.mark.parametrize("splits", [1, 0, 3])
def test_tokens_windows_splits(sa, oracle, q_len, window, splits):
    case = case_of(q_len, LENS, seed=400 + q_len, window=window, poison_pages=7)
    run(sa, oracle, case, q_len, "q_len=%d w=%d S=%d" % (q_len, window, splits), splits)


@pytest.mark.parametrize("q_len", [2, 4, 8])
def test_tile_counts_one_to_six(sa, oracle, q_len):
    """Unsplit blocks of 1 to 6 key tiles of 64, whole or with a partial last
    tile: every shape of the MMA warp's round schedule (the steady rounds, the
    two closing rounds without a next Q K^T, the last tile's zeroed rows past
    the sequence, which the poisoned pages would otherwise turn into NaN)."""
    lens = [64, 65, 128, 129, 192, 193, 256, 257, 320, 383]
    case = case_of(q_len, lens, seed=430 + q_len, poison_pages=9)
    run(sa, oracle, case, q_len, "q_len=%d tiles 1-6" % q_len, num_splits=1)


@pytest.mark.parametrize("q_len", [2, 4, 8])
@pytest.mark.parametrize("window", [1, 37])
def test_small_windows(sa, oracle, q_len, window):
    # windows shorter than the token span: each token sees its own slice
    case = case_of(q_len, [8, 40, 333], seed=420, window=window)
    run(sa, oracle, case, q_len, "q_len=%d w=%d" % (q_len, window))


@pytest.mark.parametrize("q_len", [4, 8])
@pytest.mark.parametrize("window", [0, 128])
def test_fp8_cache(sa, oracle, q_len, window):
    case = case_of(q_len, LENS, seed=430, window=window, kv_dtype="e4m3", poison_pages=3)
    run(sa, oracle, case, q_len, "fp8 q_len=%d w=%d" % (q_len, window), 0)


@pytest.mark.parametrize("hq,hkv", [(6, 2), (8, 8), (64, 8)])
@pytest.mark.parametrize("q_len", [3, 6])
def test_group_pairings(sa, oracle, hq, hkv, q_len):
    case = case_of(q_len, [50, 500], seed=440, num_qo_heads=hq, num_kv_heads=hkv, layout="NHD")
    run(sa, oracle, case, q_len, "Hq=%d Hkv=%d q_len=%d" % (hq, hkv, q_len))


def test_no_sinks_contiguous(sa, oracle):
    case = W.make_prefill_case([4, 4, 4], [4, 250, 129], sinks=False, seed=450)
    run(sa, oracle, case, 4, "no sink, contiguous")


def test_q_len_one_is_sa_decode(sa):
    """q_len = 1 runs the decode kernel exactly as sa_decode does: bitwise equal."""
    from sa_testlib import decode_gpu
    case = W.make_config(2, window=0, device="cuda")
    out_m, lse_m = multi_gpu(sa, case, 1)
    out_d, lse_d = decode_gpu(sa, case)
    assert torch.equal(out_m, out_d) and torch.equal(lse_m, lse_d)


def test_too_short_sequence_is_flagged(sa, oracle):
    """A sequence holding fewer keys than q_len: its tokens at negative
    positions see no key (out 0, lse = sink), the status word says so, and
    the other sequence's rows are unaffected."""
    case = case_of(4, [600, 4], seed=460)
    g = case.to("cuda")
    g.seqlens[1] = 2  # tokens 0, 1 of sequence 1 now sit at positions -2, -1
    out, lse = multi_gpu(sa, g, 4)
    assert sa.sa_device_status() & 0x8  # SA_DEVICE_BAD_QLEN
    ref_o, ref_l = oracle_prefill(oracle, case)
    check_close(out[:4], lse[:4], ref_o[:4], ref_l[:4], "sequence 0")
    assert torch.all(out[4:6].float() == 0)
    torch.testing.assert_close(lse[4:6].cpu(), case.sinks.unsqueeze(0).expand(2, -1).float(), atol=1e-5, rtol=0)
    # seqlens = 0 is an empty slot: every token gives out 0, lse = sink, unflagged
    g.seqlens[1] = 0
    out, lse = multi_gpu(sa, g, 4)
    assert sa.sa_device_status() == 0
    check_close(out[:4], lse[:4], ref_o[:4], ref_l[:4], "sequence 0")
    assert torch.all(out[4:].float() == 0)
    torch.testing.assert_close(lse[4:].cpu(), case.sinks.unsqueeze(0).expand(4, -1).float(), atol=1e-5, rtol=0)


@pytest.mark.parametrize("window", [0, 128])
def test_config8_full_size(sa, oracle, window):
    """B=64 sequences of L ~ U[1024, 8192] (paged), 4 draft tokens each:
    every output of 6 sampled sequences."""
    case = W.make_config(8, window=window)
    out, lse = multi_gpu(sa, case.to("cuda"), 4)
    assert sa.sa_device_status() == 0
    seqs = sorted(np.random.default_rng(88).choice(64, 6, replace=False).tolist())
    rows = np.concatenate([np.arange(4 * s, 4 * s + 4) for s in seqs]).astype(np.int32)
    ref_o, ref_l = oracle_prefill(oracle, case, rows)
    check_close(out[rows], lse[rows], ref_o, ref_l, "config 8 w=%d" % window)


@pytest.mark.parametrize("splits", [1, 3])
def test_cuda_graph_capture_and_replay(sa, oracle, splits):
    """The tcgen05 multi-token call (its Q tensor map encoded per call, held by
    value in the launch) captured into a CUDA graph and replayed after the
    output was overwritten; split and unsplit (longest-first) forms."""
    q_len = 4
    case = case_of(q_len, [100, 900, 2000, 37], seed=460)
    cg = case.to("cuda")
    R, Hq, D = cg.q.shape
    B = cg.seqlens.shape[0]
    out = torch.empty(R, Hq, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(R, Hq, device="cuda")
    ws = torch.empty(max(sa.sa_decode_multi_workspace_size(B, q_len, Hq, 8, D, 2000, 0, splits), 16),
                     dtype=torch.uint8, device="cuda")
    run = lambda: sa.sa_decode_multi(cg.q, q_len, cg.kv, cg.seqlens, cg.sinks, 0, cg.sm_scale, out, lse,
                                     max_kv_len=2000, workspace=ws, num_splits=splits)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        run()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run()
    out.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    ref_o, ref_l = oracle_prefill(oracle, case)
    check_close(out, lse, ref_o, ref_l, "multi-token graph replay S=%d" % splits)
    assert sa.sa_device_status() == 0
