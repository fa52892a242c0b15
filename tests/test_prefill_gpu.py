"""GPU parity of sa_prefill (tcgen05 / TMEM / TMA) against the fp64 oracle:
single and ragged sequences, bottom-right-aligned causal masks, 128-token and
odd windows, paged and contiguous caches, both GQA pairings, with every row
(or, at 8192 tokens, a seeded sample of rows) compared elementwise."""
import numpy as np
import pytest
import torch

import workloads as W
from sa_testlib import check_close, oracle_prefill, prefill_gpu

pytestmark = pytest.mark.gpu


def run(sa, oracle, case, what, sel=None):
    out, lse = prefill_gpu(sa, case.to("cuda"))
    if sel is None:
        ref_o, ref_l = oracle_prefill(oracle, case)
        check_close(out, lse, ref_o, ref_l, what)
    else:
        ref_o, ref_l = oracle_prefill(oracle, case, sel)
        check_close(out[sel], lse[sel], ref_o, ref_l, what)
    assert sa.sa_device_status() == 0
    return out, lse


@pytest.mark.parametrize("T", [1, 2, 100, 128, 129, 255, 256, 300, 700])
@pytest.mark.parametrize("window", [0, 128])
def test_single_sequence(sa, oracle, T, window):
    case = W.make_prefill_case([T], [T], window=window, seed=200 + T)
    run(sa, oracle, case, "T=%d w=%d" % (T, window))


@pytest.mark.parametrize("window", [0, 1, 37, 128, 200])
def test_windows(sa, oracle, window):
    case = W.make_prefill_case([400], [400], window=window, seed=210)
    run(sa, oracle, case, "w=%d" % window)


def test_no_sinks(sa, oracle):
    case = W.make_prefill_case([333], [333], sinks=False, seed=211)
    run(sa, oracle, case, "no sink")


@pytest.mark.parametrize("window", [0, 128])
def test_ragged_batch_bottom_right(sa, oracle, window):
    # L_q < L_kv: queries are the last L_q positions of each sequence
    case = W.make_prefill_case([5, 130, 1, 257, 64], [9, 300, 70, 257, 1000], window=window, seed=212)
    run(sa, oracle, case, "ragged w=%d" % window)


@pytest.mark.parametrize("layout", ["HND", "NHD"])
@pytest.mark.parametrize("window", [0, 128])
def test_paged_cache(sa, oracle, layout, window):
    case = W.make_prefill_case([200, 77], [520, 77], paged=True, page_size=16, layout=layout, window=window,
                               poison_pages=5, seed=213)
    run(sa, oracle, case, "paged %s w=%d" % (layout, window))


@pytest.mark.parametrize("hq,hkv", [(8, 8), (6, 2), (16, 2), (64, 8)])
def test_group_pairings(sa, oracle, hq, hkv):
    case = W.make_prefill_case([150], [150], num_qo_heads=hq, num_kv_heads=hkv, seed=214)
    run(sa, oracle, case, "Hq=%d Hkv=%d" % (hq, hkv))


def test_peaked_scores(sa, oracle):
    case = W.make_prefill_case([300], [300], sm_scale=1.5, seed=215)  # forces rescales of O
    run(sa, oracle, case, "scale 1.5")


@pytest.mark.parametrize("window", [0, 128])
def test_config3_full_size_sampled_rows(sa, oracle, window):
    """One 8192-token sequence (64 q / 8 kv heads): every output of a seeded
    sample of rows, covering each 128-row tile's first and last row."""
    case = W.make_config(3, window=window)
    g = np.random.default_rng(33)
    sel = np.unique(np.concatenate([np.arange(0, 8192, 128), np.arange(127, 8192, 128),
                                    g.choice(8192, 128, replace=False)])).astype(np.int32)
    run(sa, oracle, case, "config 3 w=%d" % window, sel=sel)


# ---- FP8-E4M3 cache: codes widened exactly, products in f16 ---------------
@pytest.mark.parametrize("T", [1, 63, 129, 700])
@pytest.mark.parametrize("window", [0, 128])
def test_fp8_single_sequence(sa, oracle, T, window):
    case = W.make_prefill_case([T], [T], window=window, kv_dtype="e4m3", seed=300 + T)
    run(sa, oracle, case, "fp8 T=%d w=%d" % (T, window))


@pytest.mark.parametrize("layout", ["HND", "NHD"])
@pytest.mark.parametrize("window", [0, 128])
def test_fp8_paged_ragged(sa, oracle, layout, window):
    # chunked prefill on a paged FP8 cache: L_q < L_kv, sequence ends inside tiles
    case = W.make_prefill_case([200, 77, 5, 130], [520, 77, 1000, 131], paged=True, page_size=16, layout=layout,
                               window=window, kv_dtype="e4m3", poison_pages=5, seed=310)
    run(sa, oracle, case, "fp8 paged %s w=%d" % (layout, window))


@pytest.mark.parametrize("hq,hkv", [(8, 8), (6, 2)])
def test_fp8_group_pairings(sa, oracle, hq, hkv):
    case = W.make_prefill_case([150], [150], num_qo_heads=hq, num_kv_heads=hkv, kv_dtype="e4m3", seed=311)
    run(sa, oracle, case, "fp8 Hq=%d Hkv=%d" % (hq, hkv))


def test_fp8_peaked_scores_no_sinks(sa, oracle):
    case = W.make_prefill_case([300], [300], sm_scale=1.5, sinks=False, kv_dtype="e4m3", seed=312)
    run(sa, oracle, case, "fp8 scale 1.5, no sink")


# ---- E4M3 queries on an FP8 cache (sa_prefill_q8: kind::f8f6f4 for Q K^T) ----
def quantise_q(case):
    """E4M3 codes of the case's q with a per-tensor scale amax / 448 (torch's
    round-to-nearest-even cast), and that scale."""
    q = case.q.float()
    scale = float(q.abs().max()) / 448.0
    codes = (q / scale).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale


def run_q8(sa, oracle, case, what, sel=None):
    codes, q_scale = quantise_q(case)
    g = case.to("cuda")
    T, Hq, D = case.q.shape
    out = torch.full((T, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((T, Hq), float("nan"), dtype=torch.float32, device="cuda")
    cu = case.cu_seqlens_q
    qlens = (cu[1:] - cu[:-1])
    sa.sa_prefill_q8(codes.cuda(), q_scale, g.cu_seqlens_q, g.kv, g.seqlens, g.sinks, case.window, case.sm_scale,
                     out, lse, max_q_len=int(qlens.max()), max_kv_len=int(case.seqlens.max()))
    torch.cuda.synchronize()
    assert sa.sa_device_status() == 0
    rows = oracle.prefill_rows(case.cu_seqlens_q, case.seqlens)
    if sel is None:
        sel = np.arange(T, dtype=np.int32)
    sr = np.repeat(sel, Hq)
    sh = np.tile(np.arange(Hq, dtype=np.int32), len(sel))
    ref_o, ref_l = oracle.attend(codes, rows[0], rows[1], case.kv.as_dict(), case.seqlens, case.sinks, case.window,
                                 case.sm_scale, sr, sh, q_scale=q_scale)
    check_close(out[sel], lse[sel], ref_o.reshape(len(sel), Hq, D), ref_l.reshape(len(sel), Hq), what)


@pytest.mark.parametrize("T", [1, 63, 129, 700])
@pytest.mark.parametrize("window", [0, 128])
def test_q8_single_sequence(sa, oracle, T, window):
    case = W.make_prefill_case([T], [T], window=window, kv_dtype="e4m3", seed=320 + T)
    run_q8(sa, oracle, case, "q8 T=%d w=%d" % (T, window))


@pytest.mark.parametrize("layout", ["HND", "NHD"])
@pytest.mark.parametrize("window", [0, 128])
def test_q8_paged_ragged(sa, oracle, layout, window):
    case = W.make_prefill_case([200, 77, 5, 130], [520, 77, 1000, 131], paged=True, page_size=16, layout=layout,
                               window=window, kv_dtype="e4m3", poison_pages=5, seed=330)
    run_q8(sa, oracle, case, "q8 paged %s w=%d" % (layout, window))


@pytest.mark.parametrize("hq,hkv", [(8, 8), (6, 2)])
def test_q8_group_pairings(sa, oracle, hq, hkv):
    case = W.make_prefill_case([150], [150], num_qo_heads=hq, num_kv_heads=hkv, kv_dtype="e4m3", seed=331)
    run_q8(sa, oracle, case, "q8 Hq=%d Hkv=%d" % (hq, hkv))


def test_q8_peaked_scores_no_sinks(sa, oracle):
    case = W.make_prefill_case([300], [300], sm_scale=1.5, sinks=False, kv_dtype="e4m3", seed=332)
    run_q8(sa, oracle, case, "q8 scale 1.5, no sink")


def test_q8_config7_full_size(sa, oracle):
    case = W.make_config(7, window=0)
    g = np.random.default_rng(97)
    sel = np.unique(np.concatenate([np.arange(0, 8192, 1024), np.arange(1023, 8192, 1024),
                                    g.choice(8192, 40, replace=False)])).astype(np.int32)
    run_q8(sa, oracle, case, "q8 config 7", sel=sel)


@pytest.mark.parametrize("mode", ["bf16", "e4m3", "q8"])
@pytest.mark.parametrize("window", [0, 128])
def test_one_head_per_block_long_ragged(sa, oracle, mode, window):
    """Odd GQA groups run one head per block (128 softmax threads, which then
    widen an FP8 tile in two 16-byte chunks each).  Sequences long enough for
    the staging slots and the K/V ring to wrap several times, ragged and paged."""
    kv_dtype = "bf16" if mode == "bf16" else "e4m3"
    case = W.make_prefill_case([700, 37, 300], [1000, 37, 1029], num_qo_heads=6, num_kv_heads=2, paged=True,
                               page_size=16, layout="HND", window=window, kv_dtype=kv_dtype, poison_pages=4,
                               seed=340 + window)
    what = "one head per block, %s, w=%d" % (mode, window)
    if mode == "q8":
        run_q8(sa, oracle, case, what)
    else:
        run(sa, oracle, case, what)
