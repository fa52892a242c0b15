"""Parity at the five workloads' full sizes, in the launch configuration the
benchmark uses (automatic split count).  Large caches are drawn on the device;
the oracle reads the same bytes copied back for a seeded sample of sequences
(every head of each), or every row where that is cheap."""
import numpy as np
import pytest
import torch

import workloads as W
from sa_testlib import check_close, decode_gpu, oracle_decode

pytestmark = pytest.mark.gpu


def _sampled(oracle, case_gpu, out, lse, seqs, what):
    sub = W.subset(case_gpu, seqs)
    ref_o, ref_l = oracle_decode(oracle, sub)
    check_close(out[seqs], lse[seqs], ref_o, ref_l, what)


def test_config1_decode_b1_l256(sa, oracle):
    case = W.make_config(1)
    out, lse = decode_gpu(sa, case.to("cuda"))
    ref_o, ref_l = oracle_decode(oracle, case)
    check_close(out, lse, ref_o, ref_l, "config 1")
    assert sa.sa_device_status() == 0


@pytest.mark.parametrize("window", [0, 128])
def test_config2_decode_b64_paged(sa, oracle, window):
    case = W.make_config(2, window=window)
    out, lse = decode_gpu(sa, case.to("cuda"))
    ref_o, ref_l = oracle_decode(oracle, case)
    check_close(out, lse, ref_o, ref_l, "config 2 w=%d" % window)
    assert sa.sa_device_status() == 0


def test_config4_decode_b128_l32768_split(sa, oracle):
    case = W.make_config(4, device="cuda")
    assert sa.sa_decode_num_splits(128, 8, 32768, 0) > 1  # the split-KV + merge path
    out, lse = decode_gpu(sa, case)
    assert sa.sa_device_status() == 0
    # 16 of the 128 sequences, every head of each: the split + merge path on each
    seqs = sorted(np.random.default_rng(44).choice(127, 15, replace=False).tolist() + [127])
    _sampled(oracle, case, out, lse, seqs, "config 4")


@pytest.mark.parametrize("window", [0, 128])
def test_config5_decode_fp8_b256(sa, oracle, window):
    case = W.make_config(5, window=window, device="cuda")
    out, lse = decode_gpu(sa, case)
    assert sa.sa_device_status() == 0
    if window:
        seqs = list(range(256))  # 128 keys per row: every row
    else:
        seqs = sorted(np.random.default_rng(55).choice(256, 6, replace=False).tolist())
    _sampled(oracle, case, out, lse, seqs, "config 5 w=%d" % window)


@pytest.mark.parametrize("window", [0, 128])
def test_config6_chunked_paged_prefill(sa, oracle, window):
    """Chunked prefill: 1024 new queries per sequence on paged contexts of
    2k-16k keys, bottom-right causal.  Every output of a seeded sample of rows
    (each sequence's first and last row and each 128-row tile's edges)."""
    from sa_testlib import oracle_prefill, prefill_gpu
    case = W.make_config(6, window=window)
    out, lse = prefill_gpu(sa, case.to("cuda"))
    assert sa.sa_device_status() == 0
    g = np.random.default_rng(66)
    edges = np.concatenate([np.arange(0, 8192, 128), np.arange(127, 8192, 128)])
    sel = np.unique(np.concatenate([edges[g.choice(len(edges), 48, replace=False)],
                                    np.arange(0, 8192, 1024), np.arange(1023, 8192, 1024),
                                    g.choice(8192, 32, replace=False)])).astype(np.int32)
    ref_o, ref_l = oracle_prefill(oracle, case, sel)
    check_close(out[sel], lse[sel], ref_o, ref_l, "config 6 w=%d" % window)


def test_config7_chunked_paged_prefill_fp8(sa, oracle):
    """Workload 6 on an FP8-E4M3 cache, window 0, sampled rows."""
    from sa_testlib import oracle_prefill, prefill_gpu
    case = W.make_config(7, window=0)
    out, lse = prefill_gpu(sa, case.to("cuda"))
    assert sa.sa_device_status() == 0
    g = np.random.default_rng(77)
    sel = np.unique(np.concatenate([np.arange(0, 8192, 1024), np.arange(1023, 8192, 1024),
                                    g.choice(8192, 48, replace=False)])).astype(np.int32)
    ref_o, ref_l = oracle_prefill(oracle, case, sel)
    check_close(out[sel], lse[sel], ref_o, ref_l, "config 7")


@pytest.mark.parametrize("window", [0, 128])
def test_long_context_128k(sa, oracle, window):
    """The model's 128k context: one decode query and a 64-query chunk at the
    end of a 131072-key paged cache (P=16, 8192 pages per sequence), every
    output compared.  Exercises large page tables, many split chunks and
    positions past 2^16."""
    from sa_testlib import oracle_prefill, prefill_gpu
    L = 131072
    case = W.make_decode_case([L, 5000], page_size=16, paged=True, window=window, seed=130, device="cuda")
    assert sa.sa_decode_num_splits(2, 8, L, window) >= (1 if window else 16)
    out, lse = decode_gpu(sa, case)
    assert sa.sa_device_status() == 0
    _sampled(oracle, case, out, lse, [0, 1], "decode 128k w=%d" % window)
    pcase = W.make_prefill_case([64], [L], paged=True, page_size=16, layout="HND", window=window, seed=131)
    pout, plse = prefill_gpu(sa, pcase.to("cuda"))
    assert sa.sa_device_status() == 0
    sel = np.array([0, 1, 31, 62, 63], dtype=np.int32)
    ref_o, ref_l = oracle_prefill(oracle, pcase, sel)
    check_close(pout[sel], plse[sel], ref_o, ref_l, "prefill chunk at 128k w=%d" % window)


def test_large_batch_of_short_sequences(sa, oracle):
    """5000 sequences of 0..40 keys (empty ones included), paged: a grid
    z-extent in the thousands and many empty slots; every output compared."""
    g = np.random.default_rng(132)
    lens = g.integers(0, 41, 5000).tolist()
    case = W.make_decode_case(lens, page_size=16, paged=True, poison_pages=7, seed=132)
    out, lse = decode_gpu(sa, case.to("cuda"))
    assert sa.sa_device_status() == 0
    ref_o, ref_l = oracle_decode(oracle, case)
    check_close(out, lse, ref_o, ref_l, "B=5000 short")
