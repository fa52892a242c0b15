"""A seeded random sweep over the shape space that the fixed tests cover one
axis at a time: batch, ragged lengths (0, 1, page edges), windows, page sizes,
cache layouts and dtypes, GQA groups, splits and query lengths, drawn together.
Every output of every case is compared with the fp64 oracle."""
import numpy as np
import pytest

import workloads as W
from sa_testlib import check_close, decode_gpu, oracle_decode, oracle_prefill, prefill_gpu
from test_decode_multi_gpu import multi_gpu

pytestmark = pytest.mark.gpu

GROUPS = [(64, 8), (8, 8), (6, 2), (16, 2), (32, 4)]  # (q heads, kv heads): 1 to 8 q heads per kv head


def _draw(seed):
    g = np.random.default_rng(seed)
    hq, hkv = GROUPS[int(g.integers(len(GROUPS)))]
    page = int(g.choice([16, 32, 64]))
    layout = str(g.choice(["HND", "NHD"]))
    kv_dtype = str(g.choice(["bf16", "e4m3"]))
    window = int(g.choice([0, 0, 128, 1, 37, 300]))
    return g, hq, hkv, page, layout, kv_dtype, window


@pytest.mark.parametrize("seed", range(12))
def test_random_decode(sa, oracle, seed):
    g, hq, hkv, page, layout, kv_dtype, window = _draw(1000 + seed)
    lens = [int(x) for x in g.choice([0, 1, 2, 15, 16, 17, 100, 511, 512, 513, 1500, 3000], int(g.integers(1, 9)))]
    if max(lens) == 0:
        lens[0] = 5
    splits = int(g.choice([0, 1, 2, 5]))
    case = W.make_decode_case(lens, num_qo_heads=hq, num_kv_heads=hkv, page_size=page, layout=layout,
                              kv_dtype=kv_dtype, window=window, poison_pages=2, seed=2000 + seed)
    out, lse = decode_gpu(sa, case.to("cuda"), num_splits=splits)
    ref_o, ref_l = oracle_decode(oracle, case)
    check_close(out, lse, ref_o, ref_l, "random decode %d: %s %s w=%d P=%d Hq/Hkv=%d/%d S=%d lens=%s"
                % (seed, kv_dtype, layout, window, page, hq, hkv, splits, lens))
    assert sa.sa_device_status() == 0


@pytest.mark.parametrize("seed", range(8))
def test_random_multi_token_decode(sa, oracle, seed):
    g, hq, hkv, page, layout, kv_dtype, window = _draw(3000 + seed)
    q_len = int(g.integers(2, 9))
    lens = [int(x) for x in g.choice([q_len, q_len + 1, 100, 513, 2000], int(g.integers(1, 6)))]
    splits = int(g.choice([0, 1, 3]))
    case = W.make_prefill_case([q_len] * len(lens), lens, num_qo_heads=hq, num_kv_heads=hkv, paged=True,
                               page_size=page, layout=layout, kv_dtype=kv_dtype, window=window, poison_pages=2,
                               seed=4000 + seed)
    out, lse = multi_gpu(sa, case.to("cuda"), q_len, splits)
    ref_o, ref_l = oracle_prefill(oracle, case)
    check_close(out, lse, ref_o, ref_l, "random multi-token decode %d: q_len=%d %s %s w=%d P=%d Hq/Hkv=%d/%d S=%d "
                "lens=%s" % (seed, q_len, kv_dtype, layout, window, page, hq, hkv, splits, lens))
    assert sa.sa_device_status() == 0


@pytest.mark.parametrize("seed", range(8))
def test_random_multi_token_decode_bf16(sa, oracle, seed):
    """bf16 caches (the tensor-core multi-token kernel), batches up to past
    the 128 sequences that the unsplit call orders longest first."""
    g, hq, hkv, page, layout, _, window = _draw(8000 + seed)
    q_len = int(g.integers(2, 9))
    B = int(g.choice([1, 7, 64, 129]))
    lens = [int(x) for x in g.choice([q_len, q_len + 1, 64, 100, 513, 2000], B)]
    splits = int(g.choice([0, 1, 3]))
    case = W.make_prefill_case([q_len] * len(lens), lens, num_qo_heads=hq, num_kv_heads=hkv, paged=True,
                               page_size=page, layout=layout, window=window, poison_pages=2, seed=9000 + seed)
    out, lse = multi_gpu(sa, case.to("cuda"), q_len, splits)
    ref_o, ref_l = oracle_prefill(oracle, case)
    check_close(out, lse, ref_o, ref_l, "random bf16 multi-token decode %d: q_len=%d B=%d %s w=%d P=%d Hq/Hkv=%d/%d "
                "S=%d" % (seed, q_len, B, layout, window, page, hq, hkv, splits))
    assert sa.sa_device_status() == 0


@pytest.mark.parametrize("seed", range(8))
def test_random_prefill(sa, oracle, seed):
    g, hq, hkv, page, layout, kv_dtype, window = _draw(5000 + seed)
    kv_lens = [int(x) for x in g.choice([1, 64, 129, 300, 700], int(g.integers(1, 4)))]
    q_lens = [int(g.integers(1, L + 1)) for L in kv_lens]
    paged = bool(g.integers(2))
    kw = dict(paged=True, page_size=page, layout=layout, poison_pages=2) if paged else {}
    case = W.make_prefill_case(q_lens, kv_lens, num_qo_heads=hq, num_kv_heads=hkv, kv_dtype=kv_dtype,
                               window=window, seed=6000 + seed, **kw)
    out, lse = prefill_gpu(sa, case.to("cuda"))
    ref_o, ref_l = oracle_prefill(oracle, case)
    check_close(out, lse, ref_o, ref_l, "random prefill %d: %s %s w=%d Hq/Hkv=%d/%d q=%s kv=%s paged=%s"
                % (seed, kv_dtype, layout if paged else "contiguous", window, hq, hkv, q_lens, kv_lens, paged))
    assert sa.sa_device_status() == 0


@pytest.mark.parametrize("seed", range(6))
def test_random_prefill_e4m3_queries(sa, oracle, seed):
    from test_prefill_gpu import run_q8
    g, hq, hkv, page, layout, _, window = _draw(7000 + seed)
    kv_lens = [int(x) for x in g.choice([1, 64, 129, 300, 700], int(g.integers(1, 4)))]
    q_lens = [int(g.integers(1, L + 1)) for L in kv_lens]
    case = W.make_prefill_case(q_lens, kv_lens, num_qo_heads=hq, num_kv_heads=hkv, kv_dtype="e4m3", paged=True,
                               page_size=page, layout=layout, window=window, poison_pages=2, seed=8000 + seed)
    run_q8(sa, oracle, case, "random E4M3-query prefill %d: %s w=%d P=%d Hq/Hkv=%d/%d q=%s kv=%s"
           % (seed, layout, window, page, hq, hkv, q_lens, kv_lens))


@pytest.mark.parametrize("seed", range(6))
def test_random_rope_append(sa, seed):
    from test_rope_gpu import assert_untouched, check, run_case
    g = np.random.default_rng(9000 + seed)
    hq, hkv = GROUPS[int(g.integers(len(GROUPS)))]
    seqlens = [int(x) for x in g.choice([1, 16, 17, 300, 1029], int(g.integers(1, 5)))]
    new = [int(g.integers(1, L + 1)) for L in seqlens]
    r = run_case(sa, seqlens, new, kv_dtype=str(g.choice(["bf16", "e4m3"])), layout=str(g.choice(["HND", "NHD"])),
                 hq=hq, hkv=hkv, seed=9100 + seed)
    assert r["flags"] == 0
    check(r)
    assert_untouched(r)
