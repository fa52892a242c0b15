"""Host side of the rotary step: the library's YaRN table (built on the host
in double precision) against the oracle's frequencies, and argument checks of
sa_rope_yarn_table / sa_rope_append that return before any launch."""
import ctypes

import numpy as np
import pytest

from oracle import rope as R

YARN = dict(theta=150000.0, factor=32.0, original_max_position=4096, beta_fast=32.0, beta_slow=1.0)


@pytest.fixture(scope="module")
def sa():
    import gqa_attention_sinks_head_gb300 as lib
    lib.build()
    lib.load()
    return lib


@pytest.mark.parametrize("yarn", [YARN, dict(theta=10000.0, factor=1.0, original_max_position=2048,
                                             beta_fast=32.0, beta_slow=1.0),
                                  dict(theta=500000.0, factor=8.0, original_max_position=8192, beta_fast=16.0,
                                       beta_slow=2.0)])
def test_table_matches_oracle(sa, yarn):
    n = 140000
    t = sa.sa_rope_yarn_table(n, **yarn).double().numpy()
    f, ms = R.yarn_inv_freq(64, **yarn)
    p = np.arange(n, dtype=np.float64)[:, None]
    assert np.allclose(t[:, :32], np.cos(p * f) * ms, rtol=0, atol=1e-6 * ms)
    assert np.allclose(t[:, 32:], np.sin(p * f) * ms, rtol=0, atol=1e-6 * ms)


def test_table_argument_checks(sa):
    L = sa.load()
    buf = (ctypes.c_float * 64)()
    assert L.sa_rope_yarn_table(None, 1, 64, 1e4, 1.0, 4096, 32.0, 1.0) == 1
    assert L.sa_rope_yarn_table(buf, 0, 64, 1e4, 1.0, 4096, 32.0, 1.0) == 1
    assert L.sa_rope_yarn_table(buf, 1, 128, 1e4, 1.0, 4096, 32.0, 1.0) == 2
    assert L.sa_rope_yarn_table(buf, 1, 64, 1.0, 1.0, 4096, 32.0, 1.0) == 1
    assert L.sa_rope_yarn_table(buf, 1, 64, 1e4, float("nan"), 4096, 32.0, 1.0) == 1
    assert L.sa_rope_yarn_table(buf, 1, 64, 1e4, 4.0, 4096, 0.0, 1.0) == 1
    assert L.sa_rope_yarn_table(buf, 1, 64, 1e4, 4.0, 4096, 32.0, 1.0) == 0
    assert buf[0] == pytest.approx(0.1 * np.log(4.0) + 1.0)  # position 0: cos 0 * mscale


def test_append_argument_checks(sa):
    L = sa.load()
    d = sa.KVDesc()
    d.k, d.v, d.dtype, d.num_pages, d.num_kv_heads, d.head_dim, d.page_size = 4096, 8192, 0, 10, 8, 64, 16
    d.page_table_stride, d.stride_page, d.stride_head, d.stride_token = 4, 8 * 16 * 64, 16 * 64, 64
    d.page_table, d.k_scale, d.v_scale = 1024, 1.0, 1.0
    args = lambda **kw: [kw.get("q", 4096), 4096, 4096, kw.get("T", 3), kw.get("hq", 64), 4096, 4096,
                         kw.get("table", 4096), kw.get("maxpos", 100), ctypes.byref(d), kw.get("batch", 2),
                         kw.get("qo", 4096), kw.get("qs", 0.0), None]
    assert L.sa_rope_append(*args(T=0)) == 0
    assert L.sa_rope_append(*args(T=-1)) == 1
    assert L.sa_rope_append(*args(maxpos=0)) == 1
    assert L.sa_rope_append(*args(hq=60)) == 1
    assert L.sa_rope_append(*args(q=None)) == 1
    assert L.sa_rope_append(*args(q=4100)) == 2
    assert L.sa_rope_append(*args(table=4104)) == 2
    assert L.sa_rope_append(*args(qs=-1.0)) == 1
    assert L.sa_rope_append(*args(qs=float("inf"))) == 1
