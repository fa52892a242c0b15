"""GPU parity of sa_rope_append (YaRN rotary embedding of q and k + paged
cache write of k and v) against the fp64 oracle in oracle/rope.py: every
rotated query element, every written cache element, and bit-exact checks that
nothing else in the cache changed and that bad tokens are skipped and flagged."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import rope as R
from sa_testlib import OUT_ATOL, OUT_RTOL

pytestmark = pytest.mark.gpu

YARN = dict(theta=150000.0, factor=32.0, original_max_position=4096, beta_fast=32.0, beta_slow=1.0)
SA_DEVICE_BAD_PAGE = 0x2
SA_DEVICE_BAD_TOKEN = 0x10


def _cache_np(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16).copy() if t.dtype == torch.bfloat16 else \
        t.cpu().numpy().copy()


def _tokens(seqlens, new, seed):
    """The last `new[b]` positions of each sequence b, in sequence order."""
    seq, pos = [], []
    for b, (L, n) in enumerate(zip(seqlens, new)):
        for p in range(L - n, L):
            seq.append(b)
            pos.append(p)
    g = np.random.default_rng(seed)
    return np.array(seq, np.int32), np.array(pos, np.int32), g


def run_case(sa, seqlens, new, *, kv_dtype="bf16", layout="HND", paged=True, hq=64, hkv=8, yarn=YARN,
             max_position=None, seed=0, bad=None):
    kv = W.make_kv(seqlens, hkv, 64, 16 if paged else (max(seqlens) + 15) // 16 * 16, paged=paged, kv_dtype=kv_dtype,
                   poison_pages=3 if paged else 0, seed=seed, layout=layout)
    seq, pos, g = _tokens(seqlens, new, seed)
    if bad:
        seq, pos = bad(seq.copy(), pos.copy())
    T = len(seq)
    q = torch.from_numpy(g.standard_normal((T, hq, 64)).astype(np.float32)).to(torch.bfloat16)
    k = torch.from_numpy(g.standard_normal((T, hkv, 64)).astype(np.float32)).to(torch.bfloat16)
    v = torch.from_numpy(g.standard_normal((T, hkv, 64)).astype(np.float32)).to(torch.bfloat16)
    if max_position is None:
        max_position = max(seqlens) + 8
    table = sa.sa_rope_yarn_table(max_position, **yarn)

    # oracle on CPU copies of the cache
    d = kv.as_dict()
    ck, cv = _cache_np(kv.k), _cache_np(kv.v)
    cache = dict(k=ck, v=cv, dtype=kv_dtype, page_table=None if kv.page_table is None else kv.page_table.numpy(),
                 page_size=kv.page_size, stride_page=d["stride_page"], stride_head=d["stride_head"],
                 stride_token=d["stride_token"], k_scale=kv.k_scale, v_scale=kv.v_scale)
    valid = (pos >= 0) & (pos < max_position) & (seq >= 0) & (seq < len(seqlens))
    q_ref = R.rope_append(q.double().numpy()[valid], k.double().numpy()[valid], v.double().numpy()[valid],
                          seq[valid], pos[valid], yarn, cache)

    # library
    kvg = kv.to("cuda")
    q_out = torch.full_like(q, float("nan")).cuda()
    sa.sa_rope_append(q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(seq).cuda(), torch.from_numpy(pos).cuda(),
                      table.cuda(), kvg, len(seqlens), q_out)
    torch.cuda.synchronize()
    flags = sa.sa_device_status()
    return dict(q_out=q_out.cpu(), q_ref=q_ref, valid=valid, flags=flags, kv=kv, kvg=kvg, ck=ck, cv=cv,
                before_k=_cache_np(kv.k), before_v=_cache_np(kv.v), dtype=kv_dtype)


def check(r):
    qo = r["q_out"].double().numpy()[r["valid"]]
    err = np.abs(qo - r["q_ref"])
    assert (err <= OUT_ATOL + OUT_RTOL * np.abs(r["q_ref"])).all(), float(err.max())
    gk, gv = _cache_np(r["kvg"].k), _cache_np(r["kvg"].v)
    if r["dtype"] == "bf16":
        # The kernel rotates in fp32 with an fp32 table and rounds to bf16; the
        # oracle rounds its fp64 value once.  Apart from one ulp of rounding,
        # the fp32 products of a rotation (cos and sin times the two halves)
        # carry about 2^-24 of the row's magnitude each; where they nearly
        # cancel, that exceeds half an ulp of the small result.  Bound:
        # |got - want| <= ulp(want) + 2^-20 * max |row|.
        for got, want in [(gk, r["ck"]), (gv, r["cv"])]:
            diff = got != want  # raw bits: NaN poison compares equal to itself here
            if not diff.any():
                continue
            g64, w64 = _bf16_values(got), _bf16_values(want)
            rowmax = np.abs(np.where(np.isfinite(w64), w64, 0.0)).max(axis=-1, keepdims=True)
            ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(w64), 2.0 ** -126))) - 7)
            tol = ulp + 2.0 ** -20 * np.broadcast_to(rowmax, w64.shape)
            err = np.abs(g64 - w64)
            assert np.all(err[diff] <= tol[diff]), float((err[diff] / tol[diff]).max())
    else:
        for got, want in [(gk, r["ck"]), (gv, r["cv"])]:
            mism = got != want
            # fp32 (kernel) and fp64 (oracle) values differ by ~1e-7 relative: a
            # different code is allowed only as the neighbouring code, and rarely
            a, b = got[mism].astype(np.int64), want[mism].astype(np.int64)
            assert np.all((a & 0x80) == (b & 0x80)) and np.all(np.abs((a & 0x7F) - (b & 0x7F)) == 1)
            assert mism.sum() <= max(2, got.size // 100000), int(mism.sum())


def _bf16_values(bits):
    """fp64 values of bf16 bit patterns (uint16 array of any shape)."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def assert_untouched(r):
    """Slots the oracle did not write hold their old bytes (bit-exact)."""
    gk, gv = _cache_np(r["kvg"].k), _cache_np(r["kvg"].v)
    same_k = r["ck"] == r["before_k"]
    same_v = r["cv"] == r["before_v"]
    bk, bv = r["before_k"], r["before_v"]
    # NaN poison compares unequal to itself as a float, but these are raw bits
    assert np.array_equal(gk[same_k], bk[same_k])
    assert np.array_equal(gv[same_v], bv[same_v])


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("layout", ["HND", "NHD"])
def test_decode_step_append(sa, kv_dtype, layout):
    """One new token per sequence, at its last position (the decode step)."""
    r = run_case(sa, [1, 17, 300, 1024, 4097], [1, 1, 1, 1, 1], kv_dtype=kv_dtype, layout=layout, seed=500)
    assert r["flags"] == 0
    check(r)
    assert_untouched(r)


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_prefill_chunk_append(sa, kv_dtype):
    """Chunks of new tokens (a prefill chunk per sequence), ragged."""
    r = run_case(sa, [700, 129, 2000], [700, 64, 333], kv_dtype=kv_dtype, seed=501)
    assert r["flags"] == 0
    check(r)
    assert_untouched(r)


def test_contiguous_cache_and_group_pairing(sa):
    r = run_case(sa, [40, 90], [40, 5], paged=False, hq=6, hkv=2, seed=502)
    assert r["flags"] == 0
    check(r)
    assert_untouched(r)


def test_plain_rope_factor_one(sa):
    y = dict(theta=10000.0, factor=1.0, original_max_position=4096, beta_fast=32.0, beta_slow=1.0)
    r = run_case(sa, [300, 5], [300, 5], yarn=y, seed=503)
    assert r["flags"] == 0
    check(r)


def test_bad_tokens_are_skipped_and_flagged(sa):
    def bad(seq, pos):
        seq[3] = 7          # no such sequence
        pos[5] = 10 ** 6    # past max_position
        pos[6] = -1
        return seq, pos
    r = run_case(sa, [50, 60], [20, 20], bad=bad, seed=504)
    assert r["flags"] & SA_DEVICE_BAD_TOKEN
    check(r)
    assert_untouched(r)


def test_fp8_query_output(sa):
    """q_out as E4M3 codes of rotate(q) / q_out_scale: the oracle's encoder
    on the fp64 rotation, up to a neighbouring code at rounding midpoints."""
    seqlens, new = [300, 40], [300, 40]
    kv = W.make_kv(seqlens, 8, 64, 16, paged=True, kv_dtype="e4m3", seed=505, layout="HND")
    seq, pos, g = _tokens(seqlens, new, 505)
    T = len(seq)
    q = torch.from_numpy(g.standard_normal((T, 64, 64)).astype(np.float32)).to(torch.bfloat16)
    k = torch.from_numpy(g.standard_normal((T, 8, 64)).astype(np.float32)).to(torch.bfloat16)
    v = torch.from_numpy(g.standard_normal((T, 8, 64)).astype(np.float32)).to(torch.bfloat16)
    table = sa.sa_rope_yarn_table(512, **YARN)
    q_scale = 0.02
    q_codes = torch.zeros(T, 64, 64, dtype=torch.uint8, device="cuda")
    sa.sa_rope_append(q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(seq).cuda(), torch.from_numpy(pos).cuda(),
                      table.cuda(), kv.to("cuda"), 2, q_codes, q_out_scale=q_scale)
    torch.cuda.synchronize()
    assert sa.sa_device_status() == 0
    f, ms = R.yarn_inv_freq(64, **YARN)
    want = R.e4m3_encode(R.rope_rotate(q.double().numpy(), pos[:, None], f, ms) / q_scale)
    got = q_codes.cpu().numpy()
    mism = got != want
    a, b = got[mism].astype(np.int64), want[mism].astype(np.int64)
    assert np.all((a & 0x80) == (b & 0x80)) and np.all(np.abs((a & 0x7F) - (b & 0x7F)) == 1)
    assert mism.sum() <= 4, int(mism.sum())


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_workload9_full_size(sa, kv_dtype):
    """The launch the bench times (bf16 cache), and the same on an E4M3 cache:
    8192 new tokens of one sequence at positions 0..8191, 64 q / 8 kv heads,
    YaRN (theta 150000, factor 32, original 4096) into a paged HND cache.
    Every rotated query element and every cache element is checked."""
    r = run_case(sa, [8192], [8192], kv_dtype=kv_dtype, seed=506)
    assert r["flags"] == 0
    check(r)
    assert_untouched(r)
