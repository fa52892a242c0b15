"""Pins of the fp64 oracle against things other than itself (CPU only).

Each test fixes the oracle against an independent fact: a pure-Python brute
force on tiny inputs, the identity "sink attention = ordinary SDPA with one
extra key whose value is zero" evaluated by torch in fp64, closed forms, the
limits of the sink, split invariance, and torch's own decoding of every E4M3
code and every bf16 bit pattern.  The cases are chosen so that a dropped term
(the sink in the denominator), a wrong sign, a wrong GQA index, an off-by-one
in the window or a transposed operand each fail at least one test.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------- helpers
def logical_kv(case):
    """[B, Hkv, Lmax, D] fp64 K and V rebuilt from the pages with torch gathers."""
    kv = case.kv
    L = case.seqlens.tolist()
    B, Lmax = len(L), max(L + [1])
    Hkv, D, P = kv.num_kv_heads, kv.head_dim, kv.page_size
    t = torch.arange(Lmax)
    if kv.page_table is None:
        pages = torch.arange(B)[:, None].expand(B, Lmax)
    else:
        pages = kv.page_table.long()[:, (t // P).clamp(max=kv.page_table.shape[1] - 1)]
    slot = (t % P)[None, :].expand(B, Lmax)

    def dec(x, scale):
        if kv.dtype == "bf16":
            x = x.double()
        else:
            x = x.view(torch.float8_e4m3fn).double()
        return x * scale

    def gather(x, scale):
        xd = dec(x, scale)
        if kv.layout == "HND":
            out = xd[pages, :, slot, :]          # [B, Lmax, Hkv, D]
        else:
            out = xd[pages, slot, :, :]
        return out.permute(0, 2, 1, 3).contiguous()

    return gather(kv.k, kv.k_scale), gather(kv.v, kv.v_scale)


def sdpa_reference(case, rows_seq, rows_pos, with_sink=True):
    """torch fp64 SDPA with one extra key: q' = [q, 1], k_sink = [0, sigma/scale],
    v_sink = 0, the sink column exempt from the causal/window mask."""
    K, V = logical_kv(case)
    q = case.q.double()
    n, Hq, D = q.shape
    Hkv = K.shape[1]
    G = Hq // Hkv
    L = case.seqlens.tolist()
    w = case.window
    outs = torch.zeros(n, Hq, D, dtype=torch.float64)
    lses = torch.zeros(n, Hq, dtype=torch.float64)
    for r in range(n):
        b, p = int(rows_seq[r]), int(rows_pos[r])
        Lb = L[b]
        j = torch.arange(Lb)
        allow = (j <= p) & ((j > p - w) if w > 0 else torch.ones_like(j, dtype=torch.bool))
        for h in range(Hq):
            g = h // G
            kk = K[b, g, :Lb]
            vv = V[b, g, :Lb]
            sig = float(case.sinks[h]) if (with_sink and case.sinks is not None) else -math.inf
            qq = torch.cat([q[r, h], torch.ones(1, dtype=torch.float64)])
            kk2 = torch.cat([kk, torch.zeros(Lb, 1, dtype=torch.float64)], 1)
            vv2 = vv
            mask = allow.clone()
            if sig != -math.inf:
                ks = torch.zeros(1, D + 1, dtype=torch.float64)
                ks[0, D] = sig / case.sm_scale
                kk2 = torch.cat([kk2, ks], 0)
                vv2 = torch.cat([vv, torch.zeros(1, D, dtype=torch.float64)], 0)
                mask = torch.cat([mask, torch.ones(1, dtype=torch.bool)])
            if not bool(mask.any()):
                lses[r, h] = -math.inf
                continue
            o = torch.nn.functional.scaled_dot_product_attention(
                qq[None, None, None], kk2[None, None], vv2[None, None],
                attn_mask=mask[None, None, None], scale=case.sm_scale)
            outs[r, h] = o[0, 0, 0]
            logits = (kk2 @ qq) * case.sm_scale
            lses[r, h] = torch.logsumexp(logits[mask], 0)
    return outs, lses


def brute_force(q, K, V, sinks, pos, L, window, scale):
    """Hand-expanded sums in pure Python floats for one head of one row."""
    logits, vals = [], []
    for j in range(L):
        if j > pos or (window > 0 and j <= pos - window):
            continue
        s = 0.0
        for d in range(len(q)):
            s += q[d] * K[j][d]
        logits.append(s * scale)
        vals.append(V[j])
    row = logits + ([sinks] if sinks is not None else [])
    if not row:
        return [0.0] * len(q), -math.inf
    m = max(row)
    z = sum(math.exp(x - m) for x in row)
    out = [sum(math.exp(logits[i] - m) * vals[i][d] for i in range(len(vals))) / z for d in range(len(q))]
    return out, m + math.log(z)


def run_oracle(oracle, case, rows=None, split=None, sel=None):
    if rows is None:
        if case.cu_seqlens_q is None:
            rows = oracle.decode_rows(case.seqlens)
        else:
            rows = oracle.prefill_rows(case.cu_seqlens_q, case.seqlens)
    sr, sh = (None, None) if sel is None else sel
    out, lse = oracle.attend(case.q, rows[0], rows[1], case.kv.as_dict(), case.seqlens, case.sinks,
                             case.window, case.sm_scale, sr, sh, split=split)
    n, Hq, D = case.q.shape
    if sel is None:
        return out.reshape(n, Hq, D), lse.reshape(n, Hq), rows
    return out, lse, rows


# ------------------------------------------------------------- decoders
def test_e4m3_all_codes_match_torch(oracle):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    mine = oracle.e4m3_to_f64(codes)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).double().numpy()
    nan_m, nan_r = np.isnan(mine), np.isnan(ref)
    assert (nan_m == nan_r).all()
    assert nan_m.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(mine[~nan_m], ref[~nan_r])
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9


def test_bf16_all_patterns_match_torch(oracle):
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    mine = oracle.bf16_to_f64(bits)
    ref = bits.view(torch.bfloat16).double().numpy()
    nan_m, nan_r = np.isnan(mine), np.isnan(ref)
    assert (nan_m == nan_r).all()
    assert np.array_equal(mine[~nan_m], ref[~nan_r])


# ------------------------------------------------------------ brute force
@pytest.mark.parametrize("window", [0, 2, 3])
@pytest.mark.parametrize("with_sink", [True, False])
def test_brute_force_tiny(oracle, window, with_sink):
    # Hq=4, Hkv=2 (G=2), D=2, L<=5, page size 2 with a shuffled table
    case = W.make_decode_case([5, 1, 4], num_qo_heads=4, num_kv_heads=2, head_dim=2, page_size=2,
                              paged=True, window=window, sinks=with_sink, poison_pages=2, seed=7)
    # prefill-style rows: every position of every sequence is a query
    L = case.seqlens.tolist()
    rows_seq = np.concatenate([np.full(l, b, np.int32) for b, l in enumerate(L)])
    rows_pos = np.concatenate([np.arange(l, dtype=np.int32) for l in L])
    g = torch.Generator().manual_seed(3)
    q = torch.randn(len(rows_seq), 4, 2, generator=g).to(torch.bfloat16)
    case.q = q
    out, lse = oracle.attend(q, rows_seq, rows_pos, case.kv.as_dict(), case.seqlens, case.sinks,
                             window, case.sm_scale)
    K, V = logical_kv(case)
    qd = q.double()
    for i in range(len(rows_seq)):
        b, p = int(rows_seq[i]), int(rows_pos[i])
        for h in range(4):
            g_ = h // 2
            Kl = K[b, g_].tolist()
            Vl = V[b, g_].tolist()
            sig = float(case.sinks[h]) if with_sink else None
            o_ref, l_ref = brute_force(qd[i, h].tolist(), Kl, Vl, sig, p, L[b], window, case.sm_scale)
            k = i * 4 + h
            assert np.allclose(out[k], o_ref, rtol=0, atol=1e-13)
            assert (lse[k] == l_ref) or abs(lse[k] - l_ref) < 1e-13


# ----------------------------------------------------- SDPA special case
@pytest.mark.parametrize("window", [0, 128, 5])
@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_decode_equals_sdpa_with_extra_key(oracle, window, kv_dtype):
    case = W.make_decode_case([1, 17, 130, 300], page_size=16, paged=True, window=window,
                              kv_dtype=kv_dtype, poison_pages=5, seed=11)
    out, lse, rows = run_oracle(oracle, case)
    ref_o, ref_l = sdpa_reference(case, *rows)
    assert np.allclose(out, ref_o.numpy(), rtol=0, atol=1e-12)
    assert np.allclose(lse, ref_l.numpy(), rtol=0, atol=1e-12)


def test_prefill_ragged_equals_sdpa(oracle):
    # ragged prefill, L_q < L_kv (bottom-right aligned), NHD contiguous layout
    case = W.make_prefill_case([5, 40, 1], [9, 40, 70], page_size=128, window=16, seed=5)
    out, lse, rows = run_oracle(oracle, case)
    ref_o, ref_l = sdpa_reference(case, *rows)
    assert np.allclose(out, ref_o.numpy(), rtol=0, atol=1e-12)
    assert np.allclose(lse, ref_l.numpy(), rtol=0, atol=1e-12)


def test_hnd_and_nhd_layouts_agree(oracle):
    a = W.make_decode_case([37, 64], page_size=16, paged=True, seed=2, layout="HND")
    b = W.make_decode_case([37, 64], page_size=16, paged=True, seed=2, layout="NHD")
    # same draws, different physical layout: give b the logical content of a
    Ka, Va = logical_kv(a)
    kb, vb = b.kv.k.clone(), b.kv.v.clone()
    for bb, L in enumerate(a.seqlens.tolist()):
        for t in range(L):
            pg = int(b.kv.page_table[bb, t // 16])
            kb[pg, t % 16] = Ka[bb, :, t].to(torch.bfloat16)
            vb[pg, t % 16] = Va[bb, :, t].to(torch.bfloat16)
    b.kv.k, b.kv.v, b.q, b.sinks = kb, vb, a.q, a.sinks
    oa, la, _ = run_oracle(oracle, a)
    ob, lb, _ = run_oracle(oracle, b)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


# --------------------------------------------------------- limiting cases
def test_no_sink_is_plain_softmax_attention(oracle):
    case = W.make_decode_case([50, 200], page_size=16, sinks=False, seed=4)
    out, lse, rows = run_oracle(oracle, case)
    K, V = logical_kv(case)
    q = case.q.double()
    for b, L in enumerate(case.seqlens.tolist()):
        for h in range(64):
            s = (K[b, h // 8, :L] @ q[b, h]) * case.sm_scale
            p = torch.softmax(s, 0)
            assert np.allclose(out[b, h], (p @ V[b, h // 8, :L]).numpy(), atol=1e-12)
            assert abs(lse[b, h] - float(torch.logsumexp(s, 0))) < 1e-12


def test_huge_sink_drives_output_to_zero(oracle):
    case = W.make_decode_case([33, 100], page_size=16, seed=9)
    case.sinks = torch.full((64,), 1e4, dtype=torch.float32)
    out, lse, _ = run_oracle(oracle, case)
    assert np.abs(out).max() < 1e-100
    assert np.allclose(lse, 1e4, atol=1e-9)


def test_key_probabilities_sum_to_one_minus_sink(oracle):
    case = W.make_decode_case([1, 16, 77], page_size=16, seed=12)
    ones = torch.ones_like(case.kv.v)
    case.kv.v = torch.where(torch.isnan(case.kv.v), case.kv.v, ones)
    out, lse, _ = run_oracle(oracle, case)
    p_sink = np.exp(case.sinks.double().numpy()[None, :] - lse)
    assert np.allclose(out, (1.0 - p_sink)[..., None], atol=1e-12)
    assert (p_sink > 0).all() and (p_sink < 1).all()


def test_window_128_equals_full_when_short(oracle):
    a = W.make_decode_case([1, 64, 127, 128], page_size=16, window=0, seed=21)
    b = W.make_decode_case([1, 64, 127, 128], page_size=16, window=128, seed=21)
    oa, la, _ = run_oracle(oracle, a)
    ob, lb, _ = run_oracle(oracle, b)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)
    c = W.make_decode_case([129], page_size=16, window=128, seed=21)
    d = W.make_decode_case([129], page_size=16, window=0, seed=21)
    oc, _, _ = run_oracle(oracle, c)
    od, _, _ = run_oracle(oracle, d)
    assert not np.allclose(oc, od)  # key 0 leaves the window at L = 129


def test_window_edge_is_exactly_128_keys(oracle):
    # one visible key carries a huge score; it must count iff j > p - 128
    L = 300
    for t, visible in [(L - 1 - 128, False), (L - 128, True), (L - 1, True)]:
        case = W.make_decode_case([L], num_qo_heads=8, num_kv_heads=8, page_size=16, window=128,
                                  sinks=False, seed=1)
        k = case.kv.k
        k.zero_()
        q = torch.zeros_like(case.q)
        q[0, :, 0] = 8.0
        pg = int(case.kv.page_table[0, t // 16])
        k[pg, :, t % 16, 0] = 8.0
        case.q = q
        out, lse, _ = run_oracle(oracle, case)
        # score of t is 8 (scale 1/8 * 64), the others 0: lse tells the count
        n_vis = 128
        expect = math.log(math.exp(8.0) + (n_vis - 1)) if visible else math.log(n_vis)
        assert abs(lse[0, 0] - expect) < 1e-12, (t, visible)


def test_empty_sequence(oracle):
    case = W.make_decode_case([0, 3], page_size=16, seed=2)
    rows = (np.array([0, 1], np.int32), np.array([-1, 2], np.int32))
    out, lse, _ = run_oracle(oracle, case, rows=rows)
    assert np.all(out[0] == 0.0)
    assert np.allclose(lse[0], case.sinks.double().numpy())
    case.sinks = None
    out, lse, _ = run_oracle(oracle, case, rows=rows)
    assert np.all(out[0] == 0.0) and np.all(np.isneginf(lse[0]))


# ------------------------------------------------------------ closed form
def test_closed_form_equal_keys(oracle):
    L = 50
    case = W.make_decode_case([L], page_size=16, seed=30, poison_pages=0)
    g = torch.Generator().manual_seed(1)
    krow = torch.randn(8, 64, generator=g).to(torch.bfloat16)
    vrow = torch.randn(8, 64, generator=g).to(torch.bfloat16)
    for t in range(L):
        pg = int(case.kv.page_table[0, t // 16])
        case.kv.k[pg, :, t % 16] = krow
        case.kv.v[pg, :, t % 16] = vrow
    out, lse, _ = run_oracle(oracle, case)
    q = case.q.double()[0]
    for h in range(64):
        s = float(q[h] @ krow[h // 8].double()) * case.sm_scale
        sig = float(case.sinks[h])
        denom = math.exp(sig) + L * math.exp(s)
        assert np.allclose(out[0, h], (L * math.exp(s) / denom) * vrow[h // 8].double().numpy(), atol=1e-12)
        assert abs(lse[0, h] - math.log(denom)) < 1e-12


# ---------------------------------------------------------- split algebra
@pytest.mark.parametrize("nsplit", [1, 2, 3, 7, 64])
def test_split_invariance(oracle, nsplit):
    case = W.make_decode_case([1, 50, 333, 1000], page_size=16, seed=40, window=0)
    out, lse, rows = run_oracle(oracle, case)
    chunk = (1000 + nsplit - 1) // nsplit
    out_s, lse_s, _ = run_oracle(oracle, case, split=(nsplit, chunk))
    assert np.allclose(out, out_s, atol=1e-12, rtol=0)
    assert np.allclose(lse, lse_s, atol=1e-12, rtol=0)


def test_key_ranges_merge_to_the_whole(oracle):
    """Sink-free states of [0, a) and [a, L) merged with the sink = the full row;
    a range with no visible key is (0, -inf)."""
    case = W.make_decode_case([1, 90, 500], page_size=16, seed=42, window=0)
    rows = oracle.decode_rows(case.seqlens)
    full_o, full_l, _ = run_oracle(oracle, case)
    kv = case.kv.as_dict()
    parts = []
    for lo, hi in [(0, 64), (64, 1 << 30)]:
        o, l = oracle.attend(case.q, rows[0], rows[1], kv, case.seqlens, None, 0, case.sm_scale,
                             key_range=(lo, hi))
        parts.append((o.reshape(3, 64, 64), l.reshape(3, 64)))
    mo, ml = oracle.merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]), case.sinks)
    assert np.allclose(mo, full_o, atol=1e-12) and np.allclose(ml, full_l, atol=1e-12)
    assert np.all(np.isneginf(parts[1][1][0])) and np.all(parts[1][0][0] == 0)  # L=1: nothing in [64, L)
    # a range with the sink given is the sink-seeded first chunk of the pages' online form
    o0, l0 = oracle.attend(case.q, rows[0], rows[1], kv, case.seqlens, case.sinks, 0, case.sm_scale,
                           key_range=(0, 1 << 30))
    assert np.array_equal(o0.reshape(3, 64, 64), full_o) and np.array_equal(l0.reshape(3, 64), full_l)


def test_split_invariance_window(oracle):
    case = W.make_decode_case([100, 300], page_size=16, seed=41, window=128)
    out, lse, _ = run_oracle(oracle, case)
    out_s, lse_s, _ = run_oracle(oracle, case, split=(5, 30))
    assert np.allclose(out, out_s, atol=1e-12) and np.allclose(lse, lse_s, atol=1e-12)


def test_merge_closed_form(oracle):
    g = torch.Generator().manual_seed(2)
    S, N, H, D = 3, 2, 4, 8
    o = torch.randn(S, N, H, D, generator=g, dtype=torch.float64)
    l = torch.randn(S, N, H, generator=g, dtype=torch.float64)
    l[1, 0, 0] = -math.inf  # empty chunk
    sinks = torch.randn(H, generator=g).float()
    out, lse = oracle.merge(o, l, sinks)
    for n in range(N):
        for h in range(H):
            w = [math.exp(float(l[s, n, h])) for s in range(S)]
            z = math.exp(float(sinks[h])) + sum(w)
            ref = sum(w[s] * o[s, n, h].numpy() for s in range(S)) / z
            assert np.allclose(out[n, h], ref, atol=1e-13)
            assert abs(lse[n, h] - math.log(z)) < 1e-13
    out0, lse0 = oracle.merge(o, l, None)
    w = np.exp(l.numpy())
    assert np.allclose(out0, (w[..., None] * o.numpy()).sum(0) / w.sum(0)[..., None], atol=1e-13)


# ------------------------------------------------------- golden fixtures
def test_golden_worked_examples(oracle):
    with open(os.path.join(GOLDEN, "worked_examples.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        D = len(c["q"][0][0])
        L = len(c["k"])
        k = torch.tensor(c["k"], dtype=torch.float64).to(torch.bfloat16)  # [L, D]
        v = torch.tensor(c["v"], dtype=torch.float64).to(torch.bfloat16)
        assert torch.equal(k.double(), torch.tensor(c["k"], dtype=torch.float64)), "not bf16-exact"
        kv = dict(k=k.reshape(1, 1, L, D), v=v.reshape(1, 1, L, D), dtype="bf16", num_pages=1,
                  num_kv_heads=1, head_dim=D, page_size=L, stride_page=L * D, stride_head=L * D,
                  stride_token=D, page_table=None, k_scale=1.0, v_scale=1.0)
        q = torch.tensor(c["q"], dtype=torch.float64).to(torch.bfloat16)  # [rows, 1, D]
        rows = len(c["positions"])
        sinks = None if c["sink"] is None else torch.tensor([c["sink"]], dtype=torch.float32)
        out, lse = oracle.attend(q, np.zeros(rows, np.int32), np.array(c["positions"], np.int32), kv,
                                 np.array([L], np.int32), sinks, c["window"], c["scale"])
        exp_o = np.array(c["expect_out"], np.float64)
        exp_l = np.array([float(x) for x in c["expect_lse"]], np.float64)
        assert np.allclose(out, exp_o, atol=1e-15), c["name"]
        assert np.allclose(lse, exp_l, atol=1e-15), c["name"]


# ------------------------------------------------------- E4M3 query input
@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_e4m3_query_equals_sdpa_on_decoded_values(oracle, kv_dtype):
    """A query given as E4M3 codes * q_scale: the SDPA identity evaluated on
    the codes decoded by torch (an independent decoder), for a scale that is
    not a power of two."""
    case = W.make_prefill_case([5, 33], [40, 33], window=16, kv_dtype=kv_dtype, num_qo_heads=4,
                               num_kv_heads=2, seed=77)
    q_scale = 0.0371
    g = torch.Generator().manual_seed(78)
    codes = torch.randint(0, 256, case.q.shape, generator=g, dtype=torch.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x11  # no NaN codes
    rows = oracle.prefill_rows(case.cu_seqlens_q, case.seqlens)
    out, lse = oracle.attend(codes, rows[0], rows[1], case.kv.as_dict(), case.seqlens, case.sinks, case.window,
                             case.sm_scale, q_scale=q_scale)
    decoded = codes.view(torch.float8_e4m3fn).double() * q_scale
    ref_case = W.Case(decoded, case.kv, case.seqlens, case.sinks, case.window, case.sm_scale, case.cu_seqlens_q,
                      "decoded")
    ref_o, ref_l = sdpa_reference(ref_case, rows[0], rows[1])
    n, Hq, D = case.q.shape
    assert np.allclose(out.reshape(n, Hq, D), ref_o.numpy(), rtol=1e-10, atol=1e-10)
    assert np.allclose(lse.reshape(n, Hq), ref_l.numpy(), rtol=1e-10, atol=1e-10)


def test_e4m3_query_with_power_of_two_scale_equals_bf16_query(oracle):
    """With q_scale = 2^-3 every decoded value is exact in bf16: the E4M3 path
    and the bf16 path must then agree to the last bit."""
    case = W.make_prefill_case([7], [20], seed=79)
    g = torch.Generator().manual_seed(80)
    codes = torch.randint(0, 256, case.q.shape, generator=g, dtype=torch.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x22
    vals = codes.view(torch.float8_e4m3fn).float() * 0.125
    q_bf16 = vals.to(torch.bfloat16)
    assert torch.equal(q_bf16.float(), vals)
    rows = oracle.prefill_rows(case.cu_seqlens_q, case.seqlens)
    a = oracle.attend(codes, rows[0], rows[1], case.kv.as_dict(), case.seqlens, case.sinks, 0, case.sm_scale,
                      q_scale=0.125)
    b = oracle.attend(q_bf16, rows[0], rows[1], case.kv.as_dict(), case.seqlens, case.sinks, 0, case.sm_scale)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_thread_count_does_not_change_results(oracle):
    """The oracle parallelises over (row, head) pairs only; each pair is summed
    in one fixed order, so its result is bit-identical on any thread count."""
    case = W.make_decode_case([1, 40, 333, 1024], page_size=16, window=0, poison_pages=2, seed=77)
    rows = oracle.decode_rows(case.seqlens)
    cores = oracle.num_threads()
    try:
        outs = []
        for n in (1, max(cores, 2)):
            oracle.set_num_threads(n)
            outs.append(oracle.attend(case.q, rows[0], rows[1], case.kv.as_dict(), case.seqlens, case.sinks,
                                      0, case.sm_scale))
    finally:
        oracle.set_num_threads(cores)
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
