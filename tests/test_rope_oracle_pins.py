"""Pins of the RoPE / YaRN / cache-write oracle (oracle/rope.py) against
facts that do not come from its own code: the closed form of plain rotary
embeddings, the relative-position identity that defines them, norm
preservation, the YaRN paper's description of which dimensions keep and which
interpolate their frequency, the E4M3 format (all codes, and torch's float8
cast), and a brute-force cache write; bf16 storage as one rounding of the exact value
(brute force by exact rational distances)."""
import importlib.util
import math
import os

import numpy as np
import pytest
import torch

if os.environ.get("SA_ROPE_ORACLE"):  # a planted-mistake copy (tests/test_oracle_mutants.py)
    _spec = importlib.util.spec_from_file_location("rope_mutant", os.environ["SA_ROPE_ORACLE"])
    R = importlib.util.module_from_spec(_spec)
    _spec.loader.exec_module(R)
else:
    from oracle import rope as R

GPT_OSS_LIKE = dict(theta=150000.0, factor=32.0, original_max_position=4096, beta_fast=32.0, beta_slow=1.0)


def test_plain_rope_at_factor_one():
    f, ms = R.yarn_inv_freq(64, 10000.0, 1.0, 4096, 32.0, 1.0)
    assert ms == 1.0
    for i in range(32):
        assert f[i] == pytest.approx(1.0 / 10000.0 ** (i / 32.0), rel=1e-15)
    # rotating position 1 of the first pair: (1, 0) -> (cos 1, sin 1)
    x = np.zeros(64)
    x[0] = 1.0
    y = R.rope_rotate(x, 1, f, ms)
    assert y[0] == pytest.approx(math.cos(1.0)) and y[32] == pytest.approx(math.sin(1.0))
    assert np.allclose(np.delete(y, [0, 32]), 0.0)


@pytest.mark.parametrize("yarn", [dict(theta=10000.0, factor=1.0, original_max_position=4096, beta_fast=32.0,
                                       beta_slow=1.0), GPT_OSS_LIKE])
def test_scores_depend_only_on_the_position_difference(yarn):
    f, ms = R.yarn_inv_freq(64, **yarn)
    g = np.random.default_rng(1)
    q, k = g.standard_normal(64), g.standard_normal(64)
    for p, pk, delta in [(5, 3, 100), (1000, 7, 12345), (0, 0, 77777)]:
        a = R.rope_rotate(q, p, f, ms) @ R.rope_rotate(k, pk, f, ms)
        b = R.rope_rotate(q, p + delta, f, ms) @ R.rope_rotate(k, pk + delta, f, ms)
        assert a == pytest.approx(b, rel=1e-9, abs=1e-9)
    # and at equal positions the rotation cancels: q.k * mscale^2
    assert R.rope_rotate(q, 4321, f, ms) @ R.rope_rotate(k, 4321, f, ms) == pytest.approx(ms * ms * (q @ k))


def test_rotation_scales_each_pair_by_mscale():
    f, ms = R.yarn_inv_freq(64, **GPT_OSS_LIKE)
    assert ms == pytest.approx(0.1 * math.log(32.0) + 1.0)
    x = np.random.default_rng(2).standard_normal((5, 64))
    y = R.rope_rotate(x, np.array([0, 1, 99, 4096, 131071]), f, ms)
    n_in = x[:, :32] ** 2 + x[:, 32:] ** 2
    n_out = y[:, :32] ** 2 + y[:, 32:] ** 2
    assert np.allclose(n_out, ms * ms * n_in, rtol=1e-12)
    assert np.allclose(y[0], ms * x[0])  # position 0 only scales


def test_yarn_keeps_fast_dimensions_and_interpolates_slow_ones():
    """The paper's criterion in its own terms: a dimension that turns more than
    beta_fast times over the original context keeps its frequency; one that
    turns less than beta_slow times is divided by the factor; in between the
    frequency lies between the two."""
    y = GPT_OSS_LIKE
    f, _ = R.yarn_inv_freq(64, **y)
    seen_keep = seen_interp = seen_mid = False
    for i in range(32):
        base = y["theta"] ** (-i / 32.0)
        turns = y["original_max_position"] * base / (2 * math.pi)
        if turns > y["beta_fast"]:
            assert f[i] == pytest.approx(base, rel=1e-12)
            seen_keep = True
        elif turns < y["beta_slow"]:
            assert f[i] == pytest.approx(base / y["factor"], rel=1e-12)
            seen_interp = True
        else:  # strictly between the two: a blend, not either end
            assert base / y["factor"] * (1 + 1e-9) < f[i] < base * (1 - 1e-9)
            seen_mid = True
    assert seen_keep and seen_interp and seen_mid
    assert np.all(np.diff(f) < 0)  # still strictly decreasing


def test_e4m3_encoder_round_trips_every_code_and_matches_torch():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    vals = R.e4m3_decode(codes)
    ref = torch.tensor(codes).view(torch.float8_e4m3fn).float().double().numpy()
    assert np.array_equal(vals, ref)
    enc = R.e4m3_encode(vals)
    # -0 and +0 both decode to 0; every other code comes back unchanged
    assert np.array_equal(enc[vals != 0], codes[vals != 0])
    g = np.random.default_rng(3)
    x = np.concatenate([g.standard_normal(4000) * 50, g.standard_normal(2000) * 0.01,
                        (vals[:-1] + vals[1:]) / 2])  # exact midpoints: ties to even
    x = x[np.abs(x) <= 448]
    ours = R.e4m3_encode(x)
    theirs = torch.tensor(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(R.e4m3_decode(ours), R.e4m3_decode(theirs))
    assert R.e4m3_encode(np.array([500.0, -1e9, 448.0]))[0] == 0x7E
    assert R.e4m3_encode(np.array([-1e9]))[0] == 0xFE


def test_bf16_rounding_matches_torch():
    # fp32-exact inputs: torch rounds fp64 through fp32, which is then exact
    x = (np.random.default_rng(4).standard_normal(10000) * 10).astype(np.float32).astype(np.float64)
    ours = R.bf16_bits_rne(x)
    theirs = torch.tensor(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, theirs)


def _bf16_nearest_brute_force(xs):
    """Bit patterns of the bf16 values nearest to each x, by exact rational
    distances to the two neighbouring bf16 values; ties go to the even
    pattern.  The bf16 values are torch's decoding of every pattern (an exact
    widening); inf stands at 2^128, the next value past the largest finite
    one.  Sign by symmetry."""
    from fractions import Fraction
    pats = np.arange(0, 0x7F81, dtype=np.uint16)
    vals = torch.tensor(pats.view(np.int16)).view(torch.bfloat16).double().numpy()
    vals[-1] = 2.0 ** 128
    out = []
    for x in xs:
        a = abs(float(x))
        j = int(np.searchsorted(vals, a))
        if j < len(vals) and vals[j] == a:
            best = j
        else:
            lo, hi = j - 1, j
            dl, dh = Fraction(a) - Fraction(vals[lo]), Fraction(vals[hi]) - Fraction(a)
            best = lo if dl < dh else hi if dh < dl else (lo if lo % 2 == 0 else hi)
        out.append(best | (0x8000 if math.copysign(1.0, x) < 0 else 0))
    return np.array(out, np.uint16)


def test_bf16_rounding_is_one_rounding_of_the_exact_value():
    """The cache stores the fp64 value rounded once.  Inputs a hair off a bf16
    midpoint (relative 2^-40, inside half an fp32 ulp) are the ones where a
    rounding through fp32 first lands on the midpoint and then goes to even:
    the nearer neighbour is required, the brute force decides it."""
    g = np.random.default_rng(6)
    pats = np.concatenate([g.integers(1, 0x7F7F, 1500), np.arange(1, 8), np.arange(0x7F70, 0x7F7F)]).astype(np.uint16)
    lo = torch.tensor(pats.view(np.int16)).view(torch.bfloat16).double().numpy()
    hi = torch.tensor((pats + 1).astype(np.uint16).view(np.int16)).view(torch.bfloat16).double().numpy()
    mid = (lo + hi) / 2  # exact in fp64
    xs = np.concatenate([mid * (1 + 2.0 ** -40), mid * (1 - 2.0 ** -40), mid, lo + (hi - lo) * g.random(len(lo))])
    xs = np.concatenate([xs, -xs[::7], [2.0 ** 128 * (1 - 2.0 ** -9), 2.0 ** 128 * (1 - 2.0 ** -9) * (1 - 2.0 ** -40)]])
    want = _bf16_nearest_brute_force(xs)
    assert np.array_equal(R.bf16_bits_rne(xs), want)
    # these inputs do separate one rounding from two: through fp32 first, the
    # off-midpoint ones with an odd lower neighbour come out differently
    via32 = torch.tensor(xs.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (via32 != want).sum() > 500


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_cache_write_brute_force(dtype):
    g = np.random.default_rng(5)
    T, Hq, Hkv, d, P, npages = 5, 4, 2, 64, 32, 6
    q = g.standard_normal((T, Hq, d))
    k = g.standard_normal((T, Hkv, d))
    v = g.standard_normal((T, Hkv, d))
    seq = np.array([0, 1, 1, 0, 1])
    pos = np.array([3, 0, 17, 40, 18])
    table = np.array([[5, 2, 0], [1, 4, 3]])
    store = np.uint16 if dtype == "bf16" else np.uint8
    kc = np.zeros((npages, Hkv, P, d), store)  # HND
    vc = np.zeros_like(kc)
    cache = dict(k=kc, v=vc, dtype=dtype, page_table=table, page_size=P, stride_page=Hkv * P * d,
                 stride_head=P * d, stride_token=d, k_scale=0.05, v_scale=0.02)
    y = dict(theta=10000.0, factor=4.0, original_max_position=64, beta_fast=32.0, beta_slow=1.0)
    q_out = R.rope_append(q, k, v, seq, pos, y, cache)
    f, ms = R.yarn_inv_freq(d, **y)
    for t in range(T):
        page, slot = table[seq[t], pos[t] // P], pos[t] % P
        for h in range(Hq):
            ang = pos[t] * f
            want = np.concatenate([q[t, h, :32] * np.cos(ang) - q[t, h, 32:] * np.sin(ang),
                                   q[t, h, 32:] * np.cos(ang) + q[t, h, :32] * np.sin(ang)]) * ms
            assert np.allclose(q_out[t, h], want, rtol=1e-12, atol=1e-12)
        for gg in range(Hkv):
            kr = R.rope_rotate(k[t, gg], pos[t], f, ms)
            if dtype == "bf16":
                got_k = torch.tensor(kc[page, gg, slot].view(np.int16)).view(torch.bfloat16).double().numpy()
                got_v = torch.tensor(vc[page, gg, slot].view(np.int16)).view(torch.bfloat16).double().numpy()
                assert np.allclose(got_k, kr, rtol=2 ** -8, atol=1e-30)
                assert np.allclose(got_v, v[t, gg], rtol=2 ** -8, atol=1e-30)
            else:
                got_k = R.e4m3_decode(kc[page, gg, slot]) * 0.05
                got_v = R.e4m3_decode(vc[page, gg, slot]) * 0.02
                assert np.allclose(got_k, kr, rtol=2 ** -4, atol=2 ** -10 * 0.05)
                assert np.allclose(got_v, v[t, gg], rtol=2 ** -4, atol=2 ** -10 * 0.02)
    # untouched slots stay zero
    written = {(table[seq[t], pos[t] // P], pos[t] % P) for t in range(T)}
    for pg in range(npages):
        for sl in range(P):
            if (pg, sl) not in written:
                assert not kc[pg, :, sl].any() and not vc[pg, :, sl].any()
