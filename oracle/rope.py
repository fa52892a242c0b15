"""fp64 CPU oracle for the step in front of attention: rotary position
embedding with YaRN frequency scaling applied to q and k, then the write of
k and v into the paged cache (bf16 or FP8-E4M3 codes).

TEST INFRASTRUCTURE ONLY: imported by tests/ and by the CPU legs of
``bench.py``, never by the library.  Plain numpy in fp64, one step at a time.

Sources.  "GPT-OSS on day 0" (Perplexity), model overview: the position
encoding is YaRN, as in DeepSeek-V3.  vLLM "GPT-OSS optimisations on NVIDIA
Blackwell", list of fusions: RoPE, the query and the KV-cache write fused into
one operator.  NVIDIA launch article, introduction: RoPE, 128k context.  The
pages print no formula and no parameter, so the steps below follow the
published YaRN method (Peng et al., "YaRN: Efficient Context Window Extension
of Large Language Models", sections on "NTK-by-parts" interpolation and on
the attention temperature), in the per-dimension form DeepSeek-V3 uses:

  * base frequencies  f_i = theta^(-2i/d), i = 0 .. d/2-1 (d = head_dim);
  * the dimension that completes n full turns over the original context L is
    c(n) = d * ln(L / (2 pi n)) / (2 ln theta);
  * a ramp over the dimension index between lo = floor(c(beta_fast)) and
    hi = ceil(c(beta_slow)) (clipped to [0, d-1]; hi = lo + 0.001 if equal):
    g_i = clamp((i - lo) / (hi - lo), 0, 1);
  * scaled frequencies  f'_i = f_i * (1 - g_i) + (f_i / s) * g_i: dimensions
    that turn often over L keep their frequency, slow ones are interpolated by
    the factor s;
  * attention temperature: cos and sin are multiplied by
    mscale = 0.1 ln(s) + 1 (s > 1; else 1), so q.k grows by mscale^2;
  * rotation of the two halves (x1 = x[:d/2], x2 = x[d/2:]):
    y1 = x1 cos - x2 sin,  y2 = x2 cos + x1 sin,  angle = p * f'_i.

The cache write puts token t of sequence b = seq_ids[t] at position
p = positions[t]: page table[b, p // P] (or page b for a cache without table),
slot p % P.  FP8 caches store e4m3(value / scale), rounded to nearest even and
saturated to +-448; bf16 caches store the value rounded to nearest even.

Pinned by tests/test_rope_oracle_pins.py: plain RoPE at s = 1 (closed form),
the relative-position identity of rotary embeddings, norm preservation, the
two ends of the YaRN ramp stated in the paper's own terms (turns over L),
the E4M3 encoder against every code and against torch's float8 cast, and a
brute-force cache write.
"""
from __future__ import annotations

import math

import numpy as np


def yarn_inv_freq(head_dim: int, theta: float, factor: float, original_max_position: int,
                  beta_fast: float, beta_slow: float):
    """(f' [head_dim/2] fp64, mscale) -- see the module docstring."""
    d = int(head_dim)
    half = d // 2
    i = np.arange(half, dtype=np.float64)
    base = theta ** (-2.0 * i / d)
    if factor <= 1.0:
        return base, 1.0

    def turns_dim(n):
        return d * math.log(original_max_position / (2.0 * math.pi * n)) / (2.0 * math.log(theta))

    lo = max(math.floor(turns_dim(beta_fast)), 0)
    hi = min(math.ceil(turns_dim(beta_slow)), d - 1)
    if hi == lo:
        hi = lo + 0.001
    g = np.clip((i - lo) / (hi - lo), 0.0, 1.0)
    freq = base * (1.0 - g) + (base / factor) * g
    mscale = 0.1 * math.log(factor) + 1.0
    return freq, mscale


def rope_rotate(x, positions, inv_freq, mscale):
    """Rotate the last axis of x ([..., d], fp64) by angle positions * inv_freq.
    positions broadcasts against x's leading axes."""
    x = np.asarray(x, np.float64)
    half = x.shape[-1] // 2
    ang = np.asarray(positions, np.float64)[..., None] * np.asarray(inv_freq, np.float64)
    c = np.cos(ang) * mscale
    s = np.sin(ang) * mscale
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


# ---- storage encoders (own code, from the formats) ------------------------
def bf16_bits_rne(x):
    """fp64 -> bf16 bit patterns (uint16): one round-to-nearest-even of the
    exact fp64 value to 8 significant bits (exponent range of fp32, subnormals
    below 2^-126 in steps of 2^-133, overflow to inf past the largest finite
    value by half an ulp), NaN -> 0x7FC0.  No intermediate rounding: a value
    just off a bf16 midpoint goes to its nearer neighbour."""
    x = np.asarray(x, np.float64)
    a = np.abs(x)
    with np.errstate(over="ignore", invalid="ignore"):
        _, e2 = np.frexp(a)                   # a = f * 2^e2, f in [0.5, 1): a in [2^(e2-1), 2^e2)
        qexp = np.maximum(e2 - 1, -126) - 7   # exponent of one bf16 ulp at a (fixed below 2^-126)
        m = np.rint(np.ldexp(a, -qexp))       # exact scaling; rint rounds half to even
        r = np.ldexp(m, qexp)                 # the rounded value, exact in fp64 (m <= 256)
        bits = (r.astype(np.float32).view(np.uint32) >> 16).astype(np.uint32)  # exact, or inf past the range
    bits = np.where(np.signbit(x), bits | 0x8000, bits)
    bits = np.where(np.isnan(x), 0x7FC0, bits)
    return bits.astype(np.uint16)


def e4m3_encode(x):
    """fp64 -> E4M3 codes (uint8): 1 sign, 4 exponent (bias 7), 3 mantissa
    bits; subnormals below 2^-6 in steps of 2^-9; round to nearest even;
    magnitudes past 448 saturate to 448 (code 0x7E); NaN -> 0x7F."""
    x = np.asarray(x, np.float64)
    out = np.zeros(x.shape, np.uint8)
    flat = x.reshape(-1)
    o = out.reshape(-1)
    for n, v in enumerate(flat):
        if math.isnan(v):
            o[n] = 0x7F
            continue
        sign = 0x80 if (v < 0 or (v == 0 and math.copysign(1.0, v) < 0)) else 0
        a = abs(v)
        if a >= 448.0:
            o[n] = sign | 0x7E
            continue
        if a < 2.0 ** -6:  # subnormal range: quantum 2^-9
            q = a / 2.0 ** -9
            m = _round_half_even(q)  # 0 .. 8 (8 is the smallest normal)
            o[n] = sign | (0x08 if m == 8 else m)
            continue
        e = math.floor(math.log2(a))
        # guard log2 rounding at exact powers of two
        if 2.0 ** e > a:
            e -= 1
        elif 2.0 ** (e + 1) <= a:
            e += 1
        q = a / 2.0 ** (e - 3)  # in [8, 16)
        m = _round_half_even(q)
        if m == 16:
            e, m = e + 1, 8
        if e > 8 or (e == 8 and m > 14):
            o[n] = sign | 0x7E
            continue
        o[n] = sign | ((e + 7) << 3) | (m - 8)
    return out


def e4m3_decode(codes):
    c = np.asarray(codes, np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))
    val = np.where((c & 0x7F) == 0x7F, np.nan, val)
    return s * val


def _round_half_even(q: float) -> int:
    f = math.floor(q)
    r = q - f
    if r > 0.5 or (r == 0.5 and f % 2 == 1):
        return int(f) + 1
    return int(f)


# ---- the fused step --------------------------------------------------------
def rope_append(q, k, v, seq_ids, positions, yarn, cache):
    """q [T, Hq, d], k, v [T, Hkv, d] (any float dtype; read as fp64);
    seq_ids, positions [T]; yarn = dict(theta, factor, original_max_position,
    beta_fast, beta_slow); cache = dict(k, v (uint16 bf16 bits or uint8 codes,
    writable numpy arrays), dtype 'bf16'|'e4m3', page_table [B, n] or None,
    page_size, stride_page, stride_head, stride_token (elements), k_scale,
    v_scale).  Returns q_out [T, Hq, d] fp64 and writes k / v into the cache
    arrays (flat views).  Tokens whose page lies outside the pool are skipped."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    d = q.shape[-1]
    freq, mscale = yarn_inv_freq(d, yarn["theta"], yarn["factor"], yarn["original_max_position"],
                                 yarn["beta_fast"], yarn["beta_slow"])
    pos = np.asarray(positions, np.int64)
    q_out = rope_rotate(q, pos[:, None], freq, mscale)
    k_rot = rope_rotate(k, pos[:, None], freq, mscale)
    kc = cache["k"].reshape(-1)
    vc = cache["v"].reshape(-1)
    P = int(cache["page_size"])
    table = cache.get("page_table")
    num_pages = cache["k"].shape[0]
    for t in range(q.shape[0]):
        b = int(seq_ids[t])
        p = int(pos[t])
        page = int(table[b, p // P]) if table is not None else b
        if page < 0 or page >= num_pages:
            continue
        for g in range(k.shape[1]):
            off = page * cache["stride_page"] + g * cache["stride_head"] + (p % P) * cache["stride_token"]
            if cache["dtype"] == "bf16":
                kc[off:off + d] = bf16_bits_rne(k_rot[t, g])
                vc[off:off + d] = bf16_bits_rne(v[t, g])
            else:
                kc[off:off + d] = e4m3_encode(k_rot[t, g] / cache["k_scale"])
                vc[off:off + d] = e4m3_encode(v[t, g] / cache["v_scale"])
    return q_out
