"""The oracle's pins must catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of oracle/sa_oracle.c (on the CPU),
builds it, and runs the pin suite against that build: the suite must fail.
The same for the rotary oracle, oracle/rope.py, against its own pins.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "sa_oracle.c")

MUTANTS = {
    "sink dropped from the denominator":
        ("    Z = (sigma == -INFINITY) ? 0.0 : exp(sigma - M);\n    for (j = 0; j < n; ++j) {",
         "    Z = 0.0;\n    for (j = 0; j < n; ++j) {"),
    "sink left out of the running max":
        ("    M = sigma;\n    for (j = 0; j < n; ++j)\n        if (s[j] > M)",
         "    M = -INFINITY;\n    for (j = 0; j < n; ++j)\n        if (s[j] > M)"),
    "window one key too wide": ("if (window > 0 && j <= p - window)", "if (window > 0 && j < p - window)"),
    "window one key too narrow": ("if (window > 0 && j <= p - window)", "if (window > 0 && j <= p - window + 1)"),
    "causal mask excludes the diagonal": ("if (j < 0 || j > p || j >= L)", "if (j < 0 || j >= p || j >= L)"),
    "interleaved GQA grouping": ("h / G, row_pos[r]", "h % kv->num_kv_heads, row_pos[r]"),
    "softmax scale dropped": ("    return sm_scale * acc;", "    return acc;"),
    "lse without the max": ("    *lse = M + log(Z);", "    *lse = log(Z);"),
    "keys read from the value cache": ("kv_elem(kv, kv->k, kv->k_scale, off, d)", "kv_elem(kv, kv->v, kv->k_scale, off, d)"),
    "value scale ignored": ("kv_elem(kv, kv->v, kv->v_scale, off, d)", "kv_elem(kv, kv->v, 1.0, off, d)"),
    "E4M3 bias off by one": ("mag = ldexp(1.0 + (double)m / 8.0, e - 7);", "mag = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    "E4M3 subnormal exponent": ("mag = ldexp((double)m / 8.0, 1 - 7);", "mag = ldexp((double)m / 8.0, -7);"),
    "page slot from a fixed page size": ("int64_t slot = t % kv->page_size;", "int64_t slot = t % 16;"),
    "merge drops the sink":
        ("        Z = (sigma == -INFINITY) ? 0.0 : exp(sigma - M);\n        for (s = 0; s < S; ++s) {",
         "        Z = 0.0;\n        for (s = 0; s < S; ++s) {"),
    "merge weight sign": ("            w = exp(l - M);", "            w = exp(M - l);"),
    "head and token strides swapped":
        ("return page * kv->stride_page + (int64_t)g * kv->stride_head + slot * kv->stride_token;",
         "return page * kv->stride_page + (int64_t)g * kv->stride_token + slot * kv->stride_head;"),
    "split chunks overlap by one key": ("lo, lo + chunk, part_o", "lo, lo + chunk + 1, part_o"),
    "E4M3 query scale ignored":
        ("return sao_e4m3_to_f64(((const uint8_t *)q->row)[d]) * q->scale;",
         "return sao_e4m3_to_f64(((const uint8_t *)q->row)[d]);"),
    "E4M3 query bytes swapped in pairs":
        ("return sao_e4m3_to_f64(((const uint8_t *)q->row)[d]) * q->scale;",
         "return sao_e4m3_to_f64(((const uint8_t *)q->row)[d ^ 1]) * q->scale;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, "mutation site not found: " + name
    mutated = tmp_path / "sa_oracle_mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-o", str(lib), str(mutated), "-lm"],
                   check=True, capture_output=True)
    env = dict(os.environ, SA_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, "pins did not notice: " + name


ROPE_SRC = os.path.join(ROOT, "oracle", "rope.py")
ROPE_MUTANTS = {
    "rotation pairs neighbouring dims":
        ("    x1, x2 = x[..., :half], x[..., half:]\n    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)",
         "    x1, x2 = x[..., 0::2], x[..., 1::2]\n    y = np.empty_like(x)\n    y[..., 0::2] = x1 * c - x2 * s\n"
         "    y[..., 1::2] = x2 * c + x1 * s\n    return y"),
    "rotation sign": ("x2 * c + x1 * s], axis=-1)", "x2 * c - x1 * s], axis=-1)"),
    "frequency exponent": ("base = theta ** (-2.0 * i / d)", "base = theta ** (-1.0 * i / d)"),
    "ramp direction": ("freq = base * (1.0 - g) + (base / factor) * g", "freq = base * g + (base / factor) * (1.0 - g)"),
    "no attention temperature": ("mscale = 0.1 * math.log(factor) + 1.0", "mscale = 1.0"),
    "beta roles swapped": ("lo = max(math.floor(turns_dim(beta_fast)), 0)", "lo = max(math.floor(turns_dim(beta_slow)), 0)"),
    "E4M3 ties away from zero": ("    if r > 0.5 or (r == 0.5 and f % 2 == 1):", "    if r >= 0.5:"),
    "E4M3 saturates to the NaN code": ("o[n] = sign | 0x7E", "o[n] = sign | 0x7F"),
    "cache slot ignores the page size": ("(p % P) * cache[\"stride_token\"]", "(p % 16) * cache[\"stride_token\"]"),
    "bf16 rounded through fp32 first": ("    a = np.abs(x)\n    with np.errstate", "    a = np.abs(x.astype(np.float32).astype(np.float64))\n    with np.errstate"),
}


@pytest.mark.parametrize("name", sorted(ROPE_MUTANTS))
def test_rope_pins_catch_planted_mistake(name, tmp_path):
    old, new = ROPE_MUTANTS[name]
    src = open(ROPE_SRC).read()
    assert src.count(old) >= 1, "mutation site not found: " + name
    mutated = tmp_path / "rope_mutant.py"
    mutated.write_text(src.replace(old, new))
    env = dict(os.environ, SA_ROPE_ORACLE=str(mutated))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_rope_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, "pins did not notice: " + name
