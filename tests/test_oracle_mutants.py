"""The oracle's pins must catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of oracle/sa_oracle.c (on the CPU),
builds it, and runs the pin suite against that build: the suite must fail.
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
