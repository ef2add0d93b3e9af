"""The oracle's pins have teeth: each case plants one plausible mistake in a
copy of oracle.c (built into a temporary directory, on the CPU), runs the pins
of that part against the copy in a subprocess, and expects them to fail.  The
oracle itself is never modified."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

# (name, text in oracle.c, planted replacement, pin file)
MUTATIONS = [
    ("e4m3 rounds halves away from zero",
     "    k = nearbyint(a / q); /* a / q is exact; default mode is nearest-even */",
     "    k = floor(a / q + 0.5);", "test_oracle_codecs.py"),
    ("fp8 append skips the growth re-encode", "        if (s_new > s_old) {", "        if (0) {",
     "test_oracle_append.py"),
    ("int4 clamps at 8", "uint16_t oracle_int4_group(const float* x, int n, int8_t* codes) { return int_group(x, n, 7, codes); }",
     "uint16_t oracle_int4_group(const float* x, int n, int8_t* codes) { return int_group(x, n, 8, codes); }",
     "test_oracle_codecs.py"),
    ("a row does not see its own key", "    n = L + i + 1; /* keys 0 .. L + i */", "    n = L + i;",
     "test_oracle_attention.py"),
    ("q heads grouped round-robin", "    int hk = h / G;", "    int hk = h % c->num_kv_heads;",
     "test_oracle_attention.py"),
    ("argmax ties go to the highest index", "        if (best < 0 || x[i] > x[best])",
     "        if (best < 0 || x[i] >= x[best])", "test_oracle_accept.py"),
    ("int8 clamps at 128", "uint16_t oracle_int8_group(const float* x, int n, int8_t* codes) { return int_group(x, n, 127, codes); }",
     "uint16_t oracle_int8_group(const float* x, int n, int8_t* codes) { return int_group(x, n, 128, codes); }",
     "test_oracle_formats.py"),
    ("stochastic ratio test inverted",
     "if (!((double)u_accept[b * d + i] * (double)draft_probs[((size_t)b * d + i) * vocab + xi] < p[xi])) {",
     "if (!((double)u_accept[b * d + i] * p[xi] < (double)draft_probs[((size_t)b * d + i) * vocab + xi])) {",
     "test_oracle_sampled.py"),
    ("tree rows miss their own key", "            seen[j] = 1;", "            seen[j] = j != i || i == 0;",
     "test_oracle_tree.py"),
    ("int4 nibbles in the wrong order",
     "            codes[(g * 32 + i) / 2] = (uint8_t)((q[i] & 0xF) | ((q[i + 1] & 0xF) << 4));",
     "            codes[(g * 32 + i) / 2] = (uint8_t)((q[i + 1] & 0xF) | ((q[i] & 0xF) << 4));",
     "test_oracle_append.py"),
    ("fp8 fresh page keeps the old scale", "    if (start == 0) {", "    if (0) {", "test_oracle_append.py"),
    ("lazy form ignores the per-lane counts", "        int d = num_drafts ? num_drafts[b] : dmax, a = 0;",
     "        int d = dmax, a = 0;", "test_oracle_accept.py"),
    ("residual taken as q - p",
     "                const double r = p[x] - (double)draft_probs[((size_t)b * d + a) * vocab + x];",
     "                const double r = (double)draft_probs[((size_t)b * d + a) * vocab + x] - p[x];",
     "test_oracle_sampled.py"),
]

RUNNER = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import oracle
oracle._SRC = {src!r}
oracle._LIB_PATH = {lib!r}
try:
    oracle.build()
except Exception:
    sys.exit(3)  # the planted copy must compile: only failing pins count
import pytest
sys.exit(pytest.main(["-q", "-x", "-p", "no:cacheprovider", {pins!r}]))
"""


@pytest.mark.parametrize("name,old,new,pins", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_the_planted_mistake(tmp_path, name, old, new, pins):
    text = open(SRC).read()
    assert text.count(old) == 1, f"the text to mutate is no longer unique in oracle.c: {old!r}"
    src = tmp_path / "oracle.c"
    src.write_text(text.replace(old, new))
    code = RUNNER.format(root=ROOT, tests=os.path.join(ROOT, "tests"), src=str(src),
                         lib=str(tmp_path / "liboracle.so"), pins=os.path.join(ROOT, "tests", pins))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 1, f"{name}: the pins in {pins} did not fail (rc {r.returncode})\n{r.stdout[-2000:]}"
