"""The oracle's pins catch plausible mistakes.  Each case plants one mistake
in a copy of oracle/oracle.cpp (on the CPU), compiles it to a temporary
library, and runs tests/test_oracle_pins.py against it in a subprocess: the
pins must fail.  The unchanged source, compiled the same way, must pass."""

import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(ROOT, "oracle", "oracle.cpp")

# (name, text in oracle.cpp, replacement): one plausible slip each.
MUTANTS = [
    ("top-p on the inclusive cumulative mass",
     "const double frac = before / zk;", "const double frac = (before + w[i]) / zk;"),
    ("temperature multiplies instead of dividing",
     "w[i] = std::exp((l[i] - m) / T);", "w[i] = std::exp((l[i] - m) * T);"),
    ("no renormalisation after top-p",
     "const double q = w[i] / zs;", "const double q = w[i] / zk;"),
    ("ties ranked by descending index",
     "return a < b;", "return a > b;"),
    ("argmax keeps the last of tied maxima",
     "if (l[i] > l[best]) best = i;", "if (l[i] >= l[best]) best = i;"),
    ("draw walks the sorted order",
     "  for (int i = 0; i < V; ++i) {\n    if (!in_s[i]) continue;\n    const double q = w[i] / zs;",
     "  for (int jj = 0; jj < V; ++jj) {\n    const int i = order[jj];\n    if (!in_s[i]) continue;\n"
     "    const double q = w[i] / zs;"),
    ("page counts by floor instead of ceil",
     "int64_t div_ceil(int64_t a, int64_t b) { return (a + b - 1) / b; }",
     "int64_t div_ceil(int64_t a, int64_t b) { return a / b; }"),
    ("page fill without the in-page offset",
     "(first[i] + j) * page_size + o] = start + o;", "(first[i] + j) * page_size + o] = start;"),
    ("allocation offsets restart per request",
     "offset[i] = needed;", "offset[i] = 0;"),
    ("positions shifted by one",
     "positions[j] = static_cast<int32_t>(pos);", "positions[j] = static_cast<int32_t>(pos + 1);"),
    ("out_loc read one column early",
     "out_loc[j] = ok ? page_table[t * pt_cols + pos] : -1;",
     "out_loc[j] = ok ? page_table[t * pt_cols + pos - 1] : -1;"),
    ("lazy free appends every entry, not every ps-th",
     "for (int64_t col = b; col < e; col += page_size) {", "for (int64_t col = b; col < e; col += 1) {"),
    ("integrity check without the alignment test",
     "if (page_size > 1 && slot % page_size != 0) {", "if (false) {"),
    ("Philox mixes the wrong halves",
     "const uint64_t y0 = hi1 ^ x1 ^ k0, y1 = lo1, y2 = hi0 ^ x3 ^ k1, y3 = lo0;",
     "const uint64_t y0 = hi0 ^ x1 ^ k0, y1 = lo0, y2 = hi1 ^ x3 ^ k1, y3 = lo1;"),
    ("min_p never drops a token",
     "if (w[i] < min_p) in_s[i] = 0;", "if (w[i] < 0.0) in_s[i] = 0;"),
]


def _build(src_text, tmp_path, name):
    cpp = tmp_path / f"{name}.cpp"
    lib = tmp_path / f"{name}.so"
    cpp.write_text(src_text)
    subprocess.run(["g++", "-O1", "-std=c++17", "-shared", "-fPIC", "-pthread", str(cpp), "-o",
                    str(lib)], check=True)
    return str(lib)


def _run_pins(lib):
    env = dict(os.environ, PKV_ORACLE_LIB=lib)
    return subprocess.run([sys.executable, "-m", "pytest", os.path.join(HERE, "test_oracle_pins.py"),
                           "-x", "-q", "-p", "no:cacheprovider"], cwd=ROOT, env=env,
                          capture_output=True, text=True)


def test_unchanged_source_passes(tmp_path):
    r = _run_pins(_build(open(SRC).read(), tmp_path, "control"))
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(name, old, new, tmp_path):
    text = open(SRC).read()
    assert text.count(old) == 1, f"the text to mutate is not unique: {old!r}"
    r = _run_pins(_build(text.replace(old, new), tmp_path, "mutant"))
    assert r.returncode == 1, f"no pin failed for: {name}\n{r.stdout[-1500:]}"
