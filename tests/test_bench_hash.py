"""CPU tests of bench.py's record of which kernel sources the committed DRAM
counters were taken on: the hash covers the code, not its comments."""

import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_comments_and_spacing_do_not_change_the_code():
    a = "int f(int x) {\n  return x + 1;  // one more\n}\n"
    b = "/* header\n   text */\nint f(int x)\n{\n    return x + 1;\n}\n// trailing\n"
    assert bench._code_only(a) == bench._code_only(b)


def test_code_changes_change_the_code():
    a = "int f(int x) { return x + 1; }"
    b = "int f(int x) { return x + 2; }"
    assert bench._code_only(a) != bench._code_only(b)


def test_recorded_traffic_only_for_the_sources_it_was_taken_on():
    with open(bench.TRAFFIC_FILE) as f:
        d = json.load(f)
    if d["kernel_hash"] != bench.kernel_hash():
        # Kernels changed since the counters were taken: the bench reports none.
        assert bench.recorded_traffic() is None
        pytest.skip("the committed DRAM counters predate the current kernel code")
    assert bench.recorded_traffic() == d["dram_bytes_per_launch"]
    # At least the logits, read once; at most the logits plus the call's
    # workspace read once and written back once (a 256-byte header, then per
    # (row, chunk) a 3216-byte record and 16 KB of slice histograms; the
    # mixed batch has 256 rows of 8 chunks).
    logits = 256 * 151936 * 2
    workspace = 256 + 256 * 8 * (3216 + 8 * 1024 * 2)
    assert logits <= d["dram_bytes_per_launch"] <= logits + 2 * workspace
