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
    # At least the logits, read once, and within 20 % of them.
    assert 77_800_448 <= d["dram_bytes_per_launch"] <= 1.2 * 77_800_448
