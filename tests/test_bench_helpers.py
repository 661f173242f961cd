"""Host-side helpers of bench.py: the kernel code hash that keys the recorded
ncu traffic ignores comments and blank lines but not code, and a recorded
figure is reported only for the code it was captured on."""
from __future__ import annotations

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_only_drops_comments_and_blank_lines():
    src = "int a = 1;  // one\n\n/* block\n   comment */ int b = 2;\n    \nint c = a/b; /* x */\n"
    assert bench.code_only(src) == "int a = 1;\n int b = 2;\nint c = a/b;"


def test_code_only_keeps_code_changes():
    a = "x = y * 2; // double\n"
    assert bench.code_only(a) == bench.code_only("x = y * 2; // twice\n")
    assert bench.code_only(a) != bench.code_only("x = y * 3; // double\n")


def test_recorded_traffic_is_reported_only_for_its_own_kernel_code():
    """profiles/traffic.txt holds per-launch DRAM bytes keyed by the code
    hash of the kernel they were captured on: bench.py reports a figure as
    roofline.traffic only while the code is unchanged, and null otherwise."""
    src = bench.kernel_source_hash()
    rows = [line.split() for line in open(os.path.join(ROOT, "profiles", "traffic.txt")) if line.strip()]
    assert rows and all(len(r) == 3 and float(r[2]) > 0 for r in rows)
    for tag, h, nbytes in rows:
        got = bench.profile_traffic(tag)
        if h == src:
            assert got == float(nbytes)
        elif not any(r[0] == tag and r[1] == src for r in rows):
            assert got is None
