"""Host-side helpers of bench.py: the kernel-source hash that ties the
committed DRAM-traffic counters to the code they were taken on."""
import os
import sys

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_only_drops_comments_and_blank_lines():
    src = "int a; // one\n/* two\n three */ int b;  \n\n   // four\nint c = 1; /* five */\n"
    assert bench._code_only(src) == "int a;\n int b;\nint c = 1;"


def test_comment_edits_keep_the_hash_and_code_edits_change_it():
    a = "__global__ void k() { int x = 1; } // old comment\n"
    b = "/* a new header */\n__global__ void k() { int x = 1; } // new comment\n"
    c = "__global__ void k() { int x = 2; }\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)


def test_traffic_is_tied_to_the_current_sources():
    h = bench.kernel_source_hash()
    assert len(h) == 16 and int(h, 16) >= 0
    assert bench.kernel_source_hash() == h          # deterministic
    assert bench.ncu_traffic("no such workload") is None
