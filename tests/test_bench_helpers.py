"""Host-side helpers of bench.py: the kernel-source hash that ties the
committed DRAM-traffic counters to the code they were taken on, and the
gather-ceiling sweep's probe configurations."""
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


def test_ceiling_sweep_fits_and_covers_both_copy_methods():
    """Every probe configuration of the gather-ceiling sweep fits its CTAs on
    one SM (as the probe pads them), and both copy methods are swept for each
    CTA count; the pair modes copy by TMA only."""
    import bench
    for row_bytes in (1024, 576, 512, 128):
        tile = 64 * 128 * ((row_bytes + 127) // 128)
        cfgs = bench.ceiling_configs(row_bytes)
        for k, st, pm, iw, cm in cfgs:
            assert 1 <= st <= 8 and 1 <= k <= 4
            assert k * (1024 + st * tile + 24 * 8 + 64 + 1024) <= 233472
            assert cm in (0, 1) and not (cm and (pm or iw))
        for k in {c[0] for c in cfgs if not c[2]}:
            assert {c[4] for c in cfgs if c[0] == k and not c[2]} == {0, 1}
        assert {c[2] for c in cfgs} == {0, 1, 2}


def test_shared_gpu_split_plan():
    """Calls that share the GPU are planned for half its SMs: one split per row
    for decode bf16, two for decode fp8 (two lean CTAs per SM), none for
    prefill; the 128-head path keeps its automatic plan (0)."""
    from sparse_mla_attention_04_gb300 import binding, build, inputs
    build.build()   # the library's host-only plan (nvcc cross-compiles; no GPU needed)
    want = {"decode_bf16": 1, "decode_fp8": 2, "prefill_bf16": 1, "wide_fp8": 0}
    for name, S in want.items():
        w = inputs.CONFIGS[name](seed=0)
        assert bench.shared_gpu_splits(binding, w, 152) == S, name
