"""sparse_mla_fwd_no_alloc against sparse_mla_fwd and the oracle (GPU).

The no-allocation entry point serves callers that cannot allocate device
memory for a workspace (an engine that reserved nearly all of HBM for its
KV-cache pool, or a framework that only hands a plug-in fixed buffers): the
workspace lives in a static array inside the library. Through the C ABI this
checks, on two calls in a row each, that its results equal those of the entry
point with a caller-provided workspace (the same kernels: bit for bit) and
match the fp64 oracle within the tolerances the other parity tests use:
  - bf16 cache, more than 8 splits (the array holds counters and partials);
  - E4M3 cache, fp8 dots, 16 heads, 16 splits (the same, E4M3 path);
  - E4M3 cache, fp8 dots, 128 heads, D_qk = 576 (the array holds the
    quantized q of the 128-head kernel at its single split; with more rows
    than CTA pairs the call runs one pair per row, whose q fits);
  - calls that need no workspace, including 128 heads with bf16 dots and
    calls that follow ones that used the array with another shape;
and that a call needing more than the array (the 128-row, 128-head fp8 call)
is refused. The file is collected last so that a run stopping at the first
failure has already run every other test; it also passes on its own in a
fresh process.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import parity
from parity import DEV, TOL_BF16, TOL_FP8_MIRROR, compare
from sparse_mla_attention_04_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

SCRATCH = 8 << 20


def _call_no_alloc(q, cache, kvs, idx, scale, dot, num_splits, D_v=512):
    T, H, D_qk = q.shape
    out = torch.full((T, H, D_v), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((T, H), float("nan"), dtype=torch.float32, device=DEV)
    kv_dtype = binding.SMLA_KV_FP8_E4M3 if cache.element_size() == 1 else binding.SMLA_KV_BF16
    st = binding.lib().sparse_mla_fwd_no_alloc(
        q.data_ptr(), cache.data_ptr(), kv_dtype, None if kvs is None else kvs.data_ptr(), idx.data_ptr(), T, H,
        D_qk, D_v, cache.shape[0], idx.shape[1], float(scale), binding._DOT[dot], out.data_ptr(), lse.data_ptr(),
        num_splits, torch.cuda.current_stream().cuda_stream)
    return st, out, lse


def _case(w, dot, num_splits, seed):
    """One call through each entry point on the same seeded inputs; both
    against the oracle (the fp8-dots path against the oracle that quantizes q
    the way the kernel does)."""
    w.seed = seed
    q = inputs.make_q(w)
    src = inputs.make_kv_source(w)
    idx = inputs.make_indices(w)
    cache, kvs = parity.gpu_cache(src.to(DEV), w.kv_fp8)
    qd, idd = q.to(DEV), torch.from_numpy(idx).to(DEV)
    o_ref, l_ref = binding.sparse_mla_fwd(qd, cache, idd, w.scale, kv_scale=kvs, dot_precision=dot,
                                          num_splits=num_splits, D_v=w.D_v)
    st, o_new, l_new = _call_no_alloc(qd, cache, kvs, idd, w.scale, dot, num_splits, w.D_v)
    assert st == binding.SMLA_OK, binding.status_string(st)
    torch.cuda.synchronize()
    assert torch.equal(o_new, o_ref) and torch.equal(l_new, l_ref), "differs from sparse_mla_fwd"
    ocache, oscale = parity.oracle_cache(src, w.kv_fp8)
    qm = 1 if dot == "fp8" else 0
    ro, rl, _ = oracle.sparse_mla(q, ocache, idx, w.scale, kv_fp8=w.kv_fp8, kv_scale=oscale, D_v=w.D_v, q_mode=qm)
    tol = TOL_FP8_MIRROR if dot == "fp8" else TOL_BF16
    compare(o_new.float().cpu().numpy().astype(np.float64), l_new.cpu().numpy().astype(np.float64), ro, rl, tol,
            "%s no_alloc (%s dots, %d splits)" % (w.name, dot, num_splits))


def _need(w, dot, num_splits):
    return binding.sparse_mla_fwd_ex_workspace_size(w.T, w.H, w.D_qk, w.D_v, w.topk, int(w.kv_fp8),
                                                    dot_precision=dot, num_splits=num_splits)


@pytest.mark.parametrize("num_splits", [16, 12, 0])
def test_no_alloc_bf16_many_splits(num_splits):
    w = inputs.Workload("noalloc_bf16", 4, 16, 512, 512, 6000, 2048, False, 1 / math.sqrt(512), "uniform")
    if num_splits:
        assert 0 < _need(w, "auto", num_splits) <= SCRATCH
    for seed in (41, 42):  # two calls in a row share the static array
        _case(w, "auto", num_splits, seed)


def test_no_alloc_fp8_dots_16_heads_many_splits():
    w = inputs.Workload("noalloc_fp8", 3, 16, 512, 512, 6000, 2048, True, 1 / math.sqrt(512), "uniform")
    assert 0 < _need(w, "fp8", 16) <= SCRATCH
    for seed in (43, 44):
        _case(w, "fp8", 16, seed)


def test_no_alloc_128_heads_fp8_dots():
    """The 128-head E4M3 kernel keeps its quantized q in the array at its one
    split: 4 rows x 128 heads need about 313 KB."""
    w = inputs.Workload("noalloc_wide", 4, 128, 576, 512, 5000, 700, True, 1 / math.sqrt(576), "uniform")
    need = _need(w, "fp8", 0)
    assert 0 < need <= SCRATCH
    for seed in (45, 46):
        _case(w, "fp8", 0, seed)


def test_no_alloc_128_heads_more_rows_than_pairs():
    """80 rows x 128 heads with fp8 dots: the automatic plan spreads the rows
    over CTA pairs and would keep partials of shared rows (more than the
    array holds); the entry point then runs one CTA pair per row, whose
    quantized q (5.9 MB) fits. Bit-identical to the forward asked for that
    plan, and within tolerance of the oracle."""
    w = inputs.Workload("noalloc_wide80", 80, 128, 576, 512, 4000, 256, True, 1 / math.sqrt(576), "uniform", seed=48)
    assert _need(w, "fp8", 0) > SCRATCH
    assert 0 < binding.sparse_mla_fwd_ex_workspace_size(w.T, w.H, w.D_qk, w.D_v, w.topk, 1, dot_precision="fp8",
                                                         num_splits=0, kernel="basic") <= SCRATCH
    q = inputs.make_q(w)
    src = inputs.make_kv_source(w)
    idx = inputs.make_indices(w)
    cache, kvs = parity.gpu_cache(src.to(DEV), True)
    qd, idd = q.to(DEV), torch.from_numpy(idx).to(DEV)
    for _ in range(2):  # two calls in a row through the static array
        st, o_new, l_new = _call_no_alloc(qd, cache, kvs, idd, w.scale, "fp8", 0)
        assert st == binding.SMLA_OK, binding.status_string(st)
        o_ref, l_ref = binding.sparse_mla_fwd(qd, cache, idd, w.scale, kv_scale=kvs, dot_precision="fp8",
                                              kernel="basic")
        torch.cuda.synchronize()
        assert torch.equal(o_new, o_ref) and torch.equal(l_new, l_ref)
    ocache, oscale = parity.oracle_cache(src, True)
    ro, rl, _ = oracle.sparse_mla(q, ocache, idx, w.scale, kv_fp8=True, kv_scale=oscale, q_mode=1)
    compare(o_new.float().cpu().numpy().astype(np.float64), l_new.cpu().numpy().astype(np.float64), ro, rl,
            TOL_FP8_MIRROR, "no_alloc, 128 heads, one pair per row")
    assert binding.smla_device_error() == 0


def test_no_alloc_calls_without_workspace_after_ones_with():
    """A varied sequence: calls that use the array, then calls of other
    shapes that need none (16 heads with 8 splits; 128 heads with bf16 dots,
    which run on the warp-MMA kernel), then the array again."""
    seq = [
        (inputs.Workload("s_bf16_16", 2, 16, 512, 512, 5000, 1500, False, 0.05, "uniform"), "auto", 16),
        (inputs.Workload("s_bf16_8", 3, 16, 512, 512, 5000, 1500, False, 0.05, "uniform"), "auto", 8),
        (inputs.Workload("s_wide_bf16dots", 8, 128, 576, 512, 4000, 256, True, 1 / math.sqrt(576), "uniform"),
         "auto", 0),
        (inputs.Workload("s_wide_fp8", 2, 128, 576, 512, 4000, 300, True, 1 / math.sqrt(576), "uniform"), "fp8", 0),
        (inputs.Workload("s_bf16_2", 5, 16, 512, 512, 5000, 700, False, 0.05, "uniform"), "auto", 2),
        (inputs.Workload("s_fp8_12", 2, 16, 512, 512, 5000, 1500, True, 0.05, "uniform"), "fp8", 12),
    ]
    for i, (w, dot, S) in enumerate(seq):
        _case(w, dot, S, 50 + i)


def test_no_alloc_128_head_rows_beyond_the_array_are_refused():
    """128 rows x 128 heads with fp8 dots need 9.5 MB of quantized q, more than
    the 8 MiB array: refused with SMLA_ERR_WORKSPACE_TOO_SMALL, nothing
    written. The same call with bf16 dots needs no workspace and runs."""
    T, H, topk = 128, 128, 64
    w = inputs.Workload("noalloc_big", T, H, 576, 512, 4000, topk, True, 1 / math.sqrt(576), "uniform", seed=47)
    assert _need(w, "fp8", 0) > SCRATCH
    assert _need(w, "auto", 0) == 0
    q = inputs.make_q(w).to(DEV)
    src = inputs.make_kv_source(w).to(DEV)
    cache, kvs = binding.build_fp8_cache(src)
    idx = torch.from_numpy(inputs.make_indices(w)).to(DEV)
    st, out, _ = _call_no_alloc(q, cache, kvs, idx, w.scale, "fp8", 0)
    torch.cuda.synchronize()
    assert st == binding.SMLA_ERR_WORKSPACE_TOO_SMALL
    assert torch.isnan(out.float()).all()
    st, out, lse = _call_no_alloc(q, cache, kvs, idx, w.scale, "auto", 0)
    assert st == binding.SMLA_OK, binding.status_string(st)
    o_ref, l_ref = binding.sparse_mla_fwd(q, cache, idx, w.scale, kv_scale=kvs, dot_precision="auto")
    torch.cuda.synchronize()
    assert torch.equal(out, o_ref) and torch.equal(lse, l_ref)


def test_no_alloc_rejects_oversized_workspace():
    """A call whose split partials would exceed the static array returns
    SMLA_ERR_WORKSPACE_TOO_SMALL and launches nothing."""
    T, H, topk, S = 64, 16, 4096, 64          # partials alone: 64*64*16*512*2 B = 64 MiB
    need = binding.sparse_mla_fwd_workspace_size(T, H, 512, 512, topk, binding.SMLA_KV_BF16, S)
    assert need > SCRATCH
    q = torch.zeros((T, H, 512), dtype=torch.bfloat16, device=DEV)
    kv = torch.zeros((16, 512), dtype=torch.bfloat16, device=DEV)
    idx = torch.zeros((T, topk), dtype=torch.int32, device=DEV)
    out = torch.zeros((T, H, 512), dtype=torch.bfloat16, device=DEV)
    st = binding.lib().sparse_mla_fwd_no_alloc(
        q.data_ptr(), kv.data_ptr(), binding.SMLA_KV_BF16, None, idx.data_ptr(), T, H, 512, 512, 16, topk, 0.1,
        binding.SMLA_DOT_AUTO, out.data_ptr(), None, S, None)
    assert st == binding.SMLA_ERR_WORKSPACE_TOO_SMALL
