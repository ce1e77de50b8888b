"""Helpers of the GPU parity tests: run the CUDA path through the C ABI and
the fp64 oracle on the same seeded inputs, and compare.

Tolerances (the accuracy targets of the forward, fixed here):
  bf16 cache              : rel-L2 <= 5e-3, max-abs <= 2e-2, lse abs <= 1e-2
  fp8 dots vs the oracle on the dequantized values the kernel uses (q8 * s_q,
    code * kv_scale; q_mode=1): rel-L2 <= 5e-3, max-abs <= 2e-2, lse <= 1e-2
  fp8 dots vs the oracle with q unquantized: rel-L2 <= 3e-2
  index handling (masks, empty rows, poison): bit-exact.
rel-L2 is global over the compared tensor; -inf lse entries must coincide.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from sparse_mla_attention_04_gb300 import binding, inputs

TOL_BF16 = dict(rel=5e-3, max_abs=2e-2, lse=1e-2)
# fp8 dots: the oracle on the dequantized values the kernel computes with
# (q8 * s_q and code * kv_scale) is held to the bf16 figures; the oracle that
# keeps q unquantized is held to the rel-L2 envelope of fp8 dots (the pages
# report 3.4-4.5% on model data; bound 3e-2 here), lse not compared (with a
# handful of keys, quantizing q alone moves lse by more than 1e-2).
TOL_FP8_MIRROR = dict(rel=5e-3, max_abs=2e-2, lse=1e-2)
TOL_FP8 = dict(rel=3e-2, max_abs=None, lse=None)

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


def gpu_cache(kv_src_dev: torch.Tensor, fp8: bool):
    """The cache the kernel reads, built by the library's own companion kernels."""
    if not fp8:
        return kv_src_dev, None
    return binding.build_fp8_cache(kv_src_dev)


def oracle_cache(kv_src_cpu: torch.Tensor, fp8: bool):
    """The oracle's own cache: its scale and its E4M3 codes of the same bf16 source."""
    if not fp8:
        return kv_src_cpu, 1.0
    s = oracle.fp8_scale(kv_src_cpu)
    return oracle.fp8_quantize(kv_src_cpu, s), float(s)


def fwd(kernel, *args, **kw):
    """binding.sparse_mla_fwd on the named kernel ("auto" or "mma")."""
    return binding.sparse_mla_fwd(*args, kernel=kernel, **kw)


def fwd_q8(kernel, *args, **kw):
    """binding.sparse_mla_fwd_q8 on the named kernel ("auto" or "mma")."""
    return binding.sparse_mla_fwd_q8(*args, kernel=kernel, **kw)


def run_gpu(q, cache, kvs, idx, scale, *, fp8: bool, num_splits: int = 0, D_v: int = 512, kernel: str = "auto"):
    dot = "fp8" if fp8 else "auto"
    out, lse = binding.sparse_mla_fwd(q, cache, idx, scale, kv_scale=kvs, dot_precision=dot, D_v=D_v,
                                      num_splits=num_splits, kernel=kernel)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def compare(out, lse, ref_o, ref_l, tol, what=""):
    """Assert the tolerance; return the measured figures."""
    ninf_g, ninf_r = np.isneginf(lse), np.isneginf(ref_l)
    assert (ninf_g == ninf_r).all(), "%s: -inf lse pattern differs" % what
    fin = ~ninf_r
    # rows with no valid index must be exactly zero
    empty = ninf_r
    if empty.any():
        assert (out[empty] == 0).all(), "%s: empty rows not zero" % what
    diff = out - ref_o
    nref = np.linalg.norm(ref_o)
    rel = float(np.linalg.norm(diff) / nref) if nref > 0 else float(np.linalg.norm(diff))
    mab = float(np.abs(diff).max()) if diff.size else 0.0
    lab = float(np.abs(lse[fin] - ref_l[fin]).max()) if fin.any() else 0.0
    assert np.isfinite(out).all(), "%s: non-finite output" % what
    assert rel <= tol["rel"], "%s: rel-L2 %.3e > %.1e" % (what, rel, tol["rel"])
    if tol["max_abs"] is not None:
        assert mab <= tol["max_abs"], "%s: max-abs %.3e > %.1e" % (what, mab, tol["max_abs"])
    if tol["lse"] is not None:
        assert lab <= tol["lse"], "%s: lse abs %.3e > %.1e" % (what, lab, tol["lse"])
    return dict(rel=rel, max_abs=mab, lse_abs=lab)


def case(w: inputs.Workload, *, num_splits=0, idx=None, kv_src=None, q=None, check_mirror=True,
         check_plain=True, kernel: str = "auto"):
    """Run workload `w` (small enough for the whole-pool oracle) on both sides.

    For an E4M3 cache the plain comparison (oracle with unquantized q, the
    fp8 tolerance) measures the method's error and the mirrored one (oracle
    quantizing q the same way, the bf16-level tolerance) the kernel's
    arithmetic; `check_plain=False` keeps only the latter, for inputs built
    to stress the kernel rather than to look like a workload."""
    q = inputs.make_q(w) if q is None else q
    kv_src = inputs.make_kv_source(w) if kv_src is None else kv_src
    idx = inputs.make_indices(w) if idx is None else idx
    cache, kvs = gpu_cache(kv_src.to(DEV), w.kv_fp8)
    out, lse = run_gpu(q.to(DEV), cache, kvs, torch.from_numpy(idx).to(DEV), w.scale,
                       fp8=w.kv_fp8, num_splits=num_splits, D_v=w.D_v, kernel=kernel)
    ocache, oscale = oracle_cache(kv_src, w.kv_fp8)
    ref_o, ref_l, _ = oracle.sparse_mla(q, ocache, idx, w.scale, kv_fp8=w.kv_fp8, kv_scale=oscale, D_v=w.D_v)
    res = {}
    if check_plain or not w.kv_fp8:
        res = compare(out, lse, ref_o, ref_l, TOL_FP8 if w.kv_fp8 else TOL_BF16, w.name)
    if w.kv_fp8 and check_mirror:
        mo, ml, _ = oracle.sparse_mla(q, ocache, idx, w.scale, kv_fp8=True, kv_scale=oscale, D_v=w.D_v, q_mode=1)
        res["mirror"] = compare(out, lse, mo, ml, TOL_FP8_MIRROR, w.name + " (q quantized)")
    return res, out, lse
