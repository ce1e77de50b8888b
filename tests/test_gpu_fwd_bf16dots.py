"""bf16 dots over an E4M3 cache (GPU): q stays bf16 and is dotted with the
cache values code * kv_scale. With 16 heads this runs on the tcgen05 16-head
kernel (the gathered E4M3 rows expanded exactly to binary16, q brought into
binary16 by a per-head power of two) and, asked for explicitly, on the
warp-MMA kernel; both are held to the same bar.

Source: "Enable AITER sparse MLA on gfx942, including FP8 KV", Details
("Numerics": BF16 dots are at 0.2-0.3% of an FP32 reference; a BF16-dots
option). Held to the bf16 tolerance (rel-L2 <= 5e-3, max-abs <= 2e-2,
lse <= 1e-2) against the oracle with q unquantized and the same codes.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import parity
from parity import DEV, TOL_BF16, compare
from sparse_mla_attention_04_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["auto", "mma"])
def kernel(request):
    return request.param


def _run(w, *, num_splits=0, idx=None, dot="bf16", kernel="auto", q=None):
    q = inputs.make_q(w) if q is None else q
    src = inputs.make_kv_source(w)
    cache, kvs = binding.build_fp8_cache(src.to(DEV))
    ocache, oscale = parity.oracle_cache(src, True)
    idx = inputs.make_indices(w) if idx is None else idx
    out, lse = binding.sparse_mla_fwd(q.to(DEV), cache, torch.from_numpy(idx).to(DEV), w.scale, kv_scale=kvs,
                                      dot_precision=dot, D_v=w.D_v, num_splits=num_splits, kernel=kernel)
    torch.cuda.synchronize()
    ref_o, ref_l, _ = oracle.sparse_mla(q, ocache, idx, w.scale, kv_fp8=True, kv_scale=oscale, D_v=w.D_v)
    got_o = out.float().cpu().numpy().astype(np.float64)
    got_l = lse.cpu().numpy().astype(np.float64)
    res = compare(got_o, got_l, ref_o, ref_l, TOL_BF16, w.name + " (bf16 dots)")
    assert binding.smla_device_error() == 0
    return res, got_o, got_l


def test_bf16_dots_decode_16_heads(kernel):
    w = inputs.decode(n_seqs=8, ctx=8192, topk=2048, fp8=True, short_rows=2, name="decode_fp8_bf16dots")
    res, _, _ = _run(w, kernel=kernel)
    # the pages' figure for bf16 dots is 0.2-0.3% on model data; quantizing q costs far more
    assert res["rel"] < 3e-3


@pytest.mark.parametrize("splits", [1, 3, 12])
def test_bf16_dots_splits(splits, kernel):
    w = inputs.decode(n_seqs=4, ctx=8192, topk=2048, fp8=True, name="decode_fp8_bf16dots_splits")
    _run(w, num_splits=splits, kernel=kernel)


def test_bf16_dots_auto_splits_small_batch(kernel):
    """Automatic splits for a small batch stay within the cluster merge."""
    w = inputs.decode(n_seqs=2, ctx=8192, topk=2048, fp8=True, name="decode_fp8_bf16dots_t2")
    _run(w, kernel=kernel)


def test_bf16_dots_q_magnitudes(kernel):
    """q heads whose magnitudes span far beyond binary16's range (1e-30 ..
    1e30, and an all-zero head): the tcgen05 kernel rescales each head by a
    power of two into binary16 and undoes it in the logits, so the bar is the
    same as for ordinary q."""
    w = inputs.decode(n_seqs=3, ctx=4096, topk=512, fp8=True, name="decode_fp8_bf16dots_mag")
    q = inputs.make_q(w).float()
    for h, f in enumerate([1e-30, 1e30, 1e-12, 1e12, 0.0, 3e-5, 7e4, 1.0]):
        q[:, h] *= f
    # a huge q makes the softmax one-hot: keep the logits finite and moderate
    scale = 1.0 / (np.sqrt(512) * 1e30)
    _run(dataclasses.replace(w, scale=scale), q=q.to(torch.bfloat16), kernel=kernel)


def test_bf16_dots_wide_128_heads():
    w = inputs.wide(T=3, ctx=4096, topk=2048, name="wide_bf16dots")
    _run(w)


def test_bf16_dots_ragged_and_auto_is_bf16(kernel):
    w = inputs.decode(n_seqs=5, ctx=4096, topk=700, fp8=True, name="decode_fp8_bf16dots_ragged")
    idx = inputs.make_indices(w)
    idx[1, :] = -1
    idx[3, 50:] = -1
    _, o1, l1 = _run(w, idx=idx, dot="bf16", kernel=kernel)
    _, o2, l2 = _run(w, idx=idx, dot="auto", kernel=kernel)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
