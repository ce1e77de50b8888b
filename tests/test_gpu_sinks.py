"""Attention sinks on the GPU: a per-head sink logit in the softmax
denominator, against the oracle with the same sinks.

Source: "Enable AITER sparse MLA on gfx942, including FP8 KV", Limitations
(sinks are passed through). Reading: out = sum_i e^{s_i} v_i / (e^{sink_h} +
sum_j e^{s_j}), lse = log(e^{sink_h} + sum_j e^{s_j}); an empty row gives
out = 0 and lse = sink_h. Covered: one split (epilogue), up to 8 (cluster
merge), more (workspace merge), both 16-head kernels, the 128-head kernel,
and a pre-quantized q.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
from parity import DEV, TOL_BF16, TOL_FP8_MIRROR, compare
from sparse_mla_attention_04_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


def _sinks(H, seed):
    g = np.random.default_rng(seed)
    s = g.uniform(-2.0, 4.0, H).astype(np.float32)
    s[::5] = -np.inf            # some heads have none
    s[1] = 30.0                 # one sink dominates its head
    return s


@pytest.fixture(params=["tcgen05", "mma", "basic"])
def kernel(request):
    """The kernel a test runs on: the library's own choice, the warp-MMA
    kernel, or the tcgen05 kernels that take a whole SM per CTA (asked for
    through the forward's kernel-choice field)."""
    return {"tcgen05": "auto", "mma": "mma", "basic": "basic"}[request.param]


def _bf16_case(w, sinks, num_splits, idx=None, kernel="auto"):
    q = inputs.make_q(w)
    src = inputs.make_kv_source(w)
    idx = inputs.make_indices(w) if idx is None else idx
    out, lse = binding.sparse_mla_fwd(q.to(DEV), src.to(DEV), torch.from_numpy(idx).to(DEV), w.scale,
                                      D_v=w.D_v, num_splits=num_splits,
                                      sinks=torch.from_numpy(sinks).to(DEV), kernel=kernel)
    torch.cuda.synchronize()
    ref_o, ref_l, _ = oracle.sparse_mla(q, src, idx, w.scale, D_v=w.D_v, sinks=sinks)
    return (out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), ref_o, ref_l)


@pytest.mark.parametrize("splits", [1, 2, 12])
def test_sinks_decode_bf16(kernel, splits):
    w = inputs.decode(n_seqs=6, ctx=8192, topk=2048, name="decode_bf16_sinks")
    o, l, ro, rl = _bf16_case(w, _sinks(16, 1), splits, kernel=kernel)
    compare(o, l, ro, rl, TOL_BF16, "sinks, %d split(s)" % splits)


def test_sinks_empty_rows_give_the_sink(kernel):
    w = inputs.decode(n_seqs=4, ctx=4096, topk=256, name="decode_bf16_sinks_empty")
    idx = inputs.make_indices(w)
    idx[2, :] = -1
    sinks = _sinks(16, 2)
    for splits in (1, 3, 10):
        o, l, ro, rl = _bf16_case(w, sinks, splits, idx=idx, kernel=kernel)
        compare(o, l, ro, rl, TOL_BF16, "sinks, empty row")
        assert (o[2] == 0).all()
        fin = np.isfinite(sinks)
        np.testing.assert_allclose(l[2][fin], sinks[fin].astype(np.float64), rtol=0, atol=1e-6)
        assert np.isneginf(l[2][~fin]).all()


@pytest.mark.parametrize("T", [3, 80])
def test_sinks_wide_topk_zero_gives_the_sink(T):
    """128 heads, no keys: out = 0 and lse = the head's sink (or -inf)."""
    w = inputs.wide(T=T, ctx=4096, topk=1, name="wide_sinks_topk0")
    cache, kvs = binding.build_fp8_cache(inputs.make_kv_source(w).to(DEV))
    sinks = _sinks(128, 5)
    out, lse = binding.sparse_mla_fwd(inputs.make_q(w).to(DEV), cache, torch.empty((T, 0), dtype=torch.int32,
                                      device=DEV), w.scale, kv_scale=kvs, dot_precision="fp8",
                                      sinks=torch.from_numpy(sinks).to(DEV))
    torch.cuda.synchronize()
    assert (out == 0).all()
    want = np.broadcast_to(sinks.astype(np.float32), (T, 128))
    np.testing.assert_array_equal(lse.cpu().numpy(), want)


@pytest.mark.parametrize("T,topk", [(3, 2048), (80, 200), (160, 2048)])
def test_sinks_wide_128_heads(T, topk):
    w = inputs.wide(T=T, ctx=4096, topk=topk, name="wide_sinks")
    q = inputs.make_q(w)
    src = inputs.make_kv_source(w)
    cache, kvs = binding.build_fp8_cache(src.to(DEV))
    ocache, oscale = parity.oracle_cache(src, True)
    idx = inputs.make_indices(w)
    sinks = _sinks(128, 3)
    out, lse = binding.sparse_mla_fwd(q.to(DEV), cache, torch.from_numpy(idx).to(DEV), w.scale, kv_scale=kvs,
                                      dot_precision="fp8", sinks=torch.from_numpy(sinks).to(DEV))
    torch.cuda.synchronize()
    mo, ml, _ = oracle.sparse_mla(q, ocache, idx, w.scale, kv_fp8=True, kv_scale=oscale, q_mode=1, sinks=sinks)
    compare(out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), mo, ml,
            TOL_FP8_MIRROR, "wide, sinks (q quantized)")


def test_sinks_prequantized_q():
    w = inputs.decode(n_seqs=4, ctx=8192, topk=2048, fp8=True, name="decode_fp8_q8_sinks")
    q = inputs.make_q(w)
    T, H, D = q.shape
    q_scale = np.float32(0.0137)
    codes = oracle.fp8_quantize(q.reshape(-1, D), q_scale).reshape(T, H, D)
    src = inputs.make_kv_source(w)
    cache, kvs = binding.build_fp8_cache(src.to(DEV))
    ocache, oscale = parity.oracle_cache(src, True)
    idx = inputs.make_indices(w)
    sinks = _sinks(16, 4)
    out, lse = binding.sparse_mla_fwd_q8(torch.from_numpy(codes).to(DEV), torch.tensor([q_scale], device=DEV),
                                         cache, torch.from_numpy(idx).to(DEV), w.scale, kv_scale=kvs,
                                         sinks=torch.from_numpy(sinks).to(DEV))
    torch.cuda.synchronize()
    ro, rl, _ = oracle.sparse_mla_q8(codes, q_scale, ocache, idx, w.scale, kv_fp8=True, kv_scale=oscale, sinks=sinks)
    compare(out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), ro, rl,
            TOL_FP8_MIRROR, "pre-quantized q, sinks")


@pytest.mark.parametrize("kernel", ["auto", "mma"])
@pytest.mark.parametrize("splits", [1, 4, 10])
def test_sinks_bf16_dots_over_e4m3(kernel, splits):
    """bf16 dots over an E4M3 cache with sinks (the tcgen05 16-head kernel's
    bf16-dots mode, and the warp-MMA kernel), against the oracle with q
    unquantized and the same codes; an empty row gives the sink."""
    w = inputs.decode(n_seqs=4, ctx=8192, topk=2048, fp8=True, name="decode_fp8_bf16dots_sinks")
    q = inputs.make_q(w)
    src = inputs.make_kv_source(w)
    cache, kvs = binding.build_fp8_cache(src.to(DEV))
    ocache, oscale = parity.oracle_cache(src, True)
    idx = inputs.make_indices(w)
    idx[2, :] = -1
    sinks = _sinks(16, 6)
    out, lse = binding.sparse_mla_fwd(q.to(DEV), cache, torch.from_numpy(idx).to(DEV), w.scale, kv_scale=kvs,
                                      dot_precision="bf16", num_splits=splits,
                                      sinks=torch.from_numpy(sinks).to(DEV), kernel=kernel)
    torch.cuda.synchronize()
    ro, rl, _ = oracle.sparse_mla(q, ocache, idx, w.scale, kv_fp8=True, kv_scale=oscale, sinks=sinks)
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.cpu().numpy().astype(np.float64)
    compare(o, l, ro, rl, TOL_BF16, "bf16 dots over E4M3, sinks")
    assert (o[2] == 0).all()
    fin = np.isfinite(sinks)
    np.testing.assert_allclose(l[2][fin], sinks[fin].astype(np.float64), rtol=0, atol=1e-6)
    assert binding.smla_device_error() == 0


def test_no_sinks_through_ex_is_the_plain_forward():
    """sinks = -inf for every head equals the forward without sinks, bit for bit."""
    w = inputs.decode(n_seqs=4, ctx=8192, topk=2048, name="decode_bf16_nosink")
    q, src, idx = inputs.make_q(w).to(DEV), inputs.make_kv_source(w).to(DEV), torch.from_numpy(inputs.make_indices(w)).to(DEV)
    o1, l1 = binding.sparse_mla_fwd(q, src, idx, w.scale)
    o2, l2 = binding.sparse_mla_fwd(q, src, idx, w.scale, sinks=torch.full((16,), float("-inf"), device=DEV))
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
