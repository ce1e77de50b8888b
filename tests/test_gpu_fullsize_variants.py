"""The precision variants, attention sinks and the fused producer step at the
benchmark's full sizes, in the launch configuration the benchmark times
(automatic split plan), checked on sampled rows (GPU).

As in the base full-size tests, the oracle sees only what it derives itself:
the per-tensor kv scale from the whole bf16 source (chunked amax), the E4M3
codes of the gathered rows from its own encoder (the GPU cache rows must equal
them), and q's E4M3 codes from its own quantizer (fed to both sides).
"""
import numpy as np
import pytest
import torch

import oracle
from parity import DEV, TOL_BF16, TOL_FP8_MIRROR, compare
from sparse_mla_attention_04_gb300 import binding, inputs
from test_gpu_fullsize import oracle_scale_of

pytestmark = pytest.mark.gpu


def _gathered(src_dev, cache_dev, kvs_dev, idx_np, rows, fp8):
    """The sampled rows' dense renumbering and the oracle's rows for them."""
    sel = idx_np[rows]
    uniq = np.unique(sel[sel >= 0])
    remap = np.where(sel >= 0, np.searchsorted(uniq, np.maximum(sel, 0)), -1).astype(np.int32)
    src_rows = src_dev[torch.from_numpy(uniq).to(DEV)].cpu()
    if not fp8:
        return remap, src_rows, None
    s = oracle_scale_of(src_dev)
    assert np.float32(kvs_dev.item()) == s, "per-tensor scale differs from the oracle's"
    codes = oracle.fp8_quantize(src_rows, s)
    assert (cache_dev[torch.from_numpy(uniq).to(DEV)].cpu().numpy() == codes).all()
    return remap, codes, s


def _short_rows(w, idx_np, n=2):
    return [t for t in range(w.T) if (idx_np[t] == -1).any()][:n]


@pytest.mark.parametrize("wl", ["decode_fp8", "wide_fp8"])
def test_prequantized_q_full(wl):
    """sparse_mla_fwd_q8: q as E4M3 codes with one per-tensor scale."""
    w = inputs.CONFIGS[wl]()
    idx_np = inputs.make_indices(w)
    q = inputs.make_q(w)                                   # host bf16
    T, H, D = q.shape
    qs = oracle.fp8_scale(q)
    codes = oracle.fp8_quantize(q.reshape(-1, D), qs).reshape(T, H, D)
    src = inputs.make_kv_source(w, device=DEV)
    cache, kvs = binding.build_fp8_cache(src)
    out, lse = binding.sparse_mla_fwd_q8(torch.from_numpy(codes).to(DEV),
                                         torch.tensor([qs], dtype=torch.float32, device=DEV), cache,
                                         torch.from_numpy(idx_np).to(DEV), w.scale, kv_scale=kvs, D_v=w.D_v)
    torch.cuda.synchronize()
    rows = [0, w.T - 1] + _short_rows(w, idx_np)
    remap, ocodes, s = _gathered(src, cache, kvs, idx_np, rows, True)
    ro, rl, _ = oracle.sparse_mla_q8(codes[rows], qs, ocodes, remap, w.scale, kv_fp8=True, kv_scale=float(s),
                                     D_v=w.D_v)
    print(compare(out[rows].float().cpu().numpy().astype(np.float64), lse[rows].cpu().numpy().astype(np.float64),
                  ro, rl, TOL_FP8_MIRROR, w.name + " (pre-quantized q)"))


def test_decode_bf16_sinks_full():
    w = inputs.decode_bf16()
    idx_np = inputs.make_indices(w)
    q = inputs.make_q(w, device=DEV)
    src = inputs.make_kv_source(w, device=DEV)
    g = np.random.default_rng(11)
    sk = g.uniform(-2.0, 4.0, w.H).astype(np.float32)
    sk[::5] = -np.inf           # some heads have no sink
    sk[1] = 30.0                # one sink dominates its head
    sinks = torch.from_numpy(sk)
    out, lse = binding.sparse_mla_fwd(q, src, torch.from_numpy(idx_np).to(DEV), w.scale, D_v=w.D_v,
                                      sinks=sinks.to(DEV))
    torch.cuda.synchronize()
    rows = [0, 1, 31, 63]
    remap, src_rows, _ = _gathered(src, None, None, idx_np, rows, False)
    ro, rl, _ = oracle.sparse_mla(q[rows].cpu(), src_rows, remap, w.scale, D_v=w.D_v, sinks=sinks.numpy())
    print(compare(out[rows].float().cpu().numpy().astype(np.float64), lse[rows].cpu().numpy().astype(np.float64),
                  ro, rl, TOL_BF16, w.name + " (sinks)"))


def test_decode_fp8_bf16_dots_full():
    """bf16 q dotted with the E4M3 cache values code * kv_scale."""
    w = inputs.decode_fp8()
    idx_np = inputs.make_indices(w)
    q = inputs.make_q(w, device=DEV)
    src = inputs.make_kv_source(w, device=DEV)
    cache, kvs = binding.build_fp8_cache(src)
    out, lse = binding.sparse_mla_fwd(q, cache, torch.from_numpy(idx_np).to(DEV), w.scale, kv_scale=kvs,
                                      dot_precision="bf16", D_v=w.D_v)
    torch.cuda.synchronize()
    rows = [0, 40] + _short_rows(w, idx_np)
    remap, ocodes, s = _gathered(src, cache, kvs, idx_np, rows, True)
    ro, rl, _ = oracle.sparse_mla(q[rows].cpu(), ocodes, remap, w.scale, kv_fp8=True, kv_scale=float(s),
                                  D_v=w.D_v)
    print(compare(out[rows].float().cpu().numpy().astype(np.float64), lse[rows].cpu().numpy().astype(np.float64),
                  ro, rl, TOL_BF16, w.name + " (bf16 dots)"))


def test_fused_producer_full():
    """4096 tokens x 128 heads with E4M3 q_out and cache, the benchmark's
    inputs; sampled tokens bit for bit against the oracle's binary32 mirror."""
    T, H, P = 4096, 128, 8192
    q_scale, kv_scale = np.float32(0.0137), np.float32(0.0211)
    ql, qp, kc, kp, pos, slots, ns = inputs.producer_inputs(T, H, 1, P, num_slots=2 * T)
    cs = inputs.rope_cos_sin_cache(P)
    cache = torch.zeros((ns, 576), dtype=torch.uint8, device=DEV)
    q_out = binding.smla_fused_qk_rope_cache(
        ql.to(DEV), qp.to(DEV), kc.to(DEV), kp.to(DEV), pos.to(DEV), cs.to(DEV), slots.to(DEV), cache,
        is_neox=True, kv_scale=torch.tensor([kv_scale], device=DEV), q_out_fp8=True,
        q_scale=torch.tensor([q_scale], device=DEV))
    torch.cuda.synchronize()
    assert binding.smla_device_error() == 0
    toks = [0, 1, 2047, 4095]
    ref_cache = np.zeros((ns, 576), dtype=np.uint8)
    ref_q, bad = oracle.fused_qk_rope_cache(ql[toks], qp[toks], kc[toks], kp[toks], pos[toks], cs, True,
                                            slots[toks], ref_cache, cache_fp8=True, kv_scale=kv_scale,
                                            q_out_fp8=True, q_scale=q_scale, mode=1)
    assert bad == 0
    assert np.array_equal(q_out[toks].cpu().numpy(), ref_q)
    written = [int(s) for s in slots[toks] if s >= 0]
    assert written, "the sample writes at least one cache row"
    assert np.array_equal(cache[written].cpu().numpy(), ref_cache[written])
