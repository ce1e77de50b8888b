"""The forward with a pre-quantized q (E4M3 codes and one per-tensor scale)
against the oracle fed the same codes (GPU).

Source: "Enable AITER sparse MLA on gfx942, including FP8 KV", Details ("FP8
KV on gfx942": gfx950 keeps the pre-quantized q). q enters the dots as
code * q_scale on both sides, so the kernel is held to the tolerance of the
fp8-dot mirror comparison (rel-L2 <= 5e-3, max-abs <= 2e-2, lse <= 1e-2).
Also the chain the fused producer feeds: its E4M3 q_out into this forward.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
from parity import DEV, TOL_FP8_MIRROR, compare
from sparse_mla_attention_04_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["tcgen05", "mma", "basic"])
def kernel(request):
    """The kernel a test runs on: the library's own choice, the warp-MMA
    kernel, or the tcgen05 kernels that take a whole SM per CTA (asked for
    through the forward's kernel-choice field)."""
    return {"tcgen05": "auto", "mma": "mma", "basic": "basic"}[request.param]


def _run(w, q_scale, *, num_splits=0, idx=None, kernel="auto"):
    q = inputs.make_q(w)
    T, H, D = q.shape
    codes = oracle.fp8_quantize(q.reshape(-1, D), q_scale).reshape(T, H, D)   # the pinned quantizer
    src = inputs.make_kv_source(w)
    cache, kvs = binding.build_fp8_cache(src.to(DEV))
    ocache, oscale = parity.oracle_cache(src, True)
    idx = inputs.make_indices(w) if idx is None else idx
    out, lse = binding.sparse_mla_fwd_q8(torch.from_numpy(codes).to(DEV),
                                         torch.tensor([q_scale], dtype=torch.float32, device=DEV), cache,
                                         torch.from_numpy(idx).to(DEV), w.scale, kv_scale=kvs, D_v=w.D_v,
                                         num_splits=num_splits, kernel=kernel)
    torch.cuda.synchronize()
    ref_o, ref_l, _ = oracle.sparse_mla_q8(codes, q_scale, ocache, idx, w.scale, kv_fp8=True, kv_scale=oscale,
                                           D_v=w.D_v)
    return compare(out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
                   ref_o, ref_l, TOL_FP8_MIRROR, w.name + " (pre-quantized q)")


def test_q8_decode_16_heads(kernel):
    w = inputs.decode(n_seqs=8, ctx=8192, topk=2048, fp8=True, short_rows=2, name="decode_fp8_q8")
    _run(w, np.float32(0.0137), kernel=kernel)


def test_q8_decode_splits(kernel):
    w = inputs.decode(n_seqs=4, ctx=8192, topk=2048, fp8=True, name="decode_fp8_q8_splits")
    for s in (1, 3, 12):
        _run(w, np.float32(0.011), num_splits=s, kernel=kernel)


def test_q8_wide_128_heads(kernel):
    w = inputs.wide(T=4, ctx=4096, topk=2048, name="wide_q8")
    _run(w, np.float32(0.0093), kernel=kernel)


def test_q8_ragged_and_masked():
    w = inputs.decode(n_seqs=5, ctx=4096, topk=700, fp8=True, name="decode_fp8_q8_ragged")
    idx = inputs.make_indices(w)
    idx[1, :] = -1            # an empty row
    idx[2, 100:] = -1         # a short row
    _run(w, np.float32(0.02), idx=idx)


def test_q8_chain_from_the_fused_producer():
    """The fused producer's E4M3 q_out (q = concat(ql_nope, RoPE(q_pe)) / q_scale)
    fed to the forward, against the oracle chain on the same inputs."""
    T, H, P = 6, 128, 4096
    ql, qp, kc, kp, pos, _, _ = inputs.producer_inputs(T, H, 31, P)
    cs = inputs.rope_cos_sin_cache(P)
    q_scale = np.float32(0.0137)
    # the cache the forward reads: a wide-head E4M3 pool
    w = inputs.wide(T=T, ctx=2048, topk=1024, name="wide_chain")
    src = inputs.make_kv_source(w)
    cache, kvs = binding.build_fp8_cache(src.to(DEV))
    ocache, oscale = parity.oracle_cache(src, True)
    idx = inputs.make_indices(w)
    # producer on the GPU (no cache rows: slots -1), then the forward
    no_slots = torch.full((T,), -1, dtype=torch.int64)
    q8 = binding.smla_fused_qk_rope_cache(
        ql.to(DEV), qp.to(DEV), kc.to(DEV), kp.to(DEV), pos.to(DEV), cs.to(DEV), no_slots.to(DEV),
        torch.zeros((1, 576), dtype=torch.uint8, device=DEV), kv_scale=torch.tensor([1.0], device=DEV),
        q_out_fp8=True, q_scale=torch.tensor([q_scale], device=DEV))
    out, lse = binding.sparse_mla_fwd_q8(q8, torch.tensor([q_scale], device=DEV), cache,
                                         torch.from_numpy(idx).to(DEV), w.scale, kv_scale=kvs)
    torch.cuda.synchronize()
    # the oracle chain
    ref_q8, bad = oracle.fused_qk_rope_cache(ql, qp, kc, kp, pos, cs, True, no_slots.numpy(),
                                             np.zeros((1, 576), dtype=np.uint8), cache_fp8=True,
                                             q_out_fp8=True, q_scale=q_scale, mode=1)
    assert bad == 0
    assert np.array_equal(q8.cpu().numpy(), ref_q8)
    ref_o, ref_l, _ = oracle.sparse_mla_q8(ref_q8, q_scale, ocache, idx, w.scale, kv_fp8=True, kv_scale=oscale)
    compare(out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), ref_o, ref_l,
            TOL_FP8_MIRROR, "producer -> forward (pre-quantized q)")


def test_q8_argument_errors():
    w = inputs.tiny()
    q8 = torch.zeros((w.T, w.H, w.D_qk), dtype=torch.uint8, device=DEV)
    cache = torch.zeros((w.num_slots, w.D_qk), dtype=torch.uint8, device=DEV)
    idx = torch.zeros((w.T, w.topk), dtype=torch.int32, device=DEV)
    one = torch.ones(1, dtype=torch.float32, device=DEV)
    L = binding.lib()
    st = L.sparse_mla_fwd_q8(q8.data_ptr(), None, cache.data_ptr(), one.data_ptr(), idx.data_ptr(), w.T, w.H,
                             w.D_qk, w.D_v, w.num_slots, w.topk, 0.1, torch.empty(1, device=DEV).data_ptr(), None,
                             None, 0, 0, None)
    assert st == binding.SMLA_ERR_NULL_POINTER   # no q_scale
