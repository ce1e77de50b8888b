"""The fused producer step on the GPU (RoPE on q_pe / k_pe, q concat, cache
write) against the oracle's binary32 mirror, bit for bit, and against the
split chain (rotation, then the library's own fp8 cache write).

Source: "[ROCm][MLA][Perf] Fuse decode QK-RoPE + Q-concat + KV-concat +
KV-cache write for sparse MLA", Test plan: bf16 q_out == concat(ql_nope,
RoPE(q_pe)); fp8 q_out == scaled_fp8_quant(concat(...), q_scale) with a
non-unit q_scale; kv_cache == concat_and_cache_mla(kv_c, RoPE(k_pe)); a
non-contiguous (transposed) ql_nope.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import DEV
from sparse_mla_attention_04_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

Q_SCALE = np.float32(0.0137)
KV_SCALE = np.float32(0.0211)


def _bits(x: torch.Tensor) -> np.ndarray:
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _run_pair(T, H, neox, q_fp8, cache_fp8, *, seed=0, layout="contiguous", max_position=4096, skip_every=5):
    ql, qp, kc, kp, pos, slots, ns = inputs.producer_inputs(T, H, seed, max_position, skip_every=skip_every)
    cs = inputs.rope_cos_sin_cache(max_position)
    # the oracle (binary32 mirror: the precision the fp8 codes are decided in)
    ref_cache = np.full((ns, 576), 0xA5 if cache_fp8 else 0x7E7E, dtype=np.uint8 if cache_fp8 else np.uint16)
    ref_q, bad = oracle.fused_qk_rope_cache(ql, qp, kc, kp, pos, cs, neox, slots, ref_cache, cache_fp8=cache_fp8,
                                            kv_scale=KV_SCALE, q_out_fp8=q_fp8, q_scale=Q_SCALE, mode=1)
    assert bad == 0
    # the device inputs, in the requested layout
    if layout == "production":
        # ql_nope as the transpose of a [H, T, 512] buffer; q_pe, kv_c and k_pe as
        # column slices of wider rows
        ql_d = ql.transpose(0, 1).contiguous().to(DEV).transpose(0, 1)
        qwide = torch.empty((T, H, 128), dtype=torch.bfloat16, device=DEV)
        qwide[:, :, 32:96] = qp.to(DEV)
        qp_d = qwide[:, :, 32:96]
        kva = torch.empty((T, 576), dtype=torch.bfloat16, device=DEV)
        kva[:, :512] = kc.to(DEV)
        kva[:, 512:] = kp.to(DEV)
        kc_d, kp_d = kva[:, :512], kva[:, 512:]
        assert not ql_d.is_contiguous() and not qp_d.is_contiguous() and not kc_d.is_contiguous()
    else:
        ql_d, qp_d, kc_d, kp_d = ql.to(DEV), qp.to(DEV), kc.to(DEV), kp.to(DEV)
    cache = torch.from_numpy(np.full((ns, 576), 0xA5 if cache_fp8 else 0x7E7E,
                                     dtype=np.uint8 if cache_fp8 else np.uint16).view(
        np.uint8 if cache_fp8 else np.int16)).to(DEV)
    if not cache_fp8:
        cache = cache.view(torch.bfloat16)
    q_out = binding.smla_fused_qk_rope_cache(
        ql_d, qp_d, kc_d, kp_d, pos.to(DEV), cs.to(DEV), slots.to(DEV), cache, is_neox=neox,
        kv_scale=torch.tensor([KV_SCALE], device=DEV), q_out_fp8=q_fp8,
        q_scale=torch.tensor([Q_SCALE], device=DEV))
    torch.cuda.synchronize()
    got_q = q_out.cpu().numpy() if q_fp8 else _bits(q_out)
    got_c = cache.cpu().numpy() if cache_fp8 else _bits(cache)
    return got_q, got_c, ref_q, ref_cache, (ql, qp, kc, kp, pos, slots, cs, ns)


@pytest.mark.parametrize("neox", [True, False])
@pytest.mark.parametrize("q_fp8,cache_fp8", [(False, False), (False, True), (True, True), (True, False)])
@pytest.mark.parametrize("T,H", [(1, 16), (7, 16), (64, 128)])
def test_producer_bit_exact(T, H, neox, q_fp8, cache_fp8):
    binding.smla_device_error(reset=True)
    got_q, got_c, ref_q, ref_c, _ = _run_pair(T, H, neox, q_fp8, cache_fp8, seed=T * 31 + H)
    assert np.array_equal(got_q, ref_q)
    assert np.array_equal(got_c, ref_c)
    assert binding.smla_device_error() == 0


@pytest.mark.parametrize("neox", [True, False])
def test_producer_production_layout(neox):
    """Strided ql_nope (the transpose of [H, T, 512]), q_pe, kv_c and k_pe."""
    got_q, got_c, ref_q, ref_c, _ = _run_pair(33, 128, neox, True, True, seed=3, layout="production")
    assert np.array_equal(got_q, ref_q)
    assert np.array_equal(got_c, ref_c)


def test_producer_matches_the_split_chain():
    """The fused cache rows equal the split chain: the rotated k_pe (bf16) concatenated
    with kv_c and written by the library's own fp8 cache-write kernel."""
    T, H = 40, 16
    got_q, got_c, _, _, (ql, qp, kc, kp, pos, slots, cs, ns) = _run_pair(T, H, True, False, True, seed=9)
    # the split chain's bf16 rows: the oracle's rotation with a bf16 cache
    rows = np.zeros((ns, 576), dtype=np.uint16)
    oracle.fused_qk_rope_cache(ql, qp, kc, kp, pos, cs, True, slots, rows, cache_fp8=False, mode=1)
    keep = slots.numpy() >= 0
    src = torch.from_numpy(rows[slots.numpy()[keep]].view(np.int16)).view(torch.bfloat16).to(DEV)
    chain = torch.full((ns, 576), 0xA5, dtype=torch.uint8, device=DEV)
    binding.smla_fp8_cache_write(src, slots[torch.from_numpy(keep)].to(DEV), torch.tensor([KV_SCALE], device=DEV),
                                 chain)
    assert np.array_equal(got_c, chain.cpu().numpy())
    # and the bf16 q rows are concat(ql_nope, rotated q_pe) of the same rotation
    assert np.array_equal(got_q[:, :, :512], _bits(ql))


def test_producer_bounds_and_errors():
    T, H = 6, 16
    ql, qp, kc, kp, pos, slots, ns = inputs.producer_inputs(T, H, 5, 64, num_slots=8)
    pos[1] = 64      # outside [0, 64)
    pos[2] = -3
    slots[3] = 8     # outside [0, 8)
    slots[4] = -1    # no cache row
    cs = inputs.rope_cos_sin_cache(64)
    ref_cache = np.full((8, 576), 0x5A5A, dtype=np.uint16)
    ref_q = np.full((T, H, 576), 0x5A5A, dtype=np.uint16)
    q_tmp, bad = oracle.fused_qk_rope_cache(ql, qp, kc, kp, pos, cs, False, slots, ref_cache, cache_fp8=False, mode=1)
    assert bad == 3
    good = np.array([True, False, False, True, True, True])
    ref_q[good] = q_tmp[good]
    binding.smla_device_error(reset=True)
    cache = torch.full((8, 576), 0x5A5A, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    q_out = torch.full((T, H, 576), 0x5A5A, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    binding.smla_fused_qk_rope_cache(ql.to(DEV), qp.to(DEV), kc.to(DEV), kp.to(DEV), pos.to(DEV), cs.to(DEV),
                                     slots.to(DEV), cache, is_neox=False, q_out=q_out)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(q_out), ref_q)      # tokens 1 and 2 untouched
    assert np.array_equal(_bits(cache), ref_cache)  # rows of tokens 1-4 not written
    assert binding.smla_device_error(reset=True) == 4 | 8


def test_producer_empty_and_cache_only():
    T = 5
    ql, qp, kc, kp, pos, slots, ns = inputs.producer_inputs(T, 1, 8)
    cs = inputs.rope_cos_sin_cache(4096)
    cache = torch.zeros((ns, 576), dtype=torch.uint8, device=DEV)
    kvs = torch.tensor([KV_SCALE], device=DEV)
    # T = 0: nothing to do
    binding.smla_fused_qk_rope_cache(ql[:0].to(DEV), qp[:0].to(DEV), kc[:0].to(DEV), kp[:0].to(DEV),
                                     pos[:0].to(DEV), cs.to(DEV), slots[:0].to(DEV), cache, kv_scale=kvs)
    assert not cache.any().item()
    # H = 0: cache rows only
    ref = np.zeros((ns, 576), dtype=np.uint8)
    oracle.fused_qk_rope_cache(ql[:, :0], qp[:, :0], kc, kp, pos, cs, True, slots, ref, cache_fp8=True,
                               kv_scale=KV_SCALE, mode=1)
    binding.smla_fused_qk_rope_cache(ql[:, :0].to(DEV), qp[:, :0].to(DEV), kc.to(DEV), kp.to(DEV), pos.to(DEV),
                                     cs.to(DEV), slots.to(DEV), cache, kv_scale=kvs)
    torch.cuda.synchronize()
    assert np.array_equal(cache.cpu().numpy(), ref)


def test_producer_full_size_sampled():
    """T = 4096 tokens x 128 heads (the size the benchmark times): every cache row
    and a sample of q rows, bit for bit."""
    T, H = 4096, 128
    ql, qp, kc, kp, pos, slots, ns = inputs.producer_inputs(T, H, 21, 4096, skip_every=0)
    cs = inputs.rope_cos_sin_cache(4096)
    cache = torch.zeros((ns, 576), dtype=torch.uint8, device=DEV)
    q_out = binding.smla_fused_qk_rope_cache(ql.to(DEV), qp.to(DEV), kc.to(DEV), kp.to(DEV), pos.to(DEV),
                                             cs.to(DEV), slots.to(DEV), cache, is_neox=True,
                                             kv_scale=torch.tensor([KV_SCALE], device=DEV), q_out_fp8=True,
                                             q_scale=torch.tensor([Q_SCALE], device=DEV))
    torch.cuda.synchronize()
    sample = torch.from_numpy(np.random.default_rng(0).choice(T, 64, replace=False))
    ref_cache = np.zeros((ns, 576), dtype=np.uint8)
    # q rows of the sampled tokens
    ref_qs, bad = oracle.fused_qk_rope_cache(ql[sample], qp[sample], kc[sample], kp[sample], pos[sample], cs, True,
                                             np.full(sample.shape[0], -1, dtype=np.int64),
                                             np.zeros((1, 576), dtype=np.uint8), cache_fp8=True,
                                             kv_scale=KV_SCALE, q_out_fp8=True, q_scale=Q_SCALE, mode=1)
    assert bad == 0
    assert np.array_equal(q_out.cpu().numpy()[sample], ref_qs)
    # every cache row
    oracle.fused_qk_rope_cache(ql[:, :0], qp[:, :0], kc, kp, pos, cs, True, slots, ref_cache, cache_fp8=True,
                               kv_scale=KV_SCALE, mode=1)
    assert np.array_equal(cache.cpu().numpy(), ref_cache)
