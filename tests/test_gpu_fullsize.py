"""Full-size workloads, in the launch configuration the benchmark times
(automatic split plan), checked against the oracle on sampled rows (GPU).

The oracle computes each sampled row exactly from the rows its indices name
(gathered from the device pool by torch indexing, then renumbered densely);
for an fp8 cache the oracle derives the per-tensor scale from the whole bf16
source (chunked amax) and encodes the gathered rows itself.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import DEV, TOL_BF16, TOL_FP8, TOL_FP8_MIRROR, compare
from sparse_mla_attention_04_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


def oracle_scale_of(src_dev: torch.Tensor, rows_per_chunk: int = 1 << 20) -> np.float32:
    amax = 0.0
    for r0 in range(0, src_dev.shape[0], rows_per_chunk):
        amax = max(amax, oracle.amax_bf16(src_dev[r0:r0 + rows_per_chunk].cpu()))
    return oracle.fp8_scale_from_amax(amax)


def sampled_check(w, rows, q_dev, src_dev, idx_np, out, lse, gpu_cache=None, gpu_scale=None):
    sel = idx_np[rows]
    uniq = np.unique(sel[sel >= 0])
    remap = np.where(sel >= 0, np.searchsorted(uniq, np.maximum(sel, 0)), -1).astype(np.int32)
    src_rows = src_dev[torch.from_numpy(uniq).to(DEV)].cpu()
    q_rows = q_dev[torch.from_numpy(np.asarray(rows)).to(DEV)].cpu()
    got_o = out[rows].float().cpu().numpy().astype(np.float64)
    got_l = lse[rows].cpu().numpy().astype(np.float64)
    if w.kv_fp8:
        s = oracle_scale_of(src_dev)
        assert np.float32(gpu_scale.item()) == s, "per-tensor scale differs from the oracle's"
        codes = oracle.fp8_quantize(src_rows, s)
        gpu_rows = gpu_cache[torch.from_numpy(uniq).to(DEV)].cpu().numpy()
        assert (gpu_rows == codes).all(), "GPU cache rows differ from the oracle's encoding"
        ro, rl, _ = oracle.sparse_mla(q_rows, codes, remap, w.scale, kv_fp8=True, kv_scale=float(s), D_v=w.D_v)
        res = compare(got_o, got_l, ro, rl, TOL_FP8, w.name)
        mo, ml, _ = oracle.sparse_mla(q_rows, codes, remap, w.scale, kv_fp8=True, kv_scale=float(s),
                                      D_v=w.D_v, q_mode=1)
        res["mirror"] = compare(got_o, got_l, mo, ml, TOL_FP8_MIRROR, w.name + " (q quantized)")
    else:
        ro, rl, _ = oracle.sparse_mla(q_rows, src_rows, remap, w.scale, D_v=w.D_v)
        res = compare(got_o, got_l, ro, rl, TOL_BF16, w.name)
    return res


def run_full(w, rows):
    idx_np = inputs.make_indices(w)
    q = inputs.make_q(w, device=DEV)
    src = inputs.make_kv_source(w, device=DEV)
    cache, scale = (binding.build_fp8_cache(src) if w.kv_fp8 else (src, None))
    out, lse = binding.sparse_mla_fwd(q, cache, torch.from_numpy(idx_np).to(DEV), w.scale, kv_scale=scale,
                                      dot_precision="fp8" if w.kv_fp8 else "auto", D_v=w.D_v)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    res = sampled_check(w, rows, q, src, idx_np, out, lse, cache if w.kv_fp8 else None, scale)
    print(w.name, res)
    del q, src, cache, out, lse
    torch.cuda.empty_cache()
    return res


def test_decode_bf16_full():
    run_full(inputs.decode_bf16(), [0, 1, 31, 63])


def test_decode_fp8_full():
    w = inputs.decode_fp8()
    idx = inputs.make_indices(w)
    short = [t for t in range(w.T) if (idx[t] == -1).any()][:2]
    run_full(w, [0, 40] + short)


def test_prefill_bf16_full():
    run_full(inputs.prefill(), [0, 1, 777, 2047, 2048, 5000, 8191])


def test_wide_fp8_full():
    # rows 1, 2, 65 and 126 straddle two SM pairs of the stream-K split (76 pairs on 152 SMs)
    run_full(inputs.wide(), [0, 1, 2, 65, 126, 127])
