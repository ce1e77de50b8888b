"""sparse_mla_fwd_no_alloc against sparse_mla_fwd (GPU).

The no-allocation entry point serves callers that cannot allocate device
memory for a workspace (an engine that reserved nearly all of HBM for its
KV-cache pool, or a framework that only hands a plug-in fixed buffers): the
workspace lives in a static array inside the library. This checks, through
the C ABI, that two calls in a row that need that workspace (more than 8
splits per row) and one that needs none give the same results as the
entry point with a caller-provided workspace, within the bf16 tolerances.
The file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

from parity import DEV, TOL_BF16, compare
from sparse_mla_attention_04_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


def _call_no_alloc(q, kv, idx, scale, num_splits):
    T, H, D_qk = q.shape
    out = torch.full((T, H, 512), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((T, H), float("nan"), dtype=torch.float32, device=DEV)
    st = binding.lib().sparse_mla_fwd_no_alloc(
        q.data_ptr(), kv.data_ptr(), binding.SMLA_KV_BF16, None, idx.data_ptr(), T, H, D_qk, 512, kv.shape[0],
        idx.shape[1], float(scale), binding.SMLA_DOT_AUTO, out.data_ptr(), lse.data_ptr(), num_splits,
        torch.cuda.current_stream().cuda_stream)
    assert st == binding.SMLA_OK, binding.status_string(st)
    return out, lse


@pytest.mark.parametrize("num_splits", [16, 12, 0])
def test_no_alloc_matches_workspace_entry_point(num_splits):
    results = []
    for seed in (41, 42):  # two calls in a row share the static workspace
        w = inputs.Workload("noalloc", 4, 16, 512, 512, 6000, 2048, False, 1 / np.sqrt(512), "uniform", seed=seed)
        q = inputs.make_q(w).to(DEV)
        kv = inputs.make_kv_source(w).to(DEV)
        idx = torch.from_numpy(inputs.make_indices(w)).to(DEV)
        o_ref, l_ref = binding.sparse_mla_fwd(q, kv, idx, w.scale, num_splits=num_splits)
        o_new, l_new = _call_no_alloc(q, kv, idx, w.scale, num_splits)
        results.append((o_ref.float().cpu().numpy(), l_ref.cpu().numpy(),
                        o_new.float().cpu().numpy(), l_new.cpu().numpy()))
    torch.cuda.synchronize()
    for o_ref, l_ref, o_new, l_new in results:
        compare(o_new.astype(np.float64), l_new.astype(np.float64), o_ref.astype(np.float64),
                l_ref.astype(np.float64), TOL_BF16, "no_alloc")


def test_no_alloc_rejects_oversized_workspace():
    """A call whose workspace would exceed the static array returns
    SMLA_ERR_WORKSPACE_TOO_SMALL and launches nothing."""
    T, H, topk, S = 64, 16, 4096, 64          # partials alone: 64*64*16*512*4 B = 128 MiB
    need = binding.sparse_mla_fwd_workspace_size(T, H, 512, 512, topk, binding.SMLA_KV_BF16, S)
    assert need > (8 << 20)
    q = torch.zeros((T, H, 512), dtype=torch.bfloat16, device=DEV)
    kv = torch.zeros((16, 512), dtype=torch.bfloat16, device=DEV)
    idx = torch.zeros((T, topk), dtype=torch.int32, device=DEV)
    out = torch.zeros((T, H, 512), dtype=torch.bfloat16, device=DEV)
    st = binding.lib().sparse_mla_fwd_no_alloc(
        q.data_ptr(), kv.data_ptr(), binding.SMLA_KV_BF16, None, idx.data_ptr(), T, H, 512, 512, 16, topk, 0.1,
        binding.SMLA_DOT_AUTO, out.data_ptr(), None, S, None)
    assert st == binding.SMLA_ERR_WORKSPACE_TOO_SMALL
