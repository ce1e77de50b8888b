"""Parity of the CUDA sparse MLA forward with the fp64 oracle (GPU).

Sizes span several key tiles and splits with ragged tails while the oracle
finishes in seconds; the edge cases cover empty and ragged inputs, the
degenerate cases of the method and index handling (bit-exact)."""
import math

import numpy as np
import pytest
import torch

import oracle
import parity
from parity import DEV, TOL_BF16, compare
from sparse_mla_attention_04_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

# the kernels that serve 16 heads: the library's choice (the lean tcgen05
# kernel for an E4M3 cache, the whole-SM one for bf16), the warp-MMA kernel,
# and the whole-SM tcgen05 kernel for E4M3 too (the forward's kernel-choice field)
KERNELS = ["tcgen05", "mma", "basic"]


@pytest.fixture(params=KERNELS)
def kernel(request):
    """The kernel a test runs on: the library's own choice, the warp-MMA
    kernel, or the tcgen05 kernels that take a whole SM per CTA (asked for
    through the forward's kernel-choice field)."""
    yield {"tcgen05": "auto", "mma": "mma", "basic": "basic"}[request.param]
    assert binding.smla_device_error() == 0


def test_tiny_config(kernel):
    res, _, _ = parity.case(inputs.tiny(seed=0), kernel=kernel)
    print(res)


@pytest.mark.parametrize("splits", [0, 1, 2, 3, 4, 8, 9, 16, 32])
def test_decode_bf16_small(splits, kernel):
    w = inputs.decode(n_seqs=8, ctx=8192, topk=2048, name="decode_bf16_small")
    parity.case(w, kernel=kernel, num_splits=splits)


def test_split_counts_agree(kernel):
    w = inputs.decode(n_seqs=4, ctx=8192, topk=1000, name="decode_ragged")
    outs = [parity.case(w, kernel=kernel, num_splits=s)[1] for s in (1, 2, 5, 6, 7, 11)]
    for o in outs[1:]:
        # each split count rounds P to bf16 against its own running max, so
        # runs differ by the bf16 tolerance, not by fp32 noise
        rel = np.linalg.norm(o - outs[0]) / np.linalg.norm(outs[0])
        assert rel < 5e-3, rel


@pytest.mark.parametrize("splits", [0, 1, 4, 12])
def test_decode_fp8_small(splits, kernel):
    w = inputs.decode(n_seqs=8, ctx=8192, topk=2048, fp8=True, short_rows=2, name="decode_fp8_small")
    res, _, _ = parity.case(w, num_splits=splits, kernel=kernel)
    print(res)


def test_prefill_small(kernel):
    w = inputs.prefill(T=384, topk=128, name="prefill_small")
    parity.case(w, kernel=kernel)


@pytest.fixture(params=["auto", "basic"])
def wide_kernel(request):
    """The 128-head kernel's two launch plans: the (row, key tile) sequence
    spread evenly over one CTA pair per two SMs, rows cut between pairs
    merging through the workspace (auto), and one CTA pair per row
    (basic)."""
    yield request.param
    assert binding.smla_device_error() == 0


def test_wide_head_small(wide_kernel):
    w = inputs.wide(T=4, ctx=4096, topk=2048, name="wide_small")
    res, _, _ = parity.case(w, kernel=wide_kernel)
    print(res)


# --- 128-head kernel (E4M3 cache, D_qk = 576): ragged top-k, masks, the
# rescale path, several head groups, and the fallback for explicit splits ---

@pytest.mark.parametrize("topk", [1, 31, 33, 63, 65, 700])
def test_wide_head_ragged_topk(topk, wide_kernel):
    w = inputs.Workload("wide_ragged", 3, 128, 576, 512, 3000, topk, True, 1 / math.sqrt(576), "uniform",
                        seed=topk)
    parity.case(w, kernel=wide_kernel)
    assert binding.smla_device_error() == 0


def test_wide_head_masks_and_empty_rows(wide_kernel):
    w = inputs.Workload("wide_masks", 4, 128, 576, 512, 3000, 300, True, 1 / math.sqrt(576), "uniform", seed=9)
    idx = inputs.make_indices(w)
    rng = np.random.default_rng(11)
    idx[0, rng.choice(300, 200, replace=False)] = -1   # scattered
    idx[1, :] = -1                                      # empty row
    idx[2, :299] = -1                                   # one index, at the end
    res, out, lse = parity.case(w, idx=idx, kernel=wide_kernel)
    assert (out[1] == 0).all() and np.isneginf(lse[1]).all()


def test_wide_head_rescale_path(wide_kernel):
    """Row 0 lists its keys in ascending order of head 0's logit with q
    scaled up, so the running max of most heads climbs by more than 2^8
    several times and the kernel rescales O rows in tensor memory. Scaled-up
    logits amplify the fp8 rounding of q itself, so only the mirrored
    comparison (the oracle quantizes q the same way) applies."""
    w = inputs.Workload("wide_rescale", 2, 128, 576, 512, 3000, 640, True, 1 / math.sqrt(576), "uniform", seed=13)
    q = (inputs.make_q(w).float() * 3).to(torch.bfloat16)
    kv = inputs.make_kv_source(w)
    idx = inputs.make_indices(w)
    logits0 = kv[idx[0]].float() @ q[0, 0].float()
    idx[0] = idx[0][np.argsort(logits0.numpy())]
    res, _, _ = parity.case(w, idx=idx, kv_src=kv, q=q, check_plain=False, kernel=wide_kernel)
    assert "mirror" in res


@pytest.mark.parametrize("T,H,topk", [(80, 128, 200), (90, 128, 130), (77, 128, 64), (41, 256, 300),
                                    (160, 128, 2048)])
def test_wide_head_rows_shared_between_pairs(T, H, topk, wide_kernel):
    """More rows than SM pairs: the (row, key tile) sequence is cut into one
    range per pair, so rows straddle two pairs and merge through the
    workspace (with "basic" every pair keeps one whole row); with 256 heads
    a row is one of two head groups of a query row."""
    w = inputs.Workload("wide_shared", T, H, 576, 512, 3000, topk, True, 1 / math.sqrt(576), "uniform",
                        seed=T + topk)
    idx = inputs.make_indices(w)
    idx[3, :] = -1                     # an empty row
    idx[5, topk // 2:] = -1            # a short one
    res, out, lse = parity.case(w, idx=idx, kernel=wide_kernel)
    assert (out[3] == 0).all() and np.isneginf(lse[3]).all()


@pytest.mark.parametrize("T", [3, 80])
def test_wide_head_topk_zero(T, wide_kernel):
    """No keys at all: every row is empty (out = 0, lse = -inf), also when
    the rows outnumber the SM pairs."""
    w = inputs.Workload("wide_topk0", T, 128, 576, 512, 3000, 1, True, 1 / math.sqrt(576), "uniform", seed=3)
    q = inputs.make_q(w).to(DEV)
    cache, kvs = binding.build_fp8_cache(inputs.make_kv_source(w).to(DEV))
    idx = torch.empty((T, 0), dtype=torch.int32, device=DEV)
    out, lse = parity.fwd(wide_kernel, q, cache, idx, w.scale, kv_scale=kvs, dot_precision="fp8")
    torch.cuda.synchronize()
    assert (out == 0).all() and torch.isneginf(lse).all()


def test_wide_head_two_head_groups(wide_kernel):
    w = inputs.Workload("wide_h256", 2, 256, 576, 512, 3000, 300, True, 1 / math.sqrt(576), "uniform", seed=5)
    parity.case(w, kernel=wide_kernel)


def test_wide_head_explicit_splits():
    """An explicit split count goes to the warp-MMA kernel (the 128-head
    kernel does not split the top-k list); results agree within tolerance."""
    w = inputs.Workload("wide_split", 2, 128, 576, 512, 3000, 700, True, 1 / math.sqrt(576), "uniform", seed=17)
    parity.case(w, num_splits=3)


def test_wide_head_then_many_splits_share_a_workspace():
    """The 128-head kernel's quantized q lives in the workspace after the
    merge counters: a 16-split call that follows on the same buffer still
    finds its counters at zero."""
    ww = inputs.Workload("wide_ws", 81, 128, 576, 512, 3000, 200, True, 1 / math.sqrt(576), "uniform", seed=21)
    wd = inputs.decode(n_seqs=4, ctx=8192, topk=2048, name="decode_after_wide")
    need = max(binding.sparse_mla_fwd_workspace_size(ww.T, ww.H, ww.D_qk, ww.D_v, ww.topk, 1, 0),
               binding.sparse_mla_fwd_workspace_size(wd.T, wd.H, wd.D_qk, wd.D_v, wd.topk, 0, 16))
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    for w, kw in ((ww, {}), (wd, {"num_splits": 16}), (ww, {}), (wd, {"num_splits": 16})):
        q = inputs.make_q(w)
        src = inputs.make_kv_source(w)
        idx = inputs.make_indices(w)
        cache, kvs = parity.gpu_cache(src.to(DEV), w.kv_fp8)
        out, lse = binding.sparse_mla_fwd(q.to(DEV), cache, torch.from_numpy(idx).to(DEV), w.scale, kv_scale=kvs,
                                          dot_precision="fp8" if w.kv_fp8 else "auto", workspace=ws, **kw)
        torch.cuda.synchronize()
        ocache, oscale = parity.oracle_cache(src, w.kv_fp8)
        qm = 1 if w.kv_fp8 else 0
        ro, rl, _ = oracle.sparse_mla(q, ocache, idx, w.scale, kv_fp8=w.kv_fp8, kv_scale=oscale, q_mode=qm)
        tol = parity.TOL_FP8_MIRROR if w.kv_fp8 else TOL_BF16
        compare(out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), ro, rl, tol,
                w.name)
    assert binding.smla_device_error() == 0


def test_wide_head_bf16_cache():
    w = inputs.wide(T=3, ctx=2048, topk=700, name="wide_bf16")
    w.kv_fp8 = False
    parity.case(w, num_splits=2)


@pytest.mark.parametrize("topk", [1, 31, 32, 33, 63, 64, 65, 127, 129])
@pytest.mark.parametrize("fp8", [False, True])
def test_topk_edges(topk, fp8, kernel):
    w = inputs.Workload("edge", 3, 16, 512, 512, 1000, topk, fp8, 1 / math.sqrt(512), "uniform", seed=topk)
    for s in (1, 2):
        if s <= max(1, topk // 32):
            parity.case(w, kernel=kernel, num_splits=s)


def test_masks_anywhere_and_empty_rows(kernel):
    w = inputs.Workload("masks", 5, 32, 512, 512, 3000, 200, False, 0.05, "uniform", seed=3)
    idx = inputs.make_indices(w)
    rng = np.random.default_rng(7)
    idx[0, rng.choice(200, 150, replace=False)] = -1      # scattered
    idx[1, :] = -1                                         # empty row
    idx[2, :199] = -1                                      # one index, at the end
    idx[3, ::2] = -1
    for s in (1, 3, 7):
        res, out, lse = parity.case(w, kernel=kernel, idx=idx, num_splits=s)
        assert (out[1] == 0).all() and np.isneginf(lse[1]).all()


def test_single_index_is_bit_exact(kernel):
    w = inputs.Workload("single", 3, 16, 512, 512, 500, 64, False, 0.3, "uniform", seed=4)
    idx = np.full((3, 64), -1, dtype=np.int32)
    idx[0, 5] = 17
    idx[1, 63] = 499
    idx[2, 0] = 0
    q = inputs.make_q(w)
    kv = inputs.make_kv_source(w)
    for s in (1, 2):
        out, lse = parity.fwd(kernel, q.to(DEV), kv.to(DEV), torch.from_numpy(idx).to(DEV), w.scale,
                                          num_splits=s)
        out = out.cpu()
        for t, j in ((0, 17), (1, 499), (2, 0)):
            assert torch.equal(out[t], kv[j].unsqueeze(0).expand(16, 512)), (s, t)


def test_scale_zero_gives_mean(kernel):
    w = inputs.Workload("scale0", 2, 16, 512, 512, 800, 96, False, 0.0, "uniform", seed=5)
    parity.case(w, kernel=kernel, num_splits=2)


def test_duplicate_indices_count(kernel):
    w = inputs.Workload("dups", 2, 16, 512, 512, 600, 128, False, 1 / math.sqrt(512), "uniform", seed=6)
    idx = inputs.make_indices(w)
    idx[0, 64:] = idx[0, :64]          # every slot twice
    idx[1, 1:40] = idx[1, 0]           # one slot 40 times
    parity.case(w, kernel=kernel, idx=idx, num_splits=2)


@pytest.mark.parametrize("fp8", [False, True])
def test_nan_poison_in_unreferenced_slots(fp8, kernel):
    """Slots no index names (including 0 and num_slots-1) hold NaN; the output
    must be finite and bit-identical to the run without poison."""
    w = inputs.Workload("poison", 4, 16, 512, 512, 2048, 256, fp8, 1 / math.sqrt(512), "uniform", seed=8)
    rng = np.random.default_rng(8)
    idx = np.stack([1 + rng.choice(w.num_slots - 2, 256, replace=False) for _ in range(4)]).astype(np.int32)
    idx[2, 100:] = -1
    q = inputs.make_q(w).to(DEV)
    kv_src = inputs.make_kv_source(w).to(DEV)
    cache, kvs = parity.gpu_cache(kv_src, fp8)
    used = np.zeros(w.num_slots, bool)
    used[idx[idx >= 0]] = True
    unused = torch.from_numpy(np.nonzero(~used)[0]).to(DEV)
    assert used[0] == False and used[-1] == False
    ti = torch.from_numpy(idx).to(DEV)
    dot = "fp8" if fp8 else "auto"
    for s in (1, 3):
        o1, l1 = parity.fwd(kernel, q, cache, ti, w.scale, kv_scale=kvs, dot_precision=dot, num_splits=s)
        o1, l1 = o1.clone(), l1.clone()
        poisoned = cache.clone()
        if fp8:
            poisoned[unused] = 0x7F
        else:
            poisoned[unused] = float("nan")
        o2, l2 = parity.fwd(kernel, q, poisoned, ti, w.scale, kv_scale=kvs, dot_precision=dot, num_splits=s)
        torch.cuda.synchronize()
        assert torch.isfinite(o2.float()).all()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_out_of_range_indices_are_masked_and_reported(kernel):
    w = inputs.Workload("oob", 3, 16, 512, 512, 1000, 64, False, 0.1, "uniform", seed=9)
    idx = inputs.make_indices(w)
    bad = idx.copy()
    bad[0, 3] = 1000
    bad[0, 9] = -2
    bad[1, 0] = 2 ** 31 - 1
    bad[2, 63] = -(2 ** 31)
    clean = bad.copy()
    clean[(clean < -1) | (clean >= 1000)] = -1
    q = inputs.make_q(w).to(DEV)
    kv = inputs.make_kv_source(w).to(DEV)
    o1, l1 = parity.fwd(kernel, q, kv, torch.from_numpy(bad).to(DEV), w.scale, num_splits=2)
    o2, l2 = parity.fwd(kernel, q, kv, torch.from_numpy(clean).to(DEV), w.scale, num_splits=2)
    n_bad = binding.smla_validate_indices(torch.from_numpy(bad).to(DEV), 1000)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert int(n_bad.item()) == 4
    assert int(binding.smla_validate_indices(torch.from_numpy(clean).to(DEV), 1000).item()) == 0


def test_lse_optional_and_t_zero():
    w = inputs.tiny()
    q = inputs.make_q(w).to(DEV)
    kv = inputs.make_kv_source(w).to(DEV)
    idx = torch.from_numpy(inputs.make_indices(w)).to(DEV)
    o1, _ = binding.sparse_mla_fwd(q, kv, idx, w.scale)
    o2, l2 = binding.sparse_mla_fwd(q, kv, idx, w.scale, return_lse=False)
    assert l2 is None and torch.equal(o1, o2)
    e, el = binding.sparse_mla_fwd(q[:0], kv, idx[:0], w.scale)
    assert e.shape == (0, 16, 512)


@pytest.mark.parametrize("splits", [1, 2, 9])
def test_pool_in_l2_and_in_dram_give_the_same_bits(splits):
    """A bf16 pool that fits in a quarter of L2 is gathered by eight producer
    warps, a larger one by four; the arithmetic is the same, so the same rows
    in a 4 MB pool and in that pool padded to 64 MB give identical bits."""
    w = inputs.Workload("pool_modes", 6, 16, 512, 512, 4096, 1500, False, 1 / math.sqrt(512), "uniform", seed=21)
    q = inputs.make_q(w).to(DEV)
    small = inputs.make_kv_source(w).to(DEV)
    big = torch.zeros((65536, 512), dtype=torch.bfloat16, device=DEV)
    big[:4096] = small
    big[4096:] = float("nan")  # never referenced
    idx = inputs.make_indices(w)
    idx[1, 700:] = -1
    ti = torch.from_numpy(idx).to(DEV)
    o1, l1 = binding.sparse_mla_fwd(q, small, ti, w.scale, num_splits=splits)
    o2, l2 = binding.sparse_mla_fwd(q, big, ti, w.scale, num_splits=splits)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.isfinite(o1.float()).all()
    assert binding.smla_device_error() == 0


def test_topk_zero_gives_empty_rows(kernel):
    w = inputs.tiny()
    q = inputs.make_q(w).to(DEV)
    kv = inputs.make_kv_source(w).to(DEV)
    idx = torch.empty((4, 0), dtype=torch.int32, device=DEV)
    out, lse = parity.fwd(kernel, q, kv, idx, w.scale)
    torch.cuda.synchronize()
    assert (out == 0).all() and torch.isneginf(lse).all()


def test_workspace_errors_on_device():
    w = inputs.tiny()
    q = inputs.make_q(w).to(DEV)
    kv = inputs.make_kv_source(w).to(DEV)
    idx = torch.from_numpy(inputs.make_indices(w)).to(DEV)
    small = torch.zeros(64, dtype=torch.uint8, device=DEV)
    with pytest.raises(binding.SmlaError) as ei:
        binding.sparse_mla_fwd(q, kv, idx, w.scale, num_splits=16, workspace=small)
    assert ei.value.status == binding.SMLA_ERR_WORKSPACE_TOO_SMALL
    # a misaligned q (odd bf16 offset) is refused before launch
    qq = torch.empty(q.numel() + 8, dtype=torch.bfloat16, device=DEV)[1:1 + q.numel()].view(q.shape)
    st = binding.lib().sparse_mla_fwd(qq.data_ptr(), kv.data_ptr(), 0, None, idx.data_ptr(), 4, 16, 512, 512,
                                      4096, 128, 0.1, 0, q.data_ptr(), None, None, 0, 1, None)
    assert st == binding.SMLA_ERR_MISALIGNED


def test_workspace_reuse_across_shapes(kernel):
    """One workspace buffer serves calls of different shapes and split counts
    (the merge counters live in a fixed region that every call leaves zero)."""
    ws = torch.zeros(64 << 20, dtype=torch.uint8, device=DEV)
    shapes = [(2, 16, 900, 16), (5, 32, 700, 9), (1, 16, 2048, 32), (3, 16, 512, 12), (2, 16, 900, 16)]
    for i, (T, H, topk, S) in enumerate(shapes):
        w = inputs.Workload("reuse%d" % i, T, H, 512, 512, 4000, topk, False, 0.05, "uniform", seed=20 + i)
        q = inputs.make_q(w)
        kv = inputs.make_kv_source(w)
        idx = inputs.make_indices(w)
        out, lse = parity.fwd(kernel, q.to(DEV), kv.to(DEV), torch.from_numpy(idx).to(DEV), w.scale,
                                          num_splits=S, workspace=ws)
        torch.cuda.synchronize()
        ref_o, ref_l, _ = oracle.sparse_mla(q, kv, idx, w.scale)
        compare(out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
                ref_o, ref_l, TOL_BF16, w.name)


def test_large_logits_take_the_rescale_path(kernel):
    """Logits whose running max climbs by far more than 2^8 from tile to tile
    force the rescale path (the tcgen05 kernel then rescales O in tensor
    memory): q is scaled up and row 0 lists its keys in ascending order of
    head 0's logit. V is left as drawn, so |out| stays small."""
    w = inputs.Workload("rescale", 3, 16, 512, 512, 3000, 640, False, 0.35, "uniform", seed=31)
    q = (inputs.make_q(w).float() * 4).to(torch.bfloat16)
    kv = inputs.make_kv_source(w)
    idx = inputs.make_indices(w)
    logits0 = kv[idx[0]].float() @ q[0, 0].float()
    idx[0] = idx[0][np.argsort(logits0.numpy())]
    for S in (1, 2, 3):
        parity.case(w, kernel=kernel, idx=idx, kv_src=kv, q=q, num_splits=S)


@pytest.mark.parametrize("topk", [5, 20])
@pytest.mark.parametrize("fp8", [False, True])
def test_more_splits_than_keys(topk, fp8, kernel):
    """Explicit split counts above the number of keys leave most splits empty
    (no tile, lse -inf): the cluster merge (8), the workspace merge (16) and
    the maximum (128) must all give the single-split result."""
    w = inputs.Workload("split_empty", 3, 16, 512, 512, 700, topk, fp8, 1 / math.sqrt(512), "uniform", seed=topk)
    outs = []
    for s in (1, 8, 16, 128):
        res, out, lse = parity.case(w, kernel=kernel, num_splits=s)
        assert np.isfinite(out).all() and np.isfinite(lse).all()
        outs.append(out)
    for o in outs[1:]:
        rel = np.linalg.norm(o - outs[0]) / np.linalg.norm(outs[0])
        assert rel < 5e-3, rel
