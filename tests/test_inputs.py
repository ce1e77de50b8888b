"""The seeded input recipes have the structure the workloads call for (CPU)."""
import numpy as np
import torch

from sparse_mla_attention_04_gb300 import inputs


def _check_rows(idx, w, lo_hi_per_row=None):
    for t in range(w.T):
        row = idx[t]
        valid = row[row != -1]
        # distinct, inside the pool, and -1 only as trailing padding
        assert len(np.unique(valid)) == len(valid)
        assert valid.min() >= 0 and valid.max() < w.num_slots
        n = len(valid)
        assert (row[:n] != -1).all() and (row[n:] == -1).all()


def test_tiny_recipe():
    w = inputs.tiny()
    idx = inputs.make_indices(w)
    assert idx.shape == (4, 128) and idx.dtype == np.int32
    _check_rows(idx, w)
    assert (idx != -1).all()
    assert (inputs.make_indices(w) == idx).all()          # seeded
    assert not (inputs.make_indices(w, seed=1) == idx).all()


def test_decode_recipe_owns_blocks_and_pads_short_rows():
    w = inputs.decode(n_seqs=8, ctx=4096, topk=512, fp8=True, short_rows=2)
    idx = inputs.make_indices(w)
    _check_rows(idx, w)
    counts = (idx != -1).sum(1)
    assert (counts == 512).sum() == 6
    short = counts[counts < 512]
    assert len(short) == 2 and (short >= 1).all()
    # every sequence's slots come from blocks that no other sequence touches
    owner = {}
    for t in range(w.T):
        for b in set((idx[t][idx[t] != -1] // 64).tolist()):
            assert owner.setdefault(b, t) == t


def test_prefill_recipe_is_causal():
    w = inputs.prefill(T=256, topk=64)
    idx = inputs.make_indices(w)
    _check_rows(idx, w)
    counts = (idx != -1).sum(1)
    assert (counts == np.minimum(64, np.arange(256) + 1)).all()
    # rows with t + 1 <= topk select every position of [0, t]: the same slot set
    # grows by exactly one slot per row
    for t in range(1, 64):
        a = set(idx[t - 1][:t].tolist())
        b = set(idx[t][:t + 1].tolist())
        assert a < b and len(b - a) == 1


def test_full_size_shapes():
    assert inputs.decode_bf16().num_slots == 8388608
    assert inputs.wide().num_slots == 4194304
    w = inputs.decode_fp8()
    assert w.kv_fp8 and w.short_rows == 16 and w.T == 64


def test_values_are_bf16_normal_and_seeded():
    a = inputs.normal_bf16((1000, 64), 3)
    b = inputs.normal_bf16((1000, 64), 3)
    assert a.dtype == torch.bfloat16 and torch.equal(a, b)
    x = a.float()
    assert abs(x.mean().item()) < 0.02 and abs(x.std().item() - 1) < 0.02
