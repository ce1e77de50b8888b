"""The measurement kernels bench.py reports beside the forward (GPU).

The gather probe copies the rows an index list names; the XOR of its per-CTA
checksums must equal the XOR of the first 4 bytes of every named row (a -1 or
out-of-range entry contributes zero: the copy fills the row with zeros),
whatever the row width, CTAs per SM, ring depth and copy method. The L2 read probe must be
deterministic."""
import numpy as np
import pytest
import torch

from parity import DEV
from sparse_mla_attention_04_gb300 import binding

pytestmark = pytest.mark.gpu


def _expected(pool_u8: np.ndarray, idx: np.ndarray) -> int:
    words = pool_u8[:, :4].copy().view(np.uint32)[:, 0]
    ok = (idx >= 0) & (idx < pool_u8.shape[0])
    x = np.bitwise_xor.reduce(words[idx[ok]]) if ok.any() else np.uint32(0)
    return int(x)


@pytest.mark.parametrize("row_bytes", [1024, 512, 576, 128])
@pytest.mark.parametrize("ctas_stages", [(1, 3), (2, 1), (3, 1)])
def test_gather_probe_checksum(row_bytes, ctas_stages):
    k, st = ctas_stages
    rng = np.random.default_rng(row_bytes + 7 * k)
    rows = 5000
    pool = torch.from_numpy(rng.integers(0, 256, (rows, row_bytes), dtype=np.uint8)).to(DEV)
    idx = rng.integers(0, rows, 64 * 300 + 37).astype(np.int32)     # a ragged last tile
    idx[::11] = -1
    idx[5] = rows                # out of range: masked
    idx[9] = -7
    ck = binding.smla_gather_probe(pool, torch.from_numpy(idx).to(DEV), ctas_per_sm=k, stages=st)
    torch.cuda.synchronize()
    got = int(np.bitwise_xor.reduce(ck.cpu().numpy().view(np.uint32)))
    assert got == _expected(pool.cpu().numpy(), idx)
    assert binding.smla_device_error() == 0


@pytest.mark.parametrize("row_bytes", [1024, 576, 512, 128, 16])
@pytest.mark.parametrize("ctas_stages", [(1, 3), (2, 1), (3, 1)])
def test_gather_probe_cp_async(row_bytes, ctas_stages):
    """16-byte cp.async copies fill the same swizzled ring as the TMA copies:
    row r's first chunk lands where the consumer reads it."""
    k, st = ctas_stages
    rng = np.random.default_rng(row_bytes + 5 * k + 1)
    rows = 3000
    pool = torch.from_numpy(rng.integers(0, 256, (rows, row_bytes), dtype=np.uint8)).to(DEV)
    idx = rng.integers(0, rows, 64 * 280 + 45).astype(np.int32)
    idx[::13] = -1
    idx[3] = rows
    idx[4] = -9
    ck = binding.smla_gather_probe(pool, torch.from_numpy(idx).to(DEV), ctas_per_sm=k, stages=st, copy_mode=1)
    torch.cuda.synchronize()
    got = int(np.bitwise_xor.reduce(ck.cpu().numpy().view(np.uint32)))
    assert got == _expected(pool.cpu().numpy(), idx)
    assert binding.smla_device_error() == 0


@pytest.mark.parametrize("row_bytes,issue_warps", [(576, 4), (576, 5), (576, 8), (1024, 4), (1024, 8), (128, 1),
                                                   (512, 3)])
def test_gather_probe_issue_warps(row_bytes, issue_warps):
    """The copies spread evenly over 1-8 producer warps gather the same rows."""
    rng = np.random.default_rng(row_bytes + issue_warps)
    rows = 4000
    pool = torch.from_numpy(rng.integers(0, 256, (rows, row_bytes), dtype=np.uint8)).to(DEV)
    idx = rng.integers(0, rows, 64 * 250 + 19).astype(np.int32)
    idx[::9] = -1
    ck = binding.smla_gather_probe(pool, torch.from_numpy(idx).to(DEV), ctas_per_sm=1, stages=3,
                                   issue_warps=issue_warps)
    torch.cuda.synchronize()
    got = int(np.bitwise_xor.reduce(ck.cpu().numpy().view(np.uint32)))
    assert got == _expected(pool.cpu().numpy(), idx)
    assert binding.smla_device_error() == 0


@pytest.mark.parametrize("row_bytes", [576, 1024])
@pytest.mark.parametrize("pair_mode", [1, 2, 3])
def test_gather_probe_pairs(row_bytes, pair_mode):
    rng = np.random.default_rng(row_bytes + 3)
    rows = 4000
    pool = torch.from_numpy(rng.integers(0, 256, (rows, row_bytes), dtype=np.uint8)).to(DEV)
    idx = rng.integers(0, rows, 64 * 200 + 5).astype(np.int32)
    idx[::7] = -1
    ck = binding.smla_gather_probe(pool, torch.from_numpy(idx).to(DEV), ctas_per_sm=1, stages=2, pair_mode=pair_mode)
    # (pair_mode 3 runs independent CTAs: every checksum counts)
    torch.cuda.synchronize()
    got = int(np.bitwise_xor.reduce(ck.cpu().numpy().view(np.uint32)))
    assert got == _expected(pool.cpu().numpy(), idx)
    assert binding.smla_device_error() == 0


def test_gather_probe_empty_and_hold():
    pool = torch.zeros((64, 1024), dtype=torch.uint8, device=DEV)
    ck = binding.smla_gather_probe(pool, torch.empty(0, dtype=torch.int32, device=DEV), ctas_per_sm=1, stages=1)
    torch.cuda.synchronize()
    assert int(ck.abs().sum()) == 0
    pool[3, :4] = torch.tensor([1, 2, 3, 4], dtype=torch.uint8)
    idx = torch.full((64 * 4,), 3, dtype=torch.int32, device=DEV)
    idx[0] = -1                  # an odd number of copies of row 3 remains
    ck = binding.smla_gather_probe(pool, idx, ctas_per_sm=2, stages=1, hold_ns=2000)
    torch.cuda.synchronize()
    got = int(np.bitwise_xor.reduce(ck.cpu().numpy().view(np.uint32)))
    assert got == int(np.frombuffer(bytes([1, 2, 3, 4]), dtype=np.uint32)[0])


def test_gather_probe_rejects_what_does_not_fit():
    pool = torch.zeros((64, 1024), dtype=torch.uint8, device=DEV)
    idx = torch.zeros(64, dtype=torch.int32, device=DEV)
    with pytest.raises(binding.SmlaError) as ei:
        binding.smla_gather_probe(pool, idx, ctas_per_sm=2, stages=3)   # 2 x 192 KB
    assert ei.value.status == binding.SMLA_ERR_UNSUPPORTED


def test_l2_read_probe_is_deterministic():
    # random words: an aligned arange XORs to exactly zero over each block
    g = torch.Generator(device=DEV)
    g.manual_seed(5)
    buf = torch.randint(-2 ** 31, 2 ** 31 - 1, (1 << 20,), dtype=torch.int32, device=DEV, generator=g)
    a = binding.smla_l2_read_probe(buf, 3, 40)
    b = binding.smla_l2_read_probe(buf, 3, 40)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and int(a.abs().sum()) != 0
