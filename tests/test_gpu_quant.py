"""The fp8 companion kernels against the oracle's codec, bit for bit (GPU)."""
import numpy as np
import pytest
import torch

import oracle
from parity import DEV
from sparse_mla_attention_04_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


def _all_bf16_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).reshape(-1, 64)  # [1024, 64]


@pytest.mark.parametrize("scale", [1.0, 0.37, "amax"])
def test_cache_write_bit_exact_on_every_bf16(scale):
    src = _all_bf16_patterns()
    if scale == "amax":
        s = float(oracle.fp8_scale(inputs.normal_bf16((4096, 64), 11)))
    else:
        s = float(np.float32(scale))
    n = src.shape[0]
    perm = np.random.default_rng(1).permutation(n + 10)[:n].astype(np.int64)   # scattered slots
    slots = perm.copy()
    slots[::97] = -1                                                           # skipped rows
    ref = np.full((n + 10, 64), 0xAB, dtype=np.uint8)
    oracle.fp8_cache_write(src, slots, s, ref)
    cache = torch.full((n + 10, 64), 0xAB, dtype=torch.uint8, device=DEV)
    kvs = torch.tensor([s], dtype=torch.float32, device=DEV)
    binding.smla_fp8_cache_write(src.to(DEV), torch.from_numpy(slots).to(DEV), kvs, cache)
    got = cache.cpu().numpy()
    nan_ref = (ref & 0x7F) == 0x7F
    nan_got = (got & 0x7F) == 0x7F
    assert (nan_ref == nan_got).all()
    assert (got[~nan_ref] == ref[~nan_ref]).all()


@pytest.mark.parametrize("n", [0, 1, 7, 8, 9, 1000, 65536 * 3 + 5])
def test_fp8_scale_bit_exact(n):
    x = inputs.normal_bf16((max(n, 1), 1), 5)[:n].reshape(-1).contiguous()
    if n > 10:
        x[3] = float("nan")
        x[n - 1] = -9.5
    ref = oracle.fp8_scale(x)
    got = binding.smla_compute_fp8_scale(x.to(DEV)).item()
    assert np.float32(got) == ref


def test_cache_write_wide_rows_and_bounds():
    """576-wide rows (latent + rope part); out-of-range slots are skipped."""
    src = inputs.normal_bf16((300, 576), 12)
    s = oracle.fp8_scale(src)
    slots = np.arange(300, dtype=np.int64)
    slots[5] = 300        # out of range
    slots[6] = -4         # out of range
    ref = np.zeros((300, 576), dtype=np.uint8)
    oracle.fp8_cache_write(src, slots, s, ref)
    cache = torch.zeros((300, 576), dtype=torch.uint8, device=DEV)
    binding.smla_fp8_cache_write(src.to(DEV), torch.from_numpy(slots).to(DEV),
                                 torch.tensor([float(s)], device=DEV), cache)
    assert (cache.cpu().numpy() == ref).all()
