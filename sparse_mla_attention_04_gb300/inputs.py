"""Seeded synthetic inputs for the sparse MLA forward.

This module is the only code that the CUDA path and the fp64 oracle share. It
draws random numbers and lays out indices; it holds none of the method's
arithmetic (no logits, softmax, quantization or scaling of values).

The recipes follow the workloads the pages measure on ("Route gfx942 sparse
MLA prefill to AITER pa_prefill_sparse" (vLLM PR 60102), the per-call table of
the jin-amd A/B: 16 heads, D=512, top-k 2048 at 2 / 16 / 16K rows; and the
gfx942 FP8 KV page, vLLM PR 60583, for the fp8 cache): no public dataset is
involved, every value is drawn here.

  * q and the KV source rows are N(0, 1) drawn in float32 and rounded to bf16.
  * The cache is paged with 64-slot blocks. Each sequence owns its blocks,
    through a seeded random block table; an index names a physical slot,
    block_table[pos // 64] * 64 + pos % 64, of a logical position pos.
  * Top-k positions are distinct and uniform over a row's context, unsorted;
    unused entries are -1 at the end of the row.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

BLOCK = 64


@dataclasses.dataclass
class Workload:
    """Shape and recipe of one synthetic sparse MLA call."""
    name: str
    T: int
    H: int
    D_qk: int
    D_v: int
    num_slots: int
    topk: int
    kv_fp8: bool
    scale: float
    kind: str                 # "uniform" | "decode" | "prefill" | "wide"
    ctx: int = 0              # per-sequence context (decode / wide)
    short_rows: int = 0       # rows whose context is < topk (decode fp8)
    seed: int = 0

    @property
    def kv_bytes_per_elem(self) -> int:
        return 1 if self.kv_fp8 else 2


def tiny(seed: int = 0) -> Workload:
    """T=4, H=16, D=512, a 4096-slot bf16 pool, topk=128 distinct uniform."""
    return Workload("tiny", 4, 16, 512, 512, 4096, 128, False, 1.0 / math.sqrt(512),
                    "uniform", seed=seed)


def decode(n_seqs: int = 64, ctx: int = 131072, topk: int = 2048, fp8: bool = False,
           short_rows: int = 0, H: int = 16, seed: int = 0, name: Optional[str] = None) -> Workload:
    """One query row per sequence, each with its own `ctx` paged slots."""
    assert ctx % BLOCK == 0
    nm = name or ("decode_fp8" if fp8 else "decode_bf16")
    return Workload(nm, n_seqs, H, 512, 512, n_seqs * ctx, topk, fp8, 1.0 / math.sqrt(512),
                    "decode", ctx=ctx, short_rows=short_rows, seed=seed)


def decode_bf16(seed: int = 0) -> Workload:
    """64 sequences x 1 row, H=16, D=512, 131072-token contexts (8.4M slots), topk 2048."""
    return decode(64, 131072, 2048, False, 0, seed=seed)


def decode_fp8(seed: int = 0) -> Workload:
    """As decode_bf16 with an E4M3 cache; 16 of the 64 rows have a context < 2048."""
    return decode(64, 131072, 2048, True, 16, seed=seed)


def prefill(T: int = 8192, topk: int = 2048, seed: int = 0, name: str = "prefill_bf16") -> Workload:
    """One sequence of T rows over a T-slot pool; row t selects min(topk, t+1) of [0, t]."""
    assert T % BLOCK == 0
    return Workload(name, T, 16, 512, 512, T, topk, False, 1.0 / math.sqrt(512),
                    "prefill", ctx=T, seed=seed)


def wide(T: int = 128, ctx: int = 32768, topk: int = 2048, seed: int = 0,
         name: str = "wide_fp8") -> Workload:
    """H=128, D_qk=576 (512 latent + 64 rope columns), D_v=512, E4M3 cache."""
    assert ctx % BLOCK == 0
    return Workload(name, T, 128, 576, 512, T * ctx, topk, True, 1.0 / math.sqrt(576),
                    "wide", ctx=ctx, seed=seed)


CONFIGS = {
    "tiny": tiny,
    "decode_bf16": decode_bf16,
    "decode_fp8": decode_fp8,
    "prefill_bf16": prefill,
    "wide_fp8": wide,
}


# --------------------------------------------------------------------------
# indices
# --------------------------------------------------------------------------

def _block_tables(rng: np.random.Generator, n_seqs: int, blocks_per_seq: int) -> np.ndarray:
    """A random assignment of the pool's blocks to sequences: [n_seqs, blocks_per_seq]."""
    perm = rng.permutation(n_seqs * blocks_per_seq).astype(np.int64)
    return perm.reshape(n_seqs, blocks_per_seq)


def _to_physical(table_row: np.ndarray, pos: np.ndarray) -> np.ndarray:
    return table_row[pos // BLOCK] * BLOCK + pos % BLOCK


def make_indices(w: Workload, seed: Optional[int] = None) -> np.ndarray:
    """int32 [T, topk] physical slot ids, -1 padded at the end of short rows."""
    rng = np.random.Generator(np.random.PCG64(w.seed if seed is None else seed))
    idx = np.full((w.T, w.topk), -1, dtype=np.int64)
    if w.kind == "uniform":
        for t in range(w.T):
            idx[t] = rng.choice(w.num_slots, w.topk, replace=False)
    elif w.kind in ("decode", "wide"):
        tables = _block_tables(rng, w.T, w.ctx // BLOCK)
        short = set()
        if w.short_rows:
            short = set(rng.choice(w.T, w.short_rows, replace=False).tolist())
        for t in range(w.T):
            if t in short:
                c = int(rng.integers(1, w.topk))          # context in [1, topk - 1]
                pos = rng.permutation(c)
            else:
                pos = rng.choice(w.ctx, w.topk, replace=False)
            idx[t, :len(pos)] = _to_physical(tables[t], pos)
    elif w.kind == "prefill":
        table = _block_tables(rng, 1, w.num_slots // BLOCK)[0]
        for t in range(w.T):
            n = min(w.topk, t + 1)
            pos = rng.permutation(t + 1) if n == t + 1 else rng.choice(t + 1, n, replace=False)
            idx[t, :n] = _to_physical(table, pos)
    else:
        raise ValueError(w.kind)
    return idx.astype(np.int32)


def valid_count(indices: np.ndarray) -> int:
    """Number of entries that name a slot (not -1)."""
    return int((indices != -1).sum())


# --------------------------------------------------------------------------
# values
# --------------------------------------------------------------------------

def normal_bf16(shape, seed: int, device="cpu", chunk_rows: int = 1 << 20) -> torch.Tensor:
    """N(0,1) drawn in float32 and rounded to bf16, generated in row chunks."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(shape[0], -1)
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        tmp = torch.randn((r1 - r0, flat.shape[1]), generator=gen, dtype=torch.float32, device=device)
        flat[r0:r1].copy_(tmp)
        del tmp
    return out


def make_q(w: Workload, seed: Optional[int] = None, device="cpu") -> torch.Tensor:
    s = (w.seed if seed is None else seed) * 1000003 + 17
    return normal_bf16((w.T, w.H, w.D_qk), s, device)


def make_kv_source(w: Workload, device="cpu") -> torch.Tensor:
    """bf16 [num_slots, D_qk]: the cache itself for bf16, the quantizer's input for fp8."""
    return normal_bf16((w.num_slots, w.D_qk), w.seed * 1000003 + 29, device)


# --------------------------------------------------------------------------
# inputs of the fused producer step (RoPE + q concat + cache write)
# --------------------------------------------------------------------------

def rope_cos_sin_cache(max_position: int, rot_dim: int = 64, base: float = 10000.0) -> torch.Tensor:
    """float32 [max_position, rot_dim]: for each position p the cosines of
    p * base^(-2i / rot_dim), i < rot_dim / 2, then their sines (the usual
    rotary table, an input of the producer step)."""
    inv = base ** (-np.arange(0, rot_dim, 2, dtype=np.float64) / rot_dim)
    ang = np.arange(max_position, dtype=np.float64)[:, None] * inv[None, :]
    return torch.from_numpy(np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32))


def producer_inputs(T: int, H: int, seed: int, max_position: int = 4096, num_slots: Optional[int] = None,
                    skip_every: int = 0):
    """bf16 ql_nope [T, H, 512], q_pe [T, H, 64], kv_c [T, 512], k_pe [T, 64]
    (N(0, 1)), int64 positions [T] uniform in [0, max_position), and int64
    distinct slots [T] in [0, num_slots) (every `skip_every`-th is -1)."""
    ns = num_slots if num_slots is not None else 2 * T + 7
    rng = np.random.default_rng(seed)
    ql = normal_bf16((T, H, 512), seed * 7 + 1)
    qp = normal_bf16((T, H, 64), seed * 7 + 2)
    kc = normal_bf16((T, 512), seed * 7 + 3)
    kp = normal_bf16((T, 64), seed * 7 + 4)
    pos = rng.integers(0, max_position, T).astype(np.int64)
    slots = rng.permutation(ns)[:T].astype(np.int64)
    if skip_every:
        slots[::skip_every] = -1
    return ql, qp, kc, kp, torch.from_numpy(pos), torch.from_numpy(slots), ns
