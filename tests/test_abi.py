"""The C-ABI library loads, exports every declared symbol, and rejects bad
arguments on the host before touching the GPU (CPU only: no compute call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from sparse_mla_attention_04_gb300 import build, binding
    build.build()
    return binding.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "sparse_mla.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"SMLA_API\s+[\w\s\*]+?\b(\w+)\s*\(", src))


def test_every_declared_symbol_is_exported(L):
    from sparse_mla_attention_04_gb300 import binding
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(L, n), n
    assert names == set(binding.SIGNATURES)


def test_status_strings(L):
    from sparse_mla_attention_04_gb300 import binding
    for s in range(8):
        assert binding.status_string(s).startswith("SMLA_")
    assert binding.status_string(99) == "SMLA_ERR_UNKNOWN"
    assert binding.smla_version() >> 16 == 1


def test_split_plan(L):
    from sparse_mla_attention_04_gb300 import binding as b
    assert b.smla_plan_num_splits(64, 16, 512, 2048, 0, 152) == 2     # decode bf16, tcgen05 kernel: 1 CTA/SM
    assert b.smla_plan_num_splits(64, 16, 512, 2048, 1, 152) == 4     # decode fp8, lean tcgen05 kernel: 2 CTAs/SM
    assert b.smla_plan_num_splits(4, 16, 512, 128, 0, 152) == 1       # a split keeps two key tiles
    assert b.smla_plan_num_splits(2, 16, 512, 2048, 0, 152) == 8      # few rows: up to one 8-CTA cluster
    assert b.smla_plan_num_splits(16, 16, 512, 2048, 0, 152) == 6     # many 8-CTA clusters: 6 instead
    assert b.smla_plan_num_splits(16, 16, 512, 512, 0, 152) == 4      # capped by keys per split
    assert b.smla_plan_num_splits(8192, 16, 512, 2048, 0, 152) == 1   # prefill: no split
    assert b.smla_plan_num_splits(128, 128, 576, 2048, 1, 152) == 1
    assert b.smla_plan_num_splits(1, 16, 512, 100000, 0, 152) == 8    # automatic plans stay in one cluster
    assert b.smla_plan_num_splits(4, 15, 512, 128, 0, 152) == 0       # invalid H
    # a call that shares the GPU with another, planned for half the SMs
    assert b.smla_plan_num_splits(64, 16, 512, 2048, 0, 76) == 1
    assert b.smla_plan_num_splits(64, 16, 512, 2048, 1, 76) == 2


def test_workspace_size(L):
    from sparse_mla_attention_04_gb300 import binding as b
    up = lambda x: (x + 255) // 256 * 256
    tickets = 16384 * 4
    # up to 8 splits merge inside a thread-block cluster: no workspace; more:
    # counters, then binary16 partials and their lse
    for S in (1, 2, 4, 8):
        assert b.sparse_mla_fwd_workspace_size(64, 16, 512, 512, 2048, 0, S) == 0
    for T, S in ((64, 16), (3, 9)):
        n = b.sparse_mla_fwd_workspace_size(T, 16, 512, 512, 2048, 0, S)
        assert n == up(up(tickets + T * S * 16 * 4) + T * S * 16 * 512 * 2)
    with pytest.raises(b.SmlaError):                       # more (row, group) pairs than counters
        b.sparse_mla_fwd_workspace_size(16385, 16, 512, 512, 2048, 0, 16)


def _call(L, q=0x1000, kv=0x2000, kvd=0, kvs=None, idx=0x3000, T=2, H=16, Dqk=512, Dv=512,
          slots=100, topk=8, scale=0.1, dot=0, out=0x4000, lse=None, ws=None, wsb=0, splits=1):
    return L.sparse_mla_fwd(q, kv, kvd, kvs, idx, T, H, Dqk, Dv, slots, topk, scale, dot, out, lse,
                            ws, wsb, splits, None)


def test_argument_checks_return_before_any_launch(L):
    """Every case fails a host check; the fake pointers are never dereferenced."""
    from sparse_mla_attention_04_gb300 import binding as b
    assert _call(L, q=None) == b.SMLA_ERR_NULL_POINTER
    assert _call(L, out=None) == b.SMLA_ERR_NULL_POINTER
    assert _call(L, kvd=1, dot=2, kvs=None) == b.SMLA_ERR_NULL_POINTER
    assert _call(L, T=-1) == b.SMLA_ERR_BAD_SHAPE
    assert _call(L, topk=-3) == b.SMLA_ERR_BAD_SHAPE
    assert _call(L, Dv=600) == b.SMLA_ERR_BAD_SHAPE
    assert _call(L, splits=-1) == b.SMLA_ERR_BAD_SHAPE
    assert _call(L, kvd=7) == b.SMLA_ERR_BAD_DTYPE
    assert _call(L, dot=9) == b.SMLA_ERR_BAD_DTYPE
    assert _call(L, kvd=0, dot=2) == b.SMLA_ERR_BAD_DTYPE            # fp8 dots need an fp8 cache
    assert _call(L, H=8) == b.SMLA_ERR_UNSUPPORTED
    assert _call(L, Dqk=256, Dv=256) == b.SMLA_ERR_UNSUPPORTED
    assert _call(L, kvd=1, kvs=0x5000, dot=0, q=0x1002) == b.SMLA_ERR_MISALIGNED  # bf16 dots over fp8: accepted
    assert _call(L, kvd=1, kvs=0x5000, dot=1, T=0) == b.SMLA_OK
    assert _call(L, splits=129) == b.SMLA_ERR_UNSUPPORTED
    assert _call(L, q=0x1002) == b.SMLA_ERR_MISALIGNED
    assert _call(L, out=0x4008) == b.SMLA_ERR_MISALIGNED
    assert _call(L, idx=0x3002) == b.SMLA_ERR_MISALIGNED
    assert _call(L, splits=16, ws=None) == b.SMLA_ERR_NULL_POINTER
    assert _call(L, splits=16, ws=0x8000, wsb=100) == b.SMLA_ERR_WORKSPACE_TOO_SMALL
    need = b.sparse_mla_fwd_workspace_size(2, 16, 512, 512, 8, 0, 16)
    assert _call(L, splits=16, ws=0x8010, wsb=need) == b.SMLA_ERR_MISALIGNED
    assert _call(L, T=16385, splits=16, ws=0x8000, wsb=1 << 40) == b.SMLA_ERR_UNSUPPORTED
    assert _call(L, T=0) == b.SMLA_OK                                   # no-op


def test_companion_argument_checks(L):
    from sparse_mla_attention_04_gb300 import binding as b
    assert L.smla_compute_fp8_scale(None, 10, 0x100, None) == b.SMLA_ERR_NULL_POINTER
    assert L.smla_compute_fp8_scale(0x1000, -1, 0x100, None) == b.SMLA_ERR_BAD_SHAPE
    assert L.smla_compute_fp8_scale(0x1008, 10, 0x100, None) == b.SMLA_ERR_MISALIGNED
    assert L.smla_fp8_cache_write(0x1000, 0x2000, 4, 12, 0x3000, 0x4000, 10, None) == b.SMLA_ERR_BAD_SHAPE
    assert L.smla_fp8_cache_write(0x1000, None, 4, 16, 0x3000, 0x4000, 10, None) == b.SMLA_ERR_NULL_POINTER
    assert L.smla_fp8_cache_write(0x1004, 0x2000, 4, 16, 0x3000, 0x4000, 10, None) == b.SMLA_ERR_MISALIGNED
    assert L.smla_validate_indices(None, 2, 3, 10, 0x100, None) == b.SMLA_ERR_NULL_POINTER
    assert L.smla_validate_indices(0x1000, -2, 3, 10, 0x100, None) == b.SMLA_ERR_BAD_SHAPE


def test_binding_rejects_strided_and_wrong_dtypes():
    import torch
    from sparse_mla_attention_04_gb300 import binding as b
    q = torch.zeros((2, 16, 512), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        b._need(q.transpose(0, 1), "q", torch.bfloat16, 3)
    with pytest.raises(TypeError):
        b._need(q.float(), "q", torch.bfloat16, 3)
    with pytest.raises(ValueError):
        b._need(q, "q", torch.bfloat16, 3)   # not a CUDA tensor


def test_fwd_ex_structure_size_and_checks(L):
    """The ctypes structure matches the header's size check; the checks run
    before any launch (fake pointers, T = 0 or failing checks)."""
    import ctypes
    from sparse_mla_attention_04_gb300 import binding as b
    p = b.SmlaFwdParams(ctypes.sizeof(b.SmlaFwdParams), 0x1000, None, 0x2000, 0, None, 0x3000, 0, 16, 512, 512,
                        100, 8, 0.1, 0, None, 0x4000, None, None, 0, 1, None)
    assert L.sparse_mla_fwd_ex(ctypes.byref(p)) == b.SMLA_OK           # T = 0: a no-op
    p.size = 8
    assert L.sparse_mla_fwd_ex(ctypes.byref(p)) == b.SMLA_ERR_BAD_SHAPE
    p.size = ctypes.sizeof(b.SmlaFwdParams)
    p.T, p.q_scale = 2, 0x5000                                          # E4M3 q codes with a bf16 cache
    assert L.sparse_mla_fwd_ex(ctypes.byref(p)) == b.SMLA_ERR_BAD_DTYPE
    p.q_scale, p.sinks = None, 0x6002                                   # misaligned sinks
    assert L.sparse_mla_fwd_ex(ctypes.byref(p)) == b.SMLA_ERR_MISALIGNED
    assert L.sparse_mla_fwd_ex(None) == b.SMLA_ERR_NULL_POINTER


def test_fused_producer_argument_checks(L):
    """Host-side checks of smla_fused_qk_rope_cache: each bad argument is
    refused before any launch (fake device addresses, nothing dereferenced)."""
    from sparse_mla_attention_04_gb300 import binding as b

    def call(**kw):
        a = dict(ql=0x1000, ql_st=128 * 512, ql_sh=512, qpe=0x2000, qpe_st=128 * 64, qpe_sh=64, kvc=0x3000,
                 kvc_st=512, kpe=0x4000, kpe_st=64, pos=0x5000, cs=0x6000, maxpos=4096, neox=1, slots=0x7000,
                 cache=0x8000, kvdt=b.SMLA_KV_FP8_E4M3, nslots=100, kvs=0x9000, qout=0xA000,
                 qdt=b.SMLA_KV_FP8_E4M3, qs=0xB000, T=4, H=128)
        a.update(kw)
        return L.smla_fused_qk_rope_cache(a["ql"], a["ql_st"], a["ql_sh"], a["qpe"], a["qpe_st"], a["qpe_sh"],
                                          a["kvc"], a["kvc_st"], a["kpe"], a["kpe_st"], a["pos"], a["cs"],
                                          a["maxpos"], a["neox"], a["slots"], a["cache"], a["kvdt"], a["nslots"],
                                          a["kvs"], a["qout"], a["qdt"], a["qs"], a["T"], a["H"], None)

    assert call(T=-1) == b.SMLA_ERR_BAD_SHAPE
    assert call(H=-1) == b.SMLA_ERR_BAD_SHAPE
    assert call(kvdt=7) == b.SMLA_ERR_BAD_DTYPE
    assert call(T=0) == b.SMLA_OK                          # no-op, nothing launched
    assert call(ql=None) == b.SMLA_ERR_NULL_POINTER
    assert call(kvs=None) == b.SMLA_ERR_NULL_POINTER       # an E4M3 cache needs its scale
    assert call(maxpos=0) == b.SMLA_ERR_BAD_SHAPE
    assert call(H=65535 * 8) == b.SMLA_ERR_BAD_SHAPE       # H + 1 rows exceed the grid
    assert call(ql_st=4) == b.SMLA_ERR_MISALIGNED          # latent rows move as 16-byte vectors
    assert call(ql=0x1008) == b.SMLA_ERR_MISALIGNED
    assert call(qpe_sh=3) == b.SMLA_ERR_MISALIGNED


def test_probe_host_checks(L):
    """The measurement kernels reject bad arguments before any launch."""
    from sparse_mla_attention_04_gb300 import binding as b
    P = 1 << 12   # fake, never dereferenced: every call below fails its host checks
    lib = b.lib()
    assert lib.smla_gather_probe(None, 10, 1024, P, 64, 1, 1, 0, 0, 0, 0, P, None) == b.SMLA_ERR_NULL_POINTER
    assert lib.smla_gather_probe(P, 10, 1000, P, 64, 1, 1, 0, 0, 0, 0, P, None) == b.SMLA_ERR_BAD_SHAPE   # not 16-byte rows
    assert lib.smla_gather_probe(P, 10, 2048, P, 64, 1, 1, 0, 0, 0, 0, P, None) == b.SMLA_ERR_BAD_SHAPE   # > 1 KB rows
    assert lib.smla_gather_probe(P, 10, 1024, P, 64, 5, 1, 0, 0, 0, 0, P, None) == b.SMLA_ERR_BAD_SHAPE   # > 4 CTAs/SM
    assert lib.smla_gather_probe(P, 10, 1024, P, 64, 1, 9, 0, 0, 0, 0, P, None) == b.SMLA_ERR_BAD_SHAPE   # > 8 stages
    assert lib.smla_gather_probe(P + 8, 10, 1024, P, 64, 1, 1, 0, 0, 0, 0, P, None) == b.SMLA_ERR_MISALIGNED
    assert lib.smla_gather_probe(P, 10, 1024, P, 64, 2, 1, 0, 1, 0, 0, P, None) == b.SMLA_ERR_UNSUPPORTED  # pairs: 1 CTA/SM
    assert lib.smla_gather_probe(P, 10, 1024, P, 64, 1, 1, 0, 4, 0, 0, P, None) == b.SMLA_ERR_BAD_SHAPE
    assert lib.smla_gather_probe(P, 10, 1024, P, 64, 1, 1, 0, 0, 9, 0, P, None) == b.SMLA_ERR_BAD_SHAPE  # > 8 warps
    # 1 KB rows: 128 copies a tile, more than 32 lanes of each of 3 warps
    assert lib.smla_gather_probe(P, 10, 1024, P, 64, 1, 1, 0, 0, 3, 0, P, None) == b.SMLA_ERR_BAD_SHAPE
    assert lib.smla_gather_probe(P, 10, 1024, P, 64, 1, 1, 0, 0, 0, 2, P, None) == b.SMLA_ERR_BAD_SHAPE  # copy mode
    # cp.async copies: single CTAs, every producer warp
    assert lib.smla_gather_probe(P, 10, 1024, P, 64, 1, 1, 0, 1, 0, 1, P, None) == b.SMLA_ERR_UNSUPPORTED
    assert lib.smla_gather_probe(P, 10, 1024, P, 64, 1, 1, 0, 0, 4, 1, P, None) == b.SMLA_ERR_UNSUPPORTED
    assert lib.smla_l2_read_probe(P, 1000, 1, P, 4, None) == b.SMLA_ERR_BAD_SHAPE
    assert lib.smla_l2_read_probe(None, 1024, 1, P, 4, None) == b.SMLA_ERR_NULL_POINTER


def test_exact_workspace_follows_the_call(L):
    """The exact per-call workspace query follows the dot precision: the
    128-head E4M3 kernel (fp8 dots) keeps its quantized q in the workspace,
    bf16 dots over the same cache run on the warp-MMA kernel with none."""
    from sparse_mla_attention_04_gb300 import binding as b
    fp8 = b.sparse_mla_fwd_ex_workspace_size(128, 128, 576, 512, 2048, 1, dot_precision="fp8", num_splits=1)
    bd = b.sparse_mla_fwd_ex_workspace_size(128, 128, 576, 512, 2048, 1, dot_precision="bf16", num_splits=1)
    q8 = b.sparse_mla_fwd_ex_workspace_size(128, 128, 576, 512, 2048, 1, q8=True, num_splits=1)
    mma = b.sparse_mla_fwd_ex_workspace_size(128, 128, 576, 512, 2048, 1, dot_precision="fp8", num_splits=1,
                                             kernel="mma")
    assert fp8 == q8 == b.sparse_mla_fwd_workspace_size(128, 128, 576, 512, 2048, 1, 1) > (8 << 20)
    assert bd == 0 and mma == 0
    # more than 8 splits: counters and partials whatever the dot precision
    for dp in ("auto", "fp8"):
        assert b.sparse_mla_fwd_ex_workspace_size(4, 16, 512, 512, 2048, 1, dot_precision=dp, num_splits=16) == \
            b.sparse_mla_fwd_workspace_size(4, 16, 512, 512, 2048, 1, 16)
    with pytest.raises(b.SmlaError):
        b.sparse_mla_fwd_ex_workspace_size(4, 16, 512, 512, 2048, 0, dot_precision="fp8", num_splits=1)
