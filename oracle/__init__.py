"""The fp64 CPU oracle of the sparse MLA forward (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product path (the CUDA library and
its Python binding) never loads it, and it never loads the product path: the
two share no code. The arithmetic lives in ``sparse_mla_oracle.c``; this module
compiles it with gcc (no fast-math) and marshals numpy arrays through ctypes.

Sources, by page title and section:
  * "Enable AITER sparse MLA on gfx942, including FP8 KV" (vLLM PR 60583),
    Overview and Details ("FP8 KV on gfx942", "Numerics").
  * "Fuse decode QK-RoPE + Q-concat + KV-concat + KV-cache write for sparse
    MLA" (vLLM PR 47757), Summary and Test plan (cache row layout,
    scaled_fp8_quant convention: stored = x / scale; the fused producer step:
    RoPE on q_pe / k_pe, q concat, cache write).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sparse_mla_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` (gcc, -O2, OpenMP)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off",
           "-fopenmp", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        c = ctypes
        lib.oracle_e4m3_decode.argtypes = [c.c_uint8]
        lib.oracle_e4m3_decode.restype = c.c_double
        lib.oracle_e4m3_encode.argtypes = [c.c_float]
        lib.oracle_e4m3_encode.restype = c.c_uint8
        lib.oracle_amax_bf16.argtypes = [c.c_void_p, c.c_int64]
        lib.oracle_amax_bf16.restype = c.c_float
        lib.oracle_fp8_scale_from_amax.argtypes = [c.c_float]
        lib.oracle_fp8_scale_from_amax.restype = c.c_float
        lib.oracle_fp8_scale.argtypes = [c.c_void_p, c.c_int64]
        lib.oracle_fp8_scale.restype = c.c_float
        lib.oracle_fp8_cache_write.argtypes = [
            c.c_void_p, c.c_void_p, c.c_int64, c.c_int, c.c_float,
            c.c_void_p, c.c_int64]
        lib.oracle_fp8_cache_write.restype = c.c_int64
        lib.oracle_sparse_mla.argtypes = [
            c.c_void_p, c.c_void_p, c.c_int, c.c_float, c.c_void_p,
            c.c_int, c.c_int, c.c_int, c.c_int, c.c_int64, c.c_int,
            c.c_float, c.c_int, c.c_void_p, c.c_void_p, c.c_int]
        lib.oracle_sparse_mla.restype = c.c_int64
        lib.oracle_sparse_mla_qf64.argtypes = [
            c.c_void_p, c.c_void_p, c.c_int, c.c_float, c.c_void_p,
            c.c_int, c.c_int, c.c_int, c.c_int, c.c_int64, c.c_int,
            c.c_float, c.c_void_p, c.c_void_p, c.c_int]
        lib.oracle_sparse_mla_qf64.restype = c.c_int64
        lib.oracle_sparse_mla_sinks.argtypes = [
            c.c_void_p, c.c_void_p, c.c_void_p, c.c_int, c.c_float, c.c_void_p,
            c.c_int, c.c_int, c.c_int, c.c_int, c.c_int64, c.c_int,
            c.c_float, c.c_int, c.c_void_p, c.c_void_p, c.c_void_p, c.c_int]
        lib.oracle_sparse_mla_sinks.restype = c.c_int64
        lib.oracle_rope_f64.argtypes = [c.c_void_p, c.c_int, c.c_void_p, c.c_void_p, c.c_int, c.c_void_p]
        lib.oracle_rope_f64.restype = None
        lib.oracle_fused_qk_rope_cache.argtypes = [
            c.c_void_p, c.c_void_p, c.c_void_p, c.c_void_p, c.c_void_p, c.c_void_p,
            c.c_int64, c.c_int, c.c_void_p, c.c_void_p, c.c_int, c.c_int64, c.c_float,
            c.c_void_p, c.c_int, c.c_float, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int]
        lib.oracle_fused_qk_rope_cache.restype = c.c_int64
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = c.c_int
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _as_bf16_bits(x) -> np.ndarray:
    """bf16 payload as uint16 numpy (accepts torch bf16 tensors or uint16)."""
    if hasattr(x, "dtype") and str(getattr(x, "dtype")) == "torch.bfloat16":
        import torch
        return x.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
    a = np.ascontiguousarray(x)
    if a.dtype != np.uint16:
        raise TypeError("expected bf16 bits as uint16, got %s" % a.dtype)
    return a


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def e4m3_decode(code: int) -> float:
    """Value of one OCP E4M3 code (NaN for S.1111.111)."""
    return float(_load().oracle_e4m3_decode(int(code) & 0xFF))


def e4m3_encode(x: float) -> int:
    """RNE + satfinite E4M3 code of a binary32 value (NaN -> 0x7F)."""
    return int(_load().oracle_e4m3_encode(float(np.float32(x))))


def e4m3_decode_all() -> np.ndarray:
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


def amax_bf16(x) -> float:
    a = _as_bf16_bits(x)
    return float(_load().oracle_amax_bf16(_ptr(a), a.size))


def fp8_scale_from_amax(amax: float) -> np.float32:
    return np.float32(_load().oracle_fp8_scale_from_amax(float(np.float32(amax))))


def fp8_scale(x) -> np.float32:
    """Per-tensor scale amax/448 (binary32) over a bf16 tensor."""
    a = _as_bf16_bits(x)
    return np.float32(_load().oracle_fp8_scale(_ptr(a), a.size))


def fp8_cache_write(src, slot_mapping, kv_scale, cache: np.ndarray) -> int:
    """Quantize bf16 rows src[N, D] into the uint8 cache[num_slots, D] in place."""
    s = _as_bf16_bits(src)
    N, D = s.shape
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    assert sm.shape == (N,)
    assert cache.dtype == np.uint8 and cache.flags.c_contiguous and cache.shape[1] == D
    return int(_load().oracle_fp8_cache_write(
        _ptr(s), _ptr(sm), N, D, float(np.float32(kv_scale)), _ptr(cache), cache.shape[0]))


def fp8_quantize(src, kv_scale) -> np.ndarray:
    """Codes of every row of src[N, D] (a fresh [N, D] uint8 array)."""
    s = _as_bf16_bits(src)
    N, D = s.shape
    cache = np.zeros((N, D), dtype=np.uint8)
    fp8_cache_write(s, np.arange(N, dtype=np.int64), kv_scale, cache)
    return cache


def sparse_mla(q, kv, indices, scale: float, *, kv_fp8: bool = False,
               kv_scale: float = 1.0, D_v: int = 512, q_mode: int = 0,
               nthreads: int = 0, sinks=None):
    """Exact (fp64) sparse MLA forward.

    q        bf16 [T, H, D_qk] (torch bf16 tensor or uint16 bits)
    kv       [num_slots, D_qk]: bf16 (kv_fp8=False) or uint8 E4M3 codes
    indices  int32 [T, topk], -1 = masked
    Returns (out float64 [T, H, D_v], lse float64 [T, H], n_out_of_range).
    """
    qb = _as_bf16_bits(q)
    T, H, D_qk = qb.shape
    if kv_fp8:
        kvb = kv.detach().contiguous().cpu().numpy() if hasattr(kv, "detach") else np.ascontiguousarray(kv)
        kvb = kvb.view(np.uint8)
    else:
        kvb = _as_bf16_bits(kv)
    assert kvb.ndim == 2 and kvb.shape[1] == D_qk
    idx = indices.detach().cpu().numpy() if hasattr(indices, "detach") else indices
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    assert idx.ndim == 2 and idx.shape[0] == T
    topk = idx.shape[1]
    out = np.empty((T, H, D_v), dtype=np.float64)
    lse = np.empty((T, H), dtype=np.float64)
    if sinks is None:
        bad = _load().oracle_sparse_mla(
            _ptr(qb), _ptr(kvb), 1 if kv_fp8 else 0, float(np.float32(kv_scale)), _ptr(idx),
            T, H, D_qk, D_v, kvb.shape[0], topk, float(np.float32(scale)), int(q_mode),
            _ptr(out), _ptr(lse), int(nthreads))
    else:
        sk = np.ascontiguousarray(sinks.cpu().numpy() if hasattr(sinks, "cpu") else sinks, dtype=np.float32)
        assert sk.shape == (H,)
        bad = _load().oracle_sparse_mla_sinks(
            _ptr(qb), None, _ptr(kvb), 1 if kv_fp8 else 0, float(np.float32(kv_scale)), _ptr(idx),
            T, H, D_qk, D_v, kvb.shape[0], topk, float(np.float32(scale)), int(q_mode), _ptr(sk),
            _ptr(out), _ptr(lse), int(nthreads))
    return out, lse, int(bad)


def sparse_mla_q8(q8, q_scale, kv, indices, scale: float, *, kv_fp8: bool = True,
                  kv_scale: float = 1.0, D_v: int = 512, nthreads: int = 0, sinks=None):
    """Exact (fp64) sparse MLA forward with a pre-quantized q: uint8 E4M3 codes
    [T, H, D_qk] and one per-tensor scale; q enters the dots as code * q_scale
    (the oracle's own codec, exact in fp64). kv, indices, returns as sparse_mla."""
    codes = q8.detach().cpu().numpy() if hasattr(q8, "detach") else np.asarray(q8)
    codes = np.ascontiguousarray(codes).view(np.uint8)
    T, H, D_qk = codes.shape
    table = e4m3_decode_all()
    qf = np.ascontiguousarray(table[codes] * float(np.float32(q_scale)), dtype=np.float64)
    if kv_fp8:
        kvb = kv.detach().contiguous().cpu().numpy() if hasattr(kv, "detach") else np.ascontiguousarray(kv)
        kvb = kvb.view(np.uint8)
    else:
        kvb = _as_bf16_bits(kv)
    assert kvb.ndim == 2 and kvb.shape[1] == D_qk
    idx = indices.detach().cpu().numpy() if hasattr(indices, "detach") else indices
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    topk = idx.shape[1]
    out = np.empty((T, H, D_v), dtype=np.float64)
    lse = np.empty((T, H), dtype=np.float64)
    if sinks is None:
        bad = _load().oracle_sparse_mla_qf64(
            _ptr(qf), _ptr(kvb), 1 if kv_fp8 else 0, float(np.float32(kv_scale)), _ptr(idx),
            T, H, D_qk, D_v, kvb.shape[0], topk, float(np.float32(scale)), _ptr(out), _ptr(lse), int(nthreads))
    else:
        sk = np.ascontiguousarray(sinks.cpu().numpy() if hasattr(sinks, "cpu") else sinks, dtype=np.float32)
        assert sk.shape == (H,)
        bad = _load().oracle_sparse_mla_sinks(
            None, _ptr(qf), _ptr(kvb), 1 if kv_fp8 else 0, float(np.float32(kv_scale)), _ptr(idx),
            T, H, D_qk, D_v, kvb.shape[0], topk, float(np.float32(scale)), 0, _ptr(sk),
            _ptr(out), _ptr(lse), int(nthreads))
    return out, lse, int(bad)


def rope_f64(x, cos, sin, is_neox: bool) -> np.ndarray:
    """Rotary embedding of one vector x[R] (fp64) with cos[R/2], sin[R/2]:
    each pair (a, b) becomes (a cos - b sin, b cos + a sin); neox pairs i with
    i + R/2, GPT-J pairs 2i with 2i + 1."""
    xa = np.ascontiguousarray(x, dtype=np.float64)
    ca = np.ascontiguousarray(cos, dtype=np.float64)
    sa = np.ascontiguousarray(sin, dtype=np.float64)
    R = xa.shape[0]
    assert R % 2 == 0 and ca.shape == (R // 2,) and sa.shape == (R // 2,)
    out = np.empty(R, dtype=np.float64)
    _load().oracle_rope_f64(_ptr(xa), R, _ptr(ca), _ptr(sa), 1 if is_neox else 0, _ptr(out))
    return out


def fused_qk_rope_cache(ql_nope, q_pe, kv_c, k_pe, positions, cos_sin, is_neox: bool,
                        slot_mapping, cache: np.ndarray, *, cache_fp8: bool, kv_scale: float = 1.0,
                        q_out_fp8: bool = False, q_scale: float = 1.0, mode: int = 1):
    """The fused producer step over contiguous inputs.

    ql_nope [T, H, Dn], q_pe [T, H, Dr], kv_c [T, Dn], k_pe [T, Dr]: bf16
    (torch tensors or uint16 bits); positions int64 [T]; cos_sin float32
    [max_position, Dr] (cos of the Dr/2 angles, then the sines); slot_mapping
    int64 [T] (negative: no cache row). `cache` (uint16 bf16 bits or uint8
    E4M3 codes, [num_slots, Dn + Dr]) is updated in place.
    mode 0: the rotation in fp64, rounded once to bf16; mode 1: binary32
    products and sums, the precision an fp8 code is decided in.
    Returns (q_out as uint16 bits or uint8 codes [T, H, Dn + Dr], bad).
    """
    qn = _as_bf16_bits(ql_nope)
    qp = _as_bf16_bits(q_pe)
    kc = _as_bf16_bits(kv_c)
    kp = _as_bf16_bits(k_pe)
    T, H, Dn = qn.shape
    Dr = qp.shape[2]
    assert qp.shape == (T, H, Dr) and kc.shape == (T, Dn) and kp.shape == (T, Dr)
    pos = np.ascontiguousarray(positions.cpu().numpy() if hasattr(positions, "cpu") else positions, dtype=np.int64)
    cs = np.ascontiguousarray(cos_sin.cpu().numpy() if hasattr(cos_sin, "cpu") else cos_sin, dtype=np.float32)
    sm = np.ascontiguousarray(slot_mapping.cpu().numpy() if hasattr(slot_mapping, "cpu") else slot_mapping,
                              dtype=np.int64)
    assert pos.shape == (T,) and sm.shape == (T,) and cs.ndim == 2 and cs.shape[1] == Dr
    assert cache.flags.c_contiguous and cache.shape[1] == Dn + Dr
    assert cache.dtype == (np.uint8 if cache_fp8 else np.uint16)
    q_out = np.zeros((T, H, Dn + Dr), dtype=np.uint8 if q_out_fp8 else np.uint16)
    bad = _load().oracle_fused_qk_rope_cache(
        _ptr(qn), _ptr(qp), _ptr(kc), _ptr(kp), _ptr(pos), _ptr(cs), cs.shape[0], 1 if is_neox else 0,
        _ptr(sm), _ptr(cache), 1 if cache_fp8 else 0, cache.shape[0], float(np.float32(kv_scale)),
        _ptr(q_out), 1 if q_out_fp8 else 0, float(np.float32(q_scale)), T, H, Dn, Dr, int(mode))
    return q_out, int(bad)
