"""ctypes binding of libsparse_mla.so (include/sparse_mla.h).

Argument marshalling only: every step of the computation runs in the CUDA
library. Functions keep the C names. torch supplies device memory and the
current stream; outputs and the workspace are allocated with torch when the
caller passes none (the library itself never allocates).

The library must exist: if it was not built, or fails to load, every call
raises — there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsparse_mla.so")

SMLA_OK = 0
SMLA_ERR_NULL_POINTER = 1
SMLA_ERR_BAD_SHAPE = 2
SMLA_ERR_BAD_DTYPE = 3
SMLA_ERR_MISALIGNED = 4
SMLA_ERR_UNSUPPORTED = 5
SMLA_ERR_WORKSPACE_TOO_SMALL = 6
SMLA_ERR_CUDA = 7

SMLA_KV_BF16 = 0
SMLA_KV_FP8_E4M3 = 1
SMLA_DOT_AUTO = 0
SMLA_DOT_BF16 = 1
SMLA_DOT_FP8 = 2
_DOT = {"auto": SMLA_DOT_AUTO, "bf16": SMLA_DOT_BF16, "fp8": SMLA_DOT_FP8}
SMLA_KERNEL_AUTO = 0
SMLA_KERNEL_WARP_MMA = 1
SMLA_KERNEL_TCGEN05_BASIC = 2
_KERNEL = {"auto": SMLA_KERNEL_AUTO, "mma": SMLA_KERNEL_WARP_MMA, "basic": SMLA_KERNEL_TCGEN05_BASIC}

# every function the header declares, with its ctypes signature
_c = ctypes
SIGNATURES = {
    "smla_status_string": ([_c.c_int], _c.c_char_p),
    "smla_version": ([], _c.c_int),
    "smla_plan_num_splits": ([_c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_int], _c.c_int),
    "sparse_mla_fwd_workspace_size": ([_c.c_int] * 7, _c.c_size_t),
    "sparse_mla_fwd": ([_c.c_void_p, _c.c_void_p, _c.c_int, _c.c_void_p, _c.c_void_p,
                        _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_int64, _c.c_int,
                        _c.c_float, _c.c_int, _c.c_void_p, _c.c_void_p,
                        _c.c_void_p, _c.c_size_t, _c.c_int, _c.c_void_p], _c.c_int),
    "sparse_mla_fwd_q8": ([_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                           _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_int64, _c.c_int, _c.c_float,
                           _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_size_t, _c.c_int, _c.c_void_p], _c.c_int),
    "sparse_mla_fwd_ex": ([_c.c_void_p], _c.c_int),
    "sparse_mla_fwd_ex_workspace_size": ([_c.c_void_p], _c.c_size_t),
    "smla_gather_probe": ([_c.c_void_p, _c.c_int64, _c.c_int, _c.c_void_p, _c.c_int64, _c.c_int, _c.c_int,
                           _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_void_p, _c.c_void_p], _c.c_int),
    "smla_l2_read_probe": ([_c.c_void_p, _c.c_int64, _c.c_int, _c.c_void_p, _c.c_int, _c.c_void_p], _c.c_int),
    "smla_compute_fp8_scale": ([_c.c_void_p, _c.c_int64, _c.c_void_p, _c.c_void_p], _c.c_int),
    "smla_fp8_cache_write": ([_c.c_void_p, _c.c_void_p, _c.c_int64, _c.c_int, _c.c_void_p,
                              _c.c_void_p, _c.c_int64, _c.c_void_p], _c.c_int),
    "smla_validate_indices": ([_c.c_void_p, _c.c_int, _c.c_int, _c.c_int64, _c.c_void_p,
                               _c.c_void_p], _c.c_int),
    "smla_device_error": ([_c.c_void_p, _c.c_int], _c.c_int),
    "smla_fused_qk_rope_cache": ([_c.c_void_p, _c.c_int64, _c.c_int64, _c.c_void_p, _c.c_int64, _c.c_int64,
                                  _c.c_void_p, _c.c_int64, _c.c_void_p, _c.c_int64, _c.c_void_p,
                                  _c.c_void_p, _c.c_int64, _c.c_int, _c.c_void_p, _c.c_void_p, _c.c_int,
                                  _c.c_int64, _c.c_void_p, _c.c_void_p, _c.c_int, _c.c_void_p, _c.c_int,
                                  _c.c_int, _c.c_void_p], _c.c_int),
    "smla_last_error_string": ([], _c.c_char_p),
    "sparse_mla_fwd_no_alloc": ([_c.c_void_p, _c.c_void_p, _c.c_int, _c.c_void_p, _c.c_void_p,
                                 _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_int64, _c.c_int,
                                 _c.c_float, _c.c_int, _c.c_void_p, _c.c_void_p, _c.c_int,
                                 _c.c_void_p], _c.c_int),
}



class SmlaFwdParams(ctypes.Structure):
    """smla_fwd_params of include/sparse_mla.h."""
    _fields_ = [("size", _c.c_size_t), ("q", _c.c_void_p), ("q_scale", _c.c_void_p),
                ("kv_cache", _c.c_void_p), ("kv_dtype", _c.c_int), ("kv_scale", _c.c_void_p),
                ("indices", _c.c_void_p), ("T", _c.c_int), ("H", _c.c_int), ("D_qk", _c.c_int), ("D_v", _c.c_int),
                ("num_slots", _c.c_int64), ("topk", _c.c_int), ("scale", _c.c_float), ("dot_precision", _c.c_int),
                ("sinks", _c.c_void_p), ("out", _c.c_void_p), ("lse", _c.c_void_p), ("workspace", _c.c_void_p),
                ("workspace_bytes", _c.c_size_t), ("num_splits", _c.c_int), ("stream", _c.c_void_p),
                ("kernel", _c.c_int)]


_lock = threading.Lock()
_lib = None


class SmlaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = "%s: %s" % (where, status_string(status))
        if status == SMLA_ERR_CUDA:
            msg += " (%s)" % lib().smla_last_error_string().decode()
        super().__init__(msg)


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it is missing: build it first)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError("libsparse_mla.so is not built (%s); run __graft_entry__.build()" % LIB_PATH)
            L = ctypes.CDLL(LIB_PATH)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
        return _lib


def status_string(status: int) -> str:
    return lib().smla_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != SMLA_OK:
        raise SmlaError(status, where)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(x: Optional[torch.Tensor]) -> Optional[int]:
    return None if x is None else x.data_ptr()


def _need(x: torch.Tensor, name: str, dtype, ndim: int):
    if not isinstance(x, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if x.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, x.dtype))
    if x.dim() != ndim:
        raise ValueError("%s must have %d dims, got shape %s" % (name, ndim, tuple(x.shape)))
    if not x.is_contiguous():
        raise ValueError("%s must be contiguous (strided inputs are not accepted)" % name)
    if not x.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)


def smla_device_error(reset: bool = False) -> int:
    """Error word of the device-side bounded waits (0 = none); synchronous."""
    v = ctypes.c_int(0)
    _check(lib().smla_device_error(ctypes.byref(v), int(reset)), "smla_device_error")
    return int(v.value)


def smla_version() -> int:
    return int(lib().smla_version())


def smla_plan_num_splits(T: int, H: int, D_qk: int, topk: int, kv_dtype: int, sm_count: int) -> int:
    return int(lib().smla_plan_num_splits(T, H, D_qk, topk, kv_dtype, sm_count))


def sparse_mla_fwd_workspace_size(T: int, H: int, D_qk: int, D_v: int, topk: int, kv_dtype: int,
                                  num_splits: int = 0) -> int:
    n = lib().sparse_mla_fwd_workspace_size(T, H, D_qk, D_v, topk, kv_dtype, num_splits)
    if n == ctypes.c_size_t(-1).value:
        raise SmlaError(SMLA_ERR_BAD_SHAPE, "sparse_mla_fwd_workspace_size")
    return int(n)


# zeroed workspaces, one per (device, stream); the kernel leaves them zeroed
_workspaces = {}


def workspace_for(nbytes: int, device: torch.device, stream_handle: int) -> Optional[torch.Tensor]:
    if nbytes == 0:
        return None
    key = (device.index, stream_handle)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(nbytes, dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def sparse_mla_fwd(q: torch.Tensor, kv_cache: torch.Tensor, indices: torch.Tensor, scale: float, *,
                   kv_scale: Optional[torch.Tensor] = None, dot_precision: str = "auto",
                   D_v: int = 512, out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                   return_lse: bool = True, workspace: Optional[torch.Tensor] = None,
                   num_splits: int = 0, stream=None,
                   sinks: Optional[torch.Tensor] = None,
                   kernel: str = "auto") -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """out[T,H,D_v] (bf16), lse[T,H] (fp32) of the sparse MLA forward
    (sinks: optional fp32 [H] per-head sink logits; kernel: "auto", "mma" for
    the warp-MMA kernel, or "basic" for the tcgen05 kernels that take a
    whole SM per CTA).

    q bf16 [T,H,D_qk]; kv_cache [num_slots, D_qk] bf16 or torch.float8_e4m3fn/uint8
    (E4M3 codes, then kv_scale: fp32 device scalar); indices int32 [T, topk].
    """
    _need(q, "q", torch.bfloat16, 3)
    T, H, D_qk = q.shape
    if kv_cache.dtype == torch.bfloat16:
        kv_dtype = SMLA_KV_BF16
    elif kv_cache.dtype in (torch.float8_e4m3fn, torch.uint8):
        kv_dtype = SMLA_KV_FP8_E4M3
    else:
        raise TypeError("kv_cache must be bf16 or E4M3 (float8_e4m3fn / uint8), got %s" % kv_cache.dtype)
    _need(kv_cache, "kv_cache", kv_cache.dtype, 2)
    if kv_cache.shape[1] != D_qk:
        raise ValueError("kv_cache row width %d != D_qk %d" % (kv_cache.shape[1], D_qk))
    _need(indices, "indices", torch.int32, 2)
    if indices.shape[0] != T:
        raise ValueError("indices has %d rows, q has %d" % (indices.shape[0], T))
    if kv_dtype == SMLA_KV_FP8_E4M3:
        if kv_scale is None:
            raise ValueError("an fp8 cache needs kv_scale (fp32 device scalar)")
        _need(kv_scale.reshape(1), "kv_scale", torch.float32, 1)
    if dot_precision not in _DOT:
        raise ValueError("dot_precision must be one of %s" % sorted(_DOT))
    if kernel not in _KERNEL:
        raise ValueError("kernel must be one of %s" % sorted(_KERNEL))
    topk = indices.shape[1]
    if out is None:
        out = torch.empty((T, H, D_v), dtype=torch.bfloat16, device=q.device)
    _need(out, "out", torch.bfloat16, 3)
    if lse is None and return_lse:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    sh = _stream(stream)
    need = sparse_mla_fwd_workspace_size(T, H, D_qk, D_v, topk, kv_dtype, num_splits)
    if workspace is None:
        workspace = workspace_for(need, q.device, sh)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if sinks is None and kernel == "auto":
        st = lib().sparse_mla_fwd(
            _ptr(q), _ptr(kv_cache), kv_dtype, _ptr(kv_scale), _ptr(indices),
            T, H, D_qk, D_v, kv_cache.shape[0], topk, float(scale), _DOT[dot_precision],
            _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes, int(num_splits), sh)
        _check(st, "sparse_mla_fwd")
    else:
        if sinks is not None:
            _need(sinks, "sinks", torch.float32, 1)
            if sinks.shape[0] != H:
                raise ValueError("sinks must be [H]")
        _fwd_ex(q, None, kv_cache, kv_dtype, kv_scale, indices, T, H, D_qk, D_v, topk, scale,
                _DOT[dot_precision], sinks, out, lse, workspace, ws_bytes, num_splits, sh, _KERNEL[kernel])
    return out, lse


def _fwd_ex(q, q_scale, kv_cache, kv_dtype, kv_scale, indices, T, H, D_qk, D_v, topk, scale, dot, sinks,
            out, lse, workspace, ws_bytes, num_splits, sh, kernel=SMLA_KERNEL_AUTO):
    p = SmlaFwdParams(ctypes.sizeof(SmlaFwdParams), _ptr(q), _ptr(q_scale), _ptr(kv_cache), kv_dtype,
                      _ptr(kv_scale), _ptr(indices), T, H, D_qk, D_v, kv_cache.shape[0], topk, float(scale), dot,
                      _ptr(sinks), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes, int(num_splits), sh,
                      int(kernel))
    _check(lib().sparse_mla_fwd_ex(ctypes.byref(p)), "sparse_mla_fwd_ex")


def sparse_mla_fwd_q8(q8: torch.Tensor, q_scale: torch.Tensor, kv_cache: torch.Tensor, indices: torch.Tensor,
                      scale: float, *, kv_scale: torch.Tensor, D_v: int = 512, out: Optional[torch.Tensor] = None,
                      lse: Optional[torch.Tensor] = None, return_lse: bool = True,
                      workspace: Optional[torch.Tensor] = None, num_splits: int = 0,
                      stream=None, sinks: Optional[torch.Tensor] = None,
                      kernel: str = "auto") -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """The forward with a pre-quantized q: q8 E4M3 codes [T, H, D_qk] (uint8 or
    float8_e4m3fn) and q_scale, its per-tensor fp32 device scalar; an E4M3 cache
    with kv_scale; fp8 dots."""
    if q8.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise TypeError("q8 must be E4M3 codes (uint8 / float8_e4m3fn), got %s" % q8.dtype)
    _need(q8, "q8", q8.dtype, 3)
    T, H, D_qk = q8.shape
    if kv_cache.dtype not in (torch.float8_e4m3fn, torch.uint8):
        raise TypeError("kv_cache must be E4M3 (float8_e4m3fn / uint8), got %s" % kv_cache.dtype)
    _need(kv_cache, "kv_cache", kv_cache.dtype, 2)
    if kv_cache.shape[1] != D_qk:
        raise ValueError("kv_cache row width %d != D_qk %d" % (kv_cache.shape[1], D_qk))
    _need(indices, "indices", torch.int32, 2)
    if indices.shape[0] != T:
        raise ValueError("indices has %d rows, q8 has %d" % (indices.shape[0], T))
    _need(q_scale.reshape(1), "q_scale", torch.float32, 1)
    _need(kv_scale.reshape(1), "kv_scale", torch.float32, 1)
    topk = indices.shape[1]
    if out is None:
        out = torch.empty((T, H, D_v), dtype=torch.bfloat16, device=q8.device)
    _need(out, "out", torch.bfloat16, 3)
    if lse is None and return_lse:
        lse = torch.empty((T, H), dtype=torch.float32, device=q8.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    sh = _stream(stream)
    need = sparse_mla_fwd_workspace_size(T, H, D_qk, D_v, topk, SMLA_KV_FP8_E4M3, num_splits)
    if workspace is None:
        workspace = workspace_for(need, q8.device, sh)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if kernel not in _KERNEL:
        raise ValueError("kernel must be one of %s" % sorted(_KERNEL))
    if sinks is None and kernel == "auto":
        st = lib().sparse_mla_fwd_q8(
            _ptr(q8), _ptr(q_scale), _ptr(kv_cache), _ptr(kv_scale), _ptr(indices),
            T, H, D_qk, D_v, kv_cache.shape[0], topk, float(scale),
            _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes, int(num_splits), sh)
        _check(st, "sparse_mla_fwd_q8")
    else:
        if sinks is not None:
            _need(sinks, "sinks", torch.float32, 1)
            if sinks.shape[0] != H:
                raise ValueError("sinks must be [H]")
        _fwd_ex(q8, q_scale, kv_cache, SMLA_KV_FP8_E4M3, kv_scale, indices, T, H, D_qk, D_v, topk, scale,
                SMLA_DOT_FP8, sinks, out, lse, workspace, ws_bytes, num_splits, sh, _KERNEL[kernel])
    return out, lse


def smla_gather_probe(pool: torch.Tensor, indices: torch.Tensor, *, ctas_per_sm: int = 1, stages: int = 1,
                      hold_ns: int = 0, pair_mode: int = 0, issue_warps: int = 0, copy_mode: int = 0,
                      checksum: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """The pure indexed-row copy probe: rows `indices` (int32, any shape,
    taken flat) of `pool` [num_rows, row_bytes] (any 1- or 2-byte dtype)
    gathered into shared memory (copy_mode 0: TMA gather4, 1: 16-byte cp.async)
    and folded into per-CTA checksums (uint32 device tensor
    [sm_count * ctas_per_sm], returned); pair_mode 1 / 2: CTA pairs sharing
    each tile by cluster multicast / by a bulk copy into the peer;
    issue_warps > 0: a tile's copies spread evenly over that many producer
    warps."""
    if pool.dim() != 2 or not pool.is_contiguous() or not pool.is_cuda:
        raise ValueError("pool must be a contiguous CUDA tensor [num_rows, row]")
    _need(indices.reshape(-1), "indices", torch.int32, 1)
    row_bytes = pool.shape[1] * pool.element_size()
    sms = torch.cuda.get_device_properties(pool.device).multi_processor_count
    if checksum is None:
        checksum = torch.zeros(sms * ctas_per_sm, dtype=torch.int32, device=pool.device)
    _check(lib().smla_gather_probe(_ptr(pool), pool.shape[0], row_bytes, _ptr(indices), indices.numel(),
                                   int(ctas_per_sm), int(stages), int(hold_ns), int(pair_mode), int(issue_warps),
                                   int(copy_mode), _ptr(checksum),
                                   _stream(stream)),
           "smla_gather_probe")
    return checksum


def smla_l2_read_probe(buf: torch.Tensor, reps: int, blocks: int, checksum: Optional[torch.Tensor] = None,
                       stream=None) -> torch.Tensor:
    """Stream `buf` (contiguous CUDA tensor) `reps` times from `blocks` blocks."""
    if not buf.is_contiguous() or not buf.is_cuda:
        raise ValueError("buf must be a contiguous CUDA tensor")
    if checksum is None:
        checksum = torch.zeros(blocks, dtype=torch.int32, device=buf.device)
    nbytes = buf.numel() * buf.element_size()
    _check(lib().smla_l2_read_probe(_ptr(buf), nbytes - nbytes % 16, int(reps), _ptr(checksum), int(blocks),
                                    _stream(stream)), "smla_l2_read_probe")
    return checksum


def sparse_mla_fwd_ex_workspace_size(T: int, H: int, D_qk: int, D_v: int, topk: int, kv_dtype: int, *,
                                     dot_precision: str = "auto", q8: bool = False, num_splits: int = 0,
                                     kernel: str = "auto") -> int:
    """Exact workspace bytes of one call (its dot precision, q form, kernel and splits)."""
    p = SmlaFwdParams(ctypes.sizeof(SmlaFwdParams), None, 1 if q8 else None, None, kv_dtype, None, None,
                      T, H, D_qk, D_v, 0, topk, 1.0, _DOT[dot_precision], None, None, None, None, 0,
                      int(num_splits), None, _KERNEL[kernel])
    n = lib().sparse_mla_fwd_ex_workspace_size(ctypes.byref(p))
    if n == ctypes.c_size_t(-1).value:
        raise SmlaError(SMLA_ERR_BAD_SHAPE, "sparse_mla_fwd_ex_workspace_size")
    return int(n)


def smla_compute_fp8_scale(x: torch.Tensor, scale_out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """fp32 device scalar amax(|x|)/448 of a bf16 tensor."""
    if x.dtype != torch.bfloat16 or not x.is_contiguous() or not x.is_cuda:
        raise ValueError("x must be a contiguous CUDA bf16 tensor")
    if scale_out is None:
        scale_out = torch.empty(1, dtype=torch.float32, device=x.device)
    _check(lib().smla_compute_fp8_scale(_ptr(x), x.numel(), _ptr(scale_out), _stream(stream)),
           "smla_compute_fp8_scale")
    return scale_out


def smla_fp8_cache_write(src: torch.Tensor, slot_mapping: torch.Tensor, kv_scale: torch.Tensor,
                         kv_cache: torch.Tensor, stream=None) -> torch.Tensor:
    """kv_cache[slot_mapping[n]] = E4M3(src[n] / kv_scale) (uint8 / float8_e4m3fn cache)."""
    _need(src, "src", torch.bfloat16, 2)
    _need(slot_mapping, "slot_mapping", torch.int64, 1)
    _need(kv_cache, "kv_cache", kv_cache.dtype, 2)
    if kv_cache.element_size() != 1 or kv_cache.shape[1] != src.shape[1]:
        raise ValueError("kv_cache must be 1-byte [num_slots, D]")
    N, D = src.shape
    _check(lib().smla_fp8_cache_write(_ptr(src), _ptr(slot_mapping), N, D, _ptr(kv_scale),
                                      _ptr(kv_cache), kv_cache.shape[0], _stream(stream)),
           "smla_fp8_cache_write")
    return kv_cache


def smla_validate_indices(indices: torch.Tensor, num_slots: int, bad_count: Optional[torch.Tensor] = None,
                          stream=None) -> torch.Tensor:
    """int32 device scalar: entries of indices that are neither -1 nor in [0, num_slots)."""
    _need(indices, "indices", torch.int32, 2)
    if bad_count is None:
        bad_count = torch.empty(1, dtype=torch.int32, device=indices.device)
    T, topk = indices.shape
    _check(lib().smla_validate_indices(_ptr(indices), T, topk, int(num_slots), _ptr(bad_count), _stream(stream)),
           "smla_validate_indices")
    return bad_count


def _strided(x: torch.Tensor, name: str, ndim: int):
    """A bf16 CUDA tensor whose last dimension is contiguous (other strides free)."""
    if not isinstance(x, torch.Tensor) or x.dtype != torch.bfloat16 or not x.is_cuda:
        raise TypeError("%s must be a CUDA bf16 tensor" % name)
    if x.dim() != ndim:
        raise ValueError("%s must have %d dims, got shape %s" % (name, ndim, tuple(x.shape)))
    if x.stride(-1) != 1:
        raise ValueError("%s must be contiguous in its last dimension" % name)


def smla_fused_qk_rope_cache(ql_nope: torch.Tensor, q_pe: torch.Tensor, kv_c: torch.Tensor, k_pe: torch.Tensor,
                             positions: torch.Tensor, cos_sin_cache: torch.Tensor, slot_mapping: torch.Tensor,
                             kv_cache: torch.Tensor, *, is_neox: bool = True, kv_scale: Optional[torch.Tensor] = None,
                             q_out: Optional[torch.Tensor] = None, q_out_fp8: bool = False,
                             q_scale: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """The fused producer step: q_out = concat(ql_nope, RoPE(q_pe)) (bf16, or E4M3
    codes of / q_scale) and kv_cache[slot_mapping[t]] = concat(kv_c, RoPE(k_pe))
    (bf16 cache, or a 1-byte E4M3 cache with kv_scale). ql_nope [T, H, 512] and
    q_pe [T, H, 64] may be strided (last dimension contiguous), as may kv_c
    [T, 512] and k_pe [T, 64]. Returns q_out [T, H, 576]."""
    _strided(ql_nope, "ql_nope", 3)
    _strided(q_pe, "q_pe", 3)
    _strided(kv_c, "kv_c", 2)
    _strided(k_pe, "k_pe", 2)
    T, H, Dn = ql_nope.shape
    if Dn != 512 or tuple(q_pe.shape) != (T, H, 64) or tuple(kv_c.shape) != (T, 512) or tuple(k_pe.shape) != (T, 64):
        raise ValueError("expected ql_nope [T, H, 512], q_pe [T, H, 64], kv_c [T, 512], k_pe [T, 64]")
    _need(positions, "positions", torch.int64, 1)
    _need(slot_mapping, "slot_mapping", torch.int64, 1)
    _need(cos_sin_cache, "cos_sin_cache", torch.float32, 2)
    if positions.shape[0] != T or slot_mapping.shape[0] != T or cos_sin_cache.shape[1] != 64:
        raise ValueError("positions and slot_mapping must be [T]; cos_sin_cache [max_position, 64]")
    _need(kv_cache, "kv_cache", kv_cache.dtype, 2)
    if kv_cache.shape[1] != 576:
        raise ValueError("kv_cache must be [num_slots, 576]")
    if kv_cache.element_size() == 1:
        kv_dtype = SMLA_KV_FP8_E4M3
        if kv_scale is None:
            raise ValueError("an E4M3 cache needs kv_scale")
    elif kv_cache.dtype == torch.bfloat16:
        kv_dtype = SMLA_KV_BF16
    else:
        raise TypeError("kv_cache must be bf16 or a 1-byte E4M3 cache")
    if q_out is None:
        q_out = torch.empty((T, H, 576), dtype=torch.uint8 if q_out_fp8 else torch.bfloat16, device=ql_nope.device)
    _need(q_out, "q_out", q_out.dtype, 3)
    if (q_out.element_size() == 1) != bool(q_out_fp8) or tuple(q_out.shape) != (T, H, 576):
        raise ValueError("q_out must be [T, H, 576], 1-byte when q_out_fp8 else bf16")
    if q_out_fp8 and q_scale is None:
        raise ValueError("E4M3 q_out needs q_scale")
    _check(lib().smla_fused_qk_rope_cache(
        _ptr(ql_nope), ql_nope.stride(0), ql_nope.stride(1), _ptr(q_pe), q_pe.stride(0), q_pe.stride(1),
        _ptr(kv_c), kv_c.stride(0), _ptr(k_pe), k_pe.stride(0), _ptr(positions), _ptr(cos_sin_cache),
        cos_sin_cache.shape[0], 1 if is_neox else 0, _ptr(slot_mapping), _ptr(kv_cache), kv_dtype,
        kv_cache.shape[0], _ptr(kv_scale), _ptr(q_out), SMLA_KV_FP8_E4M3 if q_out_fp8 else SMLA_KV_BF16,
        _ptr(q_scale), T, H, _stream(stream)), "smla_fused_qk_rope_cache")
    return q_out


def build_fp8_cache(kv_source: torch.Tensor, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Quantize a whole bf16 pool [num_slots, D] into a fresh E4M3 cache with its scale."""
    scale = smla_compute_fp8_scale(kv_source, stream=stream)
    cache = torch.empty(kv_source.shape, dtype=torch.uint8, device=kv_source.device)
    slots = torch.arange(kv_source.shape[0], dtype=torch.int64, device=kv_source.device)
    smla_fp8_cache_write(kv_source, slots, scale, cache, stream=stream)
    return cache, scale
