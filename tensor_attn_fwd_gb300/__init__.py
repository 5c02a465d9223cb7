"""Python binding of libattn.so -- a GB300 (sm_103a) attention-forward library.

This module only marshals arguments: it checks dtypes, shapes, contiguity and
devices, allocates outputs with PyTorch when the caller does not pass them,
and calls the C ABI declared in ``include/attn.h`` on the current CUDA stream.
Every step of the computation runs in the library's CUDA kernels; there is no
CPU or PyTorch fallback -- if the library is missing or a call fails, an
exception is raised.

Names follow the C ABI:
    attn_fwd(q, k, v, causal, scale)            -> (o, lse)
    attn_fwd_bf16o(q, k, v, causal, scale)      -> (o bf16, lse)
    attn_decode_splitkv(q, k, v, num_splits)    -> (o_part, lse_part)
    attn_decode_splitkv_varlen(q, k, v, seqlens, num_splits) -> (o_part, lse_part)
    attn_combine(o_part, lse_part)              -> (o, lse)
    decode(q, k, v, num_splits)                 -> (o, lse)   both stages
    attn_decode_splitkv_paged(q, k_cache, v_cache, block_table, seqlens, num_splits)
    decode_paged(...)                           -> (o, lse)   both stages, paged cache
    attn_bwd(q, k, v, o, lse, dout, causal, scale) -> (dq, dk, dv)
    attn_rope_table(max_pos, D, base)           -> (cos, sin) table
    attn_qkv_rope(x, w, table, Hq, Hkv)         -> (q, k, v) bf16, RoPE applied
Layouts: Q [B,Hq,Sq,D], K/V [B,Hkv,Sk,D] bf16; O [B,Hq,Sq,D], LSE [B,Hq,Sq] fp32.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

__all__ = ["AttnError", "attn_fwd", "attn_fwd_bf16o", "attn_decode_splitkv", "attn_decode_splitkv_varlen",
           "attn_decode_splitkv_paged", "attn_combine", "attn_decode_fused", "decode", "decode_paged", "attn_bwd",
           "attn_rope_table", "attn_qkv_rope", "attn_decode_num_splits",
           "attn_status_string", "attn_debug_status", "library_path", "load_library",
           "ATTN_OK", "ATTN_ERR_INVALID_ARG", "ATTN_ERR_UNSUPPORTED", "ATTN_ERR_MISALIGNED",
           "ATTN_ERR_CUDA", "ATTN_ERR_TIMEOUT", "ATTN_ERR_BOUNDS", "attn_wait_selftest", "attn_fwd_splitkv", "attn_fwd_num_splits"]

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_MISALIGNED = 3
ATTN_ERR_CUDA = 4
ATTN_ERR_TIMEOUT = 5
ATTN_ERR_BOUNDS = 6

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libattn.so"
_lib = None
_lock = threading.Lock()

_vp = ctypes.c_void_p
_int = ctypes.c_int
_flt = ctypes.c_float

# Exported symbols and their C signatures (include/attn.h).
_SIGNATURES = {
    "attn_fwd": ([_vp, _vp, _vp, _vp, _vp, _int, _int, _int, _int, _int, _int, _int, _flt,
                  _vp], _int),
    "attn_fwd_bf16o": ([_vp, _vp, _vp, _vp, _vp, _int, _int, _int, _int, _int, _int, _int, _flt,
                        _vp], _int),
    "attn_decode_splitkv": ([_vp, _vp, _vp, _vp, _vp, _int, _int, _int, _int, _int, _int,
                             _flt, _vp], _int),
    "attn_decode_splitkv_varlen": ([_vp, _vp, _vp, _vp, _vp, _vp, _int, _int, _int, _int, _int,
                                    _int, _flt, _vp], _int),
    "attn_decode_splitkv_paged": ([_vp] * 7 + [_int] * 8 + [_flt, _vp], _int),
    "attn_combine": ([_vp, _vp, _vp, _vp, _int, _int, _int, _int, _vp], _int),
    "attn_decode_fused": ([_vp] * 9 + [_int] * 6 + [_flt, _vp], _int),
    "attn_decode_fused_counters": ([_int, _int, _int, ctypes.POINTER(_int)], _int),
    "attn_decode_fused_paged": ([_vp] * 10 + [_int] * 8 + [_flt, _vp], _int),
    "attn_fwd_splitkv": ([_vp] * 5 + [_int] * 8 + [_flt, _vp], _int),
    "attn_fwd_num_splits": ([_int] * 6 + [ctypes.POINTER(_int)], _int),
    "attn_rope_table": ([_vp, _int, _int, _flt, _vp], _int),
    "attn_decode_num_splits": ([_int, _int, _int, _int, _int, ctypes.POINTER(_int)], _int),
    "attn_qkv_rope": ([_vp] * 7 + [_int] * 8 + [_vp], _int),
    "attn_bwd": ([_vp] * 10 + [_int] * 7 + [_flt, _vp], _int),
    "attn_status_string": ([_int], ctypes.c_char_p),
    "attn_debug_status": ([_vp], _int),
    "attn_wait_selftest": ([ctypes.c_ulonglong, _vp, _vp], _int),
    "attn_version": ([], _int),
}


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = int(status)
        msg = attn_status_string(status)
        super().__init__(f"{what}: {msg}" if what else msg)


def library_path() -> str:
    return os.path.join(_PKG_DIR, _LIB_NAME)


def load_library():
    """Load libattn.so (built by ``tensor_attn_fwd_gb300.build``); raise if absent."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise ImportError(
                    f"{path} is missing: build it with `python -m tensor_attn_fwd_gb300.build` "
                    "(or __graft_entry__.build()); there is no fallback implementation")
            lib = ctypes.CDLL(path)
            for name, (argtypes, restype) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = argtypes
                fn.restype = restype
            _lib = lib
    return _lib


def attn_status_string(status: int) -> str:
    return load_library().attn_status_string(int(status)).decode()


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def attn_debug_status(stream=None) -> int:
    """Synchronise ``stream`` and return (and clear) the device status word."""
    return int(load_library().attn_debug_status(_stream_handle(stream)))


def attn_wait_selftest(limit_ns: int, stream=None):
    """Run the bounded-wait self-test kernel (a wait on an mbarrier that nothing
    arrives on, given up after ``limit_ns``) and return ``(status, waited_ns)``:
    the device status it left (ATTN_ERR_TIMEOUT when the bounded wait works) and
    how long the wait took on the device clock."""
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    st = int(load_library().attn_wait_selftest(int(limit_ns), waited.data_ptr(),
                                                _stream_handle(stream)))
    if st != ATTN_OK:
        raise AttnError(st, "attn_wait_selftest")
    status = attn_debug_status(stream)
    return status, int(waited.item())


def _check(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def _check_bf16(name: str, t: torch.Tensor, ndim: int):
    _check(isinstance(t, torch.Tensor), f"{name} must be a torch.Tensor")
    _check(t.is_cuda, f"{name} must be a CUDA tensor")
    _check(t.dtype == torch.bfloat16, f"{name} must be bfloat16, got {t.dtype}")
    _check(t.dim() == ndim, f"{name} must have {ndim} dims, got {t.dim()}")
    _check(t.is_contiguous(), f"{name} must be contiguous")


def _out(t, shape, device, name):
    if t is None:
        return torch.empty(shape, dtype=torch.float32, device=device)
    _check(t.is_cuda and t.dtype == torch.float32 and t.is_contiguous(),
           f"{name} must be a contiguous float32 CUDA tensor")
    _check(tuple(t.shape) == tuple(shape), f"{name} must have shape {tuple(shape)}")
    _check(t.device == device, f"{name} must be on {device}")
    return t


def _out_bf16(t, shape, device, name):
    if t is None:
        return torch.empty(shape, dtype=torch.bfloat16, device=device)
    _check(t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous(),
           f"{name} must be a contiguous bf16 CUDA tensor")
    _check(tuple(t.shape) == tuple(shape), f"{name} must have shape {tuple(shape)}")
    _check(t.device == device, f"{name} must be on {device}")
    return t


def _raise_if(status: int, what: str):
    if status != ATTN_OK:
        raise AttnError(status, what)


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
             scale: float | None = None, o: torch.Tensor | None = None,
             lse: torch.Tensor | None = None, stream=None, num_splits=1):
    """Attention forward: O = softmax(Q K^T * scale (+ causal mask)) V and its LSE.

    q [B,Hq,Sq,D], k/v [B,Hkv,Sk,D] (bf16, contiguous, same device).
    ``num_splits``: 1 (one pass), an int > 1 (split the keys, then combine:
    attn_fwd_splitkv + attn_combine, for too few query rows to fill the GPU),
    or "auto" (attn_fwd_num_splits picks).
    Returns (o [B,Hq,Sq,D] fp32, lse [B,Hq,Sq] fp32).
    """
    _check_bf16("q", q, 4)
    _check_bf16("k", k, 4)
    _check_bf16("v", v, 4)
    B, Hq, Sq, D = q.shape
    Bk, Hkv, Sk, Dk = k.shape
    _check(Bk == B and Dk == D and tuple(v.shape) == tuple(k.shape), "q/k/v shape mismatch")
    _check(k.device == q.device and v.device == q.device, "q/k/v must share a device")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = _out(o, (B, Hq, Sq, D), q.device, "o")
    lse = _out(lse, (B, Hq, Sq), q.device, "lse")
    if num_splits == "auto":
        num_splits = attn_fwd_num_splits(B, Hq, Hkv, Sq, Sk, D, device=q.device)
    if int(num_splits) > 1:
        o_part, lse_part = attn_fwd_splitkv(q, k, v, int(num_splits), causal, scale,
                                            stream=stream)
        lib = load_library()
        with torch.cuda.device(q.device):
            st = lib.attn_combine(o_part.data_ptr(), lse_part.data_ptr(), o.data_ptr(),
                                  lse.data_ptr(), B * Sq, Hq, D, int(num_splits),
                                  _stream_handle(stream))
        _raise_if(st, "attn_combine")
        return o, lse
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                          lse.data_ptr(), B, Hq, Hkv, Sq, Sk, D, int(bool(causal)),
                          float(scale), _stream_handle(stream))
    _raise_if(st, "attn_fwd")
    return o, lse


def attn_fwd_splitkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, num_splits: int,
                     causal: bool = False, scale: float | None = None,
                     o_part: torch.Tensor | None = None, lse_part: torch.Tensor | None = None,
                     stream=None):
    """Prefill forward over ``num_splits`` KV splits: the partials
    (o_part [ns,B,Hq,Sq,D] fp32, lse_part [ns,B,Hq,Sq] fp32) that attn_combine
    merges (see include/attn.h)."""
    _check_bf16("q", q, 4)
    _check_bf16("k", k, 4)
    _check_bf16("v", v, 4)
    B, Hq, Sq, D = q.shape
    Bk, Hkv, Sk, Dk = k.shape
    _check(Bk == B and Dk == D and tuple(v.shape) == tuple(k.shape), "q/k/v shape mismatch")
    _check(k.device == q.device and v.device == q.device, "q/k/v must share a device")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    ns = int(num_splits)
    o_part = _out(o_part, (ns, B, Hq, Sq, D), q.device, "o_part")
    lse_part = _out(lse_part, (ns, B, Hq, Sq), q.device, "lse_part")
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.attn_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o_part.data_ptr(),
                                  lse_part.data_ptr(), B, Hq, Hkv, Sq, Sk, D,
                                  int(bool(causal)), ns, float(scale), _stream_handle(stream))
    _raise_if(st, "attn_fwd_splitkv")
    return o_part, lse_part


def attn_fwd_num_splits(B: int, Hq: int, Hkv: int, Sq: int, Sk: int, D: int,
                        device=None) -> int:
    """Split count for attn_fwd_splitkv on ``device`` (measured rule, host only)."""
    lib = load_library()
    n = _int(0)
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        st = lib.attn_fwd_num_splits(int(B), int(Hq), int(Hkv), int(Sq), int(Sk), int(D),
                                     ctypes.byref(n))
    _raise_if(st, "attn_fwd_num_splits")
    return int(n.value)


def attn_fwd_bf16o(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
                   scale: float | None = None, o: torch.Tensor | None = None,
                   lse: torch.Tensor | None = None, stream=None):
    """attn_fwd with O returned in bf16 (LSE stays fp32)."""
    _check_bf16("q", q, 4)
    _check_bf16("k", k, 4)
    _check_bf16("v", v, 4)
    B, Hq, Sq, D = q.shape
    Bk, Hkv, Sk, Dk = k.shape
    _check(Bk == B and Dk == D and tuple(v.shape) == tuple(k.shape), "q/k/v shape mismatch")
    _check(k.device == q.device and v.device == q.device, "q/k/v must share a device")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if o is None:
        o = torch.empty((B, Hq, Sq, D), dtype=torch.bfloat16, device=q.device)
    _check(o.is_cuda and o.dtype == torch.bfloat16 and o.is_contiguous()
           and tuple(o.shape) == (B, Hq, Sq, D) and o.device == q.device,
           "o must be a contiguous bf16 CUDA tensor [B,Hq,Sq,D]")
    lse = _out(lse, (B, Hq, Sq), q.device, "lse")
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.attn_fwd_bf16o(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                lse.data_ptr(), B, Hq, Hkv, Sq, Sk, D, int(bool(causal)),
                                float(scale), _stream_handle(stream))
    _raise_if(st, "attn_fwd_bf16o")
    return o, lse


def attn_decode_splitkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, num_splits: int,
                        scale: float | None = None, o_part: torch.Tensor | None = None,
                        lse_part: torch.Tensor | None = None, stream=None):
    """Split-KV decode partials for q [B,Hq,1,D] against k/v [B,Hkv,Sk,D].

    Returns (o_part [num_splits,B,Hq,D], lse_part [num_splits,B,Hq]) fp32.
    """
    _check_bf16("q", q, 4)
    _check_bf16("k", k, 4)
    _check_bf16("v", v, 4)
    B, Hq, Sq, D = q.shape
    _check(Sq == 1, "decode takes one query row per head (q.shape[2] == 1)")
    Bk, Hkv, Sk, Dk = k.shape
    _check(Bk == B and Dk == D and tuple(v.shape) == tuple(k.shape), "q/k/v shape mismatch")
    _check(k.device == q.device and v.device == q.device, "q/k/v must share a device")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    ns = int(num_splits)
    o_part = _out(o_part, (ns, B, Hq, D), q.device, "o_part")
    lse_part = _out(lse_part, (ns, B, Hq), q.device, "lse_part")
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.attn_decode_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                     o_part.data_ptr(), lse_part.data_ptr(), B, Hq, Hkv, Sk, D,
                                     ns, float(scale), _stream_handle(stream))
    _raise_if(st, "attn_decode_splitkv")
    return o_part, lse_part


def attn_decode_splitkv_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                               seqlens: torch.Tensor, num_splits: int,
                               scale: float | None = None, o_part: torch.Tensor | None = None,
                               lse_part: torch.Tensor | None = None, stream=None):
    """Split-KV decode partials where sequence b attends to its first seqlens[b] keys.

    k/v are [B,Hkv,Sk,D] buffers of capacity Sk; seqlens is an int32 CUDA tensor [B].
    """
    _check_bf16("q", q, 4)
    _check_bf16("k", k, 4)
    _check_bf16("v", v, 4)
    B, Hq, Sq, D = q.shape
    _check(Sq == 1, "decode takes one query row per head (q.shape[2] == 1)")
    Bk, Hkv, Sk, Dk = k.shape
    _check(Bk == B and Dk == D and tuple(v.shape) == tuple(k.shape), "q/k/v shape mismatch")
    _check(isinstance(seqlens, torch.Tensor) and seqlens.is_cuda and seqlens.dtype == torch.int32
           and seqlens.is_contiguous() and tuple(seqlens.shape) == (B,),
           "seqlens must be a contiguous int32 CUDA tensor of shape [B]")
    _check(k.device == q.device and v.device == q.device and seqlens.device == q.device,
           "q/k/v/seqlens must share a device")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    ns = int(num_splits)
    o_part = _out(o_part, (ns, B, Hq, D), q.device, "o_part")
    lse_part = _out(lse_part, (ns, B, Hq), q.device, "lse_part")
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.attn_decode_splitkv_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                            seqlens.data_ptr(), o_part.data_ptr(),
                                            lse_part.data_ptr(), B, Hq, Hkv, Sk, D, ns,
                                            float(scale), _stream_handle(stream))
    _raise_if(st, "attn_decode_splitkv_varlen")
    return o_part, lse_part


def attn_decode_splitkv_paged(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                              block_table: torch.Tensor, seqlens: torch.Tensor, num_splits: int,
                              scale: float | None = None, o_part: torch.Tensor | None = None,
                              lse_part: torch.Tensor | None = None, stream=None):
    """Split-KV decode partials over a paged cache.

    k_cache/v_cache [num_pages,Hkv,page_size,D] bf16; block_table int32 CUDA
    [B,max_pages]; seqlens int32 CUDA [B].  Key t of sequence b is row
    t % page_size of page block_table[b, t // page_size].
    """
    _check_bf16("q", q, 4)
    _check_bf16("k_cache", k_cache, 4)
    _check_bf16("v_cache", v_cache, 4)
    B, Hq, Sq, D = q.shape
    _check(Sq == 1, "decode takes one query row per head (q.shape[2] == 1)")
    num_pages, Hkv, page_size, Dk = k_cache.shape
    _check(Dk == D and tuple(v_cache.shape) == tuple(k_cache.shape), "q/cache shape mismatch")
    for name, t in (("block_table", block_table), ("seqlens", seqlens)):
        _check(isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.int32
               and t.is_contiguous() and t.device == q.device,
               f"{name} must be a contiguous int32 tensor on q's device")
    _check(block_table.dim() == 2 and block_table.shape[0] == B, "block_table must be [B, max_pages]")
    _check(tuple(seqlens.shape) == (B,), "seqlens must be [B]")
    _check(k_cache.device == q.device and v_cache.device == q.device, "q and caches must share a device")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    ns = int(num_splits)
    o_part = _out(o_part, (ns, B, Hq, D), q.device, "o_part")
    lse_part = _out(lse_part, (ns, B, Hq), q.device, "lse_part")
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.attn_decode_splitkv_paged(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                           block_table.data_ptr(), seqlens.data_ptr(),
                                           o_part.data_ptr(), lse_part.data_ptr(), B, Hq, Hkv,
                                           num_pages, page_size, block_table.shape[1], D, ns,
                                           float(scale), _stream_handle(stream))
    _raise_if(st, "attn_decode_splitkv_paged")
    return o_part, lse_part


def decode_paged(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                 block_table: torch.Tensor, seqlens: torch.Tensor, num_splits: int,
                 scale: float | None = None, workspace=None, o=None, lse=None, stream=None,
                 counters: torch.Tensor | None = None):
    """Paged split-KV decode with the LSE combine fused in (one launch,
    attn_decode_fused_paged); returns (o [B,Hq,D], lse [B,Hq]).

    Cache layout and arguments as attn_decode_splitkv_paged; ``workspace`` is an
    optional (o_part, lse_part) pair for the partials, ``counters`` as
    attn_decode_fused.
    """
    _check_bf16("q", q, 4)
    _check_bf16("k_cache", k_cache, 4)
    _check_bf16("v_cache", v_cache, 4)
    B, Hq, Sq, D = q.shape
    _check(Sq == 1, "decode takes one query row per head (q.shape[2] == 1)")
    num_pages, Hkv, page_size, Dk = k_cache.shape
    _check(Dk == D and tuple(v_cache.shape) == tuple(k_cache.shape), "q/cache shape mismatch")
    for name, t in (("block_table", block_table), ("seqlens", seqlens)):
        _check(isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.int32
               and t.is_contiguous() and t.device == q.device,
               f"{name} must be a contiguous int32 tensor on q's device")
    _check(block_table.dim() == 2 and block_table.shape[0] == B, "block_table must be [B, max_pages]")
    _check(tuple(seqlens.shape) == (B,), "seqlens must be [B]")
    _check(k_cache.device == q.device and v_cache.device == q.device, "q and caches must share a device")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    ns = int(num_splits)
    o_part, lse_part = (None, None) if workspace is None else workspace
    o_part = _out(o_part, (ns, B, Hq, D), q.device, "o_part")
    lse_part = _out(lse_part, (ns, B, Hq), q.device, "lse_part")
    o = _out(o, (B, Hq, D), q.device, "o")
    lse = _out(lse, (B, Hq), q.device, "lse")
    lib = load_library()
    n = ctypes.c_int(0)
    _raise_if(lib.attn_decode_fused_counters(B, Hq, Hkv, ctypes.byref(n)),
              "attn_decode_fused_counters")
    if counters is None:
        counters = _stream_counters(q.device, stream, n.value)
    _check(isinstance(counters, torch.Tensor) and counters.is_cuda
           and counters.dtype == torch.int32 and counters.is_contiguous()
           and counters.numel() >= n.value and counters.device == q.device,
           f"counters must be a contiguous int32 CUDA tensor with >= {n.value} entries")
    with torch.cuda.device(q.device):
        st = lib.attn_decode_fused_paged(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                         block_table.data_ptr(), seqlens.data_ptr(), o.data_ptr(),
                                         lse.data_ptr(), o_part.data_ptr(), lse_part.data_ptr(),
                                         counters.data_ptr(), B, Hq, Hkv, num_pages, page_size,
                                         block_table.shape[1], D, ns, float(scale),
                                         _stream_handle(stream))
    _raise_if(st, "attn_decode_fused_paged")
    return o, lse


def attn_rope_table(max_pos: int, D: int, base: float = 10000.0, device=None,
                    out: torch.Tensor | None = None, stream=None):
    """(cos, sin) table [max_pos, D/2, 2] fp32 of pos * base^(-2i/D), built on the GPU."""
    if out is None:
        dev = torch.device("cuda") if device is None else torch.device(device)
        out = torch.empty((int(max_pos), int(D) // 2, 2), dtype=torch.float32, device=dev)
    _check(out.is_cuda and out.dtype == torch.float32 and out.is_contiguous()
           and tuple(out.shape) == (int(max_pos), int(D) // 2, 2),
           "out must be a contiguous float32 CUDA tensor [max_pos, D/2, 2]")
    lib = load_library()
    with torch.cuda.device(out.device):
        st = lib.attn_rope_table(out.data_ptr(), int(max_pos), int(D), float(base),
                                 _stream_handle(stream))
    _raise_if(st, "attn_rope_table")
    return out


def attn_qkv_rope(x: torch.Tensor, w: torch.Tensor, rope_table: torch.Tensor, Hq: int, Hkv: int,
                  positions: torch.Tensor | None = None, style: int = 0,
                  q: torch.Tensor | None = None, k: torch.Tensor | None = None,
                  v: torch.Tensor | None = None, stream=None):
    """Q, K, V = RoPE(x w^T) split into heads, in the [B, H, S, D] layout of attn_fwd.

    x [B, S, hidden] bf16; w [(Hq+2*Hkv)*D, hidden] bf16 (rows of Wq, Wk, Wv);
    rope_table from attn_rope_table ([max_pos, D/2, 2]); positions int32 [B, S]
    (default: s).  style 0 rotates dims (2i, 2i+1), style 1 dims (i, i+D/2).
    Returns bf16 q [B,Hq,S,D], k [B,Hkv,S,D], v [B,Hkv,S,D].
    """
    _check_bf16("x", x, 3)
    _check(isinstance(w, torch.Tensor) and w.is_cuda and w.dtype == torch.bfloat16
           and w.is_contiguous() and w.dim() == 2, "w must be a contiguous 2-D bf16 CUDA tensor")
    B, S, hidden = x.shape
    max_pos, half, two = rope_table.shape
    D = 2 * half
    _check(two == 2 and rope_table.dtype == torch.float32 and rope_table.is_contiguous()
           and rope_table.device == x.device, "rope_table must come from attn_rope_table")
    _check(tuple(w.shape) == ((Hq + 2 * Hkv) * D, hidden), "w must be [(Hq+2*Hkv)*D, hidden]")
    _check(w.device == x.device, "x and w must share a device")
    pos_ptr = 0
    if positions is not None:
        _check(positions.is_cuda and positions.dtype == torch.int32 and positions.is_contiguous()
               and positions.numel() == B * S and positions.device == x.device,
               "positions must be a contiguous int32 CUDA tensor with B*S entries")
        pos_ptr = positions.data_ptr()
    q = _out_bf16(q, (B, Hq, S, D), x.device, "q")
    k = _out_bf16(k, (B, Hkv, S, D), x.device, "k")
    v = _out_bf16(v, (B, Hkv, S, D), x.device, "v")
    lib = load_library()
    with torch.cuda.device(x.device):
        st = lib.attn_qkv_rope(x.data_ptr(), w.data_ptr(), rope_table.data_ptr(), pos_ptr or None,
                               q.data_ptr(), k.data_ptr(), v.data_ptr(), B, S, hidden, Hq, Hkv,
                               D, max_pos, int(style), _stream_handle(stream))
    _raise_if(st, "attn_qkv_rope")
    return q, k, v


def attn_combine(o_part: torch.Tensor, lse_part: torch.Tensor, o: torch.Tensor | None = None,
                 lse: torch.Tensor | None = None, stream=None):
    """LSE combine: o_part [ns,B,Hq,D], lse_part [ns,B,Hq] -> (o [B,Hq,D], lse [B,Hq])."""
    _check(o_part.is_cuda and o_part.dtype == torch.float32 and o_part.is_contiguous()
           and o_part.dim() == 4, "o_part must be a contiguous [ns,B,Hq,D] float32 CUDA tensor")
    ns, B, Hq, D = o_part.shape
    _check(lse_part.is_cuda and lse_part.dtype == torch.float32 and lse_part.is_contiguous()
           and tuple(lse_part.shape) == (ns, B, Hq), "lse_part must be [ns,B,Hq] float32")
    o = _out(o, (B, Hq, D), o_part.device, "o")
    lse = _out(lse, (B, Hq), o_part.device, "lse")
    lib = load_library()
    with torch.cuda.device(o_part.device):
        st = lib.attn_combine(o_part.data_ptr(), lse_part.data_ptr(), o.data_ptr(),
                              lse.data_ptr(), B, Hq, D, ns, _stream_handle(stream))
    _raise_if(st, "attn_combine")
    return o, lse


def attn_decode_num_splits(B: int, Hq: int, Hkv: int, Sk: int, D: int = 128,
                           device=None) -> int:
    """Split count for the decode kernels on ``device`` (measured rule, host only)."""
    lib = load_library()
    n = _int(0)
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        st = lib.attn_decode_num_splits(int(B), int(Hq), int(Hkv), int(Sk), int(D),
                                        ctypes.byref(n))
    _raise_if(st, "attn_decode_num_splits")
    return int(n.value)


# Zeroed int32 counter arrays for attn_decode_fused, one per (device, stream):
# a call leaves its counters zero, so calls on one stream share an array and
# calls on different streams (which may overlap) never do.  At most
# _COUNTERS_KEPT streams are remembered (the least recently used is dropped;
# its array was allocated on its own stream, so the allocator reuses it only
# after that stream's work).
_counters = {}
_counters_lock = threading.Lock()
_COUNTERS_KEPT = 256


def _stream_counters(device: torch.device, stream, n: int) -> torch.Tensor:
    handle = _stream_handle(stream)
    key = (device.index, handle)
    with _counters_lock:
        buf = _counters.pop(key, None)
        if buf is None or buf.numel() < n:
            # Zeroed on the call's own stream, so the memset precedes the kernel.
            with torch.cuda.device(device), torch.cuda.stream(
                    torch.cuda.ExternalStream(handle, device=device)):
                buf = torch.zeros(max(n, 1024), dtype=torch.int32, device=device)
        _counters[key] = buf  # most recently used last
        while len(_counters) > _COUNTERS_KEPT:
            _counters.pop(next(iter(_counters)))
    return buf


def attn_decode_fused(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, num_splits: int,
                      scale: float | None = None, seqlens: torch.Tensor | None = None,
                      o_part: torch.Tensor | None = None, lse_part: torch.Tensor | None = None,
                      o: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                      counters: torch.Tensor | None = None, stream=None):
    """Split-KV decode and its LSE combine in one launch; returns (o [B,Hq,D], lse [B,Hq]).

    The partials land in o_part [num_splits,B,Hq,D] / lse_part [num_splits,B,Hq]
    as with attn_decode_splitkv.  ``counters`` (int32 CUDA, at least
    attn_decode_fused_counters entries, zero) defaults to a cached zeroed array of
    the call's stream.  With ``seqlens`` sequence b attends to its first seqlens[b] keys.
    """
    _check_bf16("q", q, 4)
    _check_bf16("k", k, 4)
    _check_bf16("v", v, 4)
    B, Hq, Sq, D = q.shape
    _check(Sq == 1, "decode takes one query row per head (q.shape[2] == 1)")
    Bk, Hkv, Sk, Dk = k.shape
    _check(Bk == B and Dk == D and tuple(v.shape) == tuple(k.shape), "q/k/v shape mismatch")
    _check(k.device == q.device and v.device == q.device, "q/k/v must share a device")
    seq_ptr = None
    if seqlens is not None:
        _check(isinstance(seqlens, torch.Tensor) and seqlens.is_cuda
               and seqlens.dtype == torch.int32 and seqlens.is_contiguous()
               and tuple(seqlens.shape) == (B,) and seqlens.device == q.device,
               "seqlens must be a contiguous int32 CUDA tensor of shape [B] on q's device")
        seq_ptr = seqlens.data_ptr()
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    ns = int(num_splits)
    o_part = _out(o_part, (ns, B, Hq, D), q.device, "o_part")
    lse_part = _out(lse_part, (ns, B, Hq), q.device, "lse_part")
    o = _out(o, (B, Hq, D), q.device, "o")
    lse = _out(lse, (B, Hq), q.device, "lse")
    lib = load_library()
    n = ctypes.c_int(0)
    _raise_if(lib.attn_decode_fused_counters(B, Hq, Hkv, ctypes.byref(n)),
              "attn_decode_fused_counters")
    if counters is None:
        counters = _stream_counters(q.device, stream, n.value)
    _check(isinstance(counters, torch.Tensor) and counters.is_cuda
           and counters.dtype == torch.int32 and counters.is_contiguous()
           and counters.numel() >= n.value and counters.device == q.device,
           f"counters must be a contiguous int32 CUDA tensor with >= {n.value} entries")
    with torch.cuda.device(q.device):
        st = lib.attn_decode_fused(q.data_ptr(), k.data_ptr(), v.data_ptr(), seq_ptr,
                                   o.data_ptr(), lse.data_ptr(), o_part.data_ptr(),
                                   lse_part.data_ptr(), counters.data_ptr(), B, Hq, Hkv, Sk, D,
                                   ns, float(scale), _stream_handle(stream))
    _raise_if(st, "attn_decode_fused")
    return o, lse


def decode(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, num_splits: int | None = None,
           scale: float | None = None, workspace=None, o=None, lse=None, stream=None,
           seqlens: torch.Tensor | None = None):
    """Split-KV decode with the LSE combine fused in (one launch, attn_decode_fused);
    returns (o [B,Hq,D], lse [B,Hq]).

    With ``seqlens`` (int32 CUDA [B]) sequence b attends to its first seqlens[b] keys.
    ``num_splits=None`` picks attn_decode_num_splits for the shape; ``workspace`` is
    an optional (o_part, lse_part) pair for the partials.
    """
    if num_splits is None:
        num_splits = attn_decode_num_splits(q.shape[0], q.shape[1], k.shape[1], k.shape[2],
                                            k.shape[3], q.device)
    o_part, lse_part = (None, None) if workspace is None else workspace
    return attn_decode_fused(q, k, v, num_splits, scale, seqlens, o_part, lse_part, o, lse,
                             stream=stream)


def attn_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
             lse: torch.Tensor, dout: torch.Tensor, causal: bool = False,
             scale: float | None = None, dq: torch.Tensor | None = None,
             dk: torch.Tensor | None = None, dv: torch.Tensor | None = None,
             delta_ws: torch.Tensor | None = None, stream=None):
    """Gradients of sum(dout * O) for O = attn_fwd(q, k, v): returns (dq, dk, dv) fp32.

    o and lse are attn_fwd's fp32 outputs; dout is bf16 like q.
    """
    _check_bf16("q", q, 4)
    _check_bf16("k", k, 4)
    _check_bf16("v", v, 4)
    _check_bf16("dout", dout, 4)
    B, Hq, Sq, D = q.shape
    Bk, Hkv, Sk, Dk = k.shape
    _check(Bk == B and Dk == D and tuple(v.shape) == tuple(k.shape), "q/k/v shape mismatch")
    _check(tuple(dout.shape) == tuple(q.shape), "dout must match q")
    for name, t in (("k", k), ("v", v), ("dout", dout)):
        _check(t.device == q.device, f"{name} must be on {q.device}")
    o = _out(o, (B, Hq, Sq, D), q.device, "o")
    lse = _out(lse, (B, Hq, Sq), q.device, "lse")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq = _out(dq, (B, Hq, Sq, D), q.device, "dq")
    dk = _out(dk, (B, Hkv, Sk, D), q.device, "dk")
    dv = _out(dv, (B, Hkv, Sk, D), q.device, "dv")
    delta_ws = _out(delta_ws, (B, Hq, Sq), q.device, "delta_ws")
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                          dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                          delta_ws.data_ptr(), B, Hq, Hkv, Sq, Sk, D, int(bool(causal)),
                          float(scale), _stream_handle(stream))
    _raise_if(st, "attn_bwd")
    return dq, dk, dv
