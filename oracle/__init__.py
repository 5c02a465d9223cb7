"""fp64 CPU oracle for the attention forward -- TEST INFRASTRUCTURE ONLY.

The arithmetic lives in ``attn_oracle.c`` (plain C, double precision, OpenMP
over rows); this module compiles it with gcc and marshals arguments through
ctypes.  It shares no code with the CUDA library and imports nothing from it.
Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may use it.

Definition followed: "A Thread-Register Decoupled GPU Execution Model for
Efficient Tensor Computation", Background (Equ. 1, multi-head attention) and
Methodology (GQA / MQA head sharing, FlashDecoding for decode); the equation
itself is not printed on the page, so the standard scaled-dot-product
attention with a bottom-right causal mask and a natural-log LSE is written out
in the C file's header.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_dbl = ctypes.c_double
_vp = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (gcc, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_attn_fwd_rows.argtypes = [
                _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _i64, ctypes.c_int,
                _dbl, _vp, _i64, _vp, _vp]
            lib.oracle_attn_fwd_rows.restype = ctypes.c_int
            lib.oracle_decode_split.argtypes = [
                _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _dbl, _vp, _vp]
            lib.oracle_decode_split.restype = ctypes.c_int
            lib.oracle_combine.argtypes = [_vp, _vp, _i64, _i64, _i64, _vp, _vp]
            lib.oracle_combine.restype = ctypes.c_int
            lib.oracle_attn_fwd_f64.argtypes = [
                _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _i64, ctypes.c_int, _dbl, _vp, _vp]
            lib.oracle_attn_fwd_f64.restype = ctypes.c_int
            lib.oracle_attn_bwd_f64.argtypes = [
                _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _i64, ctypes.c_int, _dbl,
                _vp, _vp, _vp]
            lib.oracle_attn_bwd_f64.restype = ctypes.c_int
            lib.oracle_attn_bwd_sampled.argtypes = [
                _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _i64, ctypes.c_int, _dbl,
                _vp, _i64, _vp, _i64, _vp, _vp, _vp]
            lib.oracle_attn_bwd_sampled.restype = ctypes.c_int
            lib.oracle_qkv_rope.argtypes = [
                _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _dbl, ctypes.c_int, _vp, _i64,
                _vp, _vp, _vp]
            lib.oracle_qkv_rope.restype = ctypes.c_int
            _lib = lib
    return _lib


def _bf16_bits(x) -> np.ndarray:
    """Contiguous uint16 view of a bf16 tensor (torch) or a uint16 array."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("numpy inputs must be uint16 bf16 bit patterns")
        return np.ascontiguousarray(x)
    import torch  # local: plain CPU tensors only
    if x.dtype != torch.bfloat16:
        raise TypeError("oracle inputs must be bf16")
    return x.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_vp)


def attn_fwd(q, k, v, causal: bool, scale: float, rows=None):
    """O (float64 [..., D]) and LSE (float64) for Q [B,Hq,Sq,D], K/V [B,Hkv,Sk,D].

    ``rows`` (optional): flat row ids (b*Hq + h)*Sq + i; then O is [n, D] and
    LSE is [n].  Otherwise O is [B,Hq,Sq,D] and LSE is [B,Hq,Sq].
    """
    B, Hq, Sq, D = (int(s) for s in q.shape)
    Bk, Hkv, Sk, Dk = (int(s) for s in k.shape)
    if Bk != B or Dk != D or tuple(v.shape) != tuple(k.shape):
        raise ValueError("shape mismatch")
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    if rows is None:
        n = B * Hq * Sq
        rp = None
    else:
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n = rows.size
        rp = _ptr(rows)
    o = np.empty((n, D), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    rc = _load().oracle_attn_fwd_rows(_ptr(qb), _ptr(kb), _ptr(vb), B, Hq, Hkv, Sq,
                                      Sk, D, int(bool(causal)), float(scale), rp, n,
                                      _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_attn_fwd_rows failed ({rc})")
    if rows is None:
        return o.reshape(B, Hq, Sq, D), lse.reshape(B, Hq, Sq)
    return o, lse


def decode_split(q, k, v, num_splits: int, scale: float, align: int = 1):
    """Per-split partials: O_s [ns,B,Hq,D] and LSE_s [ns,B,Hq] (float64).

    Split s covers keys [s*c, min(Sk, (s+1)*c)) with c = ceil(Sk/ns) rounded up
    to a multiple of ``align``.
    """
    B, Hq, Sq, D = (int(s) for s in q.shape)
    if Sq != 1:
        raise ValueError("decode takes one query row per head")
    _, Hkv, Sk, _ = (int(s) for s in k.shape)
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    ns = int(num_splits)
    o = np.empty((ns, B, Hq, D), dtype=np.float64)
    lse = np.empty((ns, B, Hq), dtype=np.float64)
    rc = _load().oracle_decode_split(_ptr(qb), _ptr(kb), _ptr(vb), B, Hq, Hkv, Sk, D,
                                     ns, int(align), float(scale), _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_decode_split failed ({rc})")
    return o, lse


def combine(o_part, lse_part):
    """LSE combine: o_part [ns,...,D], lse_part [ns,...] -> (O [...,D], LSE [...])."""
    o_part = np.ascontiguousarray(np.asarray(o_part, dtype=np.float64))
    lse_part = np.ascontiguousarray(np.asarray(lse_part, dtype=np.float64))
    ns = o_part.shape[0]
    D = o_part.shape[-1]
    rest = o_part.shape[1:-1]
    R = int(np.prod(rest)) if rest else 1
    if lse_part.shape != (ns,) + tuple(rest):
        raise ValueError("lse_part shape mismatch")
    o = np.empty(tuple(rest) + (D,), dtype=np.float64)
    lse = np.empty(tuple(rest), dtype=np.float64)
    rc = _load().oracle_combine(_ptr(o_part), _ptr(lse_part), R, D, ns, _ptr(o),
                                _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_combine failed ({rc})")
    return o, lse


def _f64(x) -> np.ndarray:
    """Contiguous float64 copy of a tensor/array (bf16 values widen exactly)."""
    if isinstance(x, np.ndarray):
        return np.ascontiguousarray(x, dtype=np.float64)
    import torch
    return x.detach().to("cpu").to(torch.float64).contiguous().numpy()


def attn_fwd_f64(q, k, v, causal: bool, scale: float):
    """Forward on double inputs: O [B,Hq,Sq,D] and LSE [B,Hq,Sq] (float64)."""
    qd, kd, vd = _f64(q), _f64(k), _f64(v)
    B, Hq, Sq, D = qd.shape
    _, Hkv, Sk, _ = kd.shape
    o = np.empty((B, Hq, Sq, D))
    lse = np.empty((B, Hq, Sq))
    rc = _load().oracle_attn_fwd_f64(_ptr(qd), _ptr(kd), _ptr(vd), B, Hq, Hkv, Sq, Sk, D,
                                     int(bool(causal)), float(scale), _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_attn_fwd_f64 failed ({rc})")
    return o, lse


def attn_bwd(q, k, v, dout, causal: bool, scale: float):
    """Gradients (dQ, dK, dV) of sum(dO * O) for Q [B,Hq,Sq,D], K/V [B,Hkv,Sk,D] (float64)."""
    qd, kd, vd, dod = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, Hq, Sq, D = qd.shape
    _, Hkv, Sk, _ = kd.shape
    if dod.shape != qd.shape:
        raise ValueError("dO must match Q")
    dq = np.empty_like(qd)
    dk = np.empty_like(kd)
    dv = np.empty_like(vd)
    rc = _load().oracle_attn_bwd_f64(_ptr(qd), _ptr(kd), _ptr(vd), _ptr(dod), B, Hq, Hkv, Sq, Sk,
                                     D, int(bool(causal)), float(scale), _ptr(dq), _ptr(dk),
                                     _ptr(dv))
    if rc != 0:
        raise ValueError(f"oracle_attn_bwd_f64 failed ({rc})")
    return dq, dk, dv


def attn_bwd_sampled(q, k, v, dout, causal: bool, scale: float, qrows, keys):
    """Backward at sampled positions on bf16 inputs (any size).

    ``qrows``: flat query-row ids (b*Hq + h)*Sq + i -> dQ [nq, D].
    ``keys``: flat key ids (b*Hkv + g)*Sk + j -> dK, dV [nk, D] (summed over the
    group's query heads).  All float64.
    """
    B, Hq, Sq, D = (int(s) for s in q.shape)
    _, Hkv, Sk, _ = (int(s) for s in k.shape)
    if tuple(dout.shape) != tuple(q.shape) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("shape mismatch")
    qb, kb, vb, db = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v), _bf16_bits(dout)
    qrows = np.ascontiguousarray(np.asarray(qrows, dtype=np.int64))
    keys = np.ascontiguousarray(np.asarray(keys, dtype=np.int64))
    dq = np.empty((qrows.size, D))
    dk = np.empty((keys.size, D))
    dv = np.empty((keys.size, D))
    rc = _load().oracle_attn_bwd_sampled(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(db), B, Hq, Hkv, Sq,
                                         Sk, D, int(bool(causal)), float(scale), _ptr(qrows),
                                         qrows.size, _ptr(keys), keys.size, _ptr(dq), _ptr(dk),
                                         _ptr(dv))
    if rc != 0:
        raise ValueError(f"oracle_attn_bwd_sampled failed ({rc})")
    return dq, dk, dv


def gather_paged(cache, block_table, seqlens, b: int):
    """The keys (or values) of sequence ``b`` from a paged cache, in order.

    cache [num_pages, Hkv, page_size, D]; block_table [B, max_pages]; key t of
    sequence b is cache[block_table[b, t // page_size], :, t % page_size, :].
    Returns [1, Hkv, seqlens[b], D] with the cache's dtype.  Pure indexing.
    """
    import torch
    cache = cache.detach().to("cpu")
    table = block_table.detach().to("cpu").to(torch.int64)
    n = int(seqlens[b])
    num_pages, Hkv, page, D = cache.shape
    t = torch.arange(n, dtype=torch.int64)
    pages = table[b, t // page]
    if n and (int(pages.min()) < 0 or int(pages.max()) >= num_pages):
        raise ValueError("block table entry out of range")
    rows = cache[pages, :, t % page, :]          # [n, Hkv, D]
    return rows.permute(1, 0, 2).unsqueeze(0).contiguous()


def qkv_rope(x, w, positions, Hq: int, Hkv: int, D: int, base: float = 10000.0,
             style: int = 0, tokens=None):
    """QKV projection of x [T, hidden] by w [(Hq+2Hkv)*D, hidden] (bf16), then
    RoPE on the Q and K heads at positions [T] (int32).

    style 0 rotates dims (2i, 2i+1), style 1 rotates dims (i, i+D/2).
    Returns float64 q [n, Hq, D], k [n, Hkv, D], v [n, Hkv, D] for the tokens
    listed in ``tokens`` (default: all T).
    """
    xb, wb = _bf16_bits(x), _bf16_bits(w)
    T, hidden = xb.shape
    if wb.shape != ((Hq + 2 * Hkv) * D, hidden):
        raise ValueError("w must be [(Hq+2*Hkv)*D, hidden]")
    pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int32))
    if pos.shape != (T,):
        raise ValueError("positions must be [T]")
    toks = np.arange(T, dtype=np.int64) if tokens is None else \
        np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
    n = toks.size
    q = np.empty((n, Hq, D))
    k = np.empty((n, Hkv, D))
    v = np.empty((n, Hkv, D))
    rc = _load().oracle_qkv_rope(_ptr(xb), _ptr(wb), _ptr(pos), T, hidden, Hq, Hkv, D,
                                 float(base), int(style), _ptr(toks), n, _ptr(q), _ptr(k),
                                 _ptr(v))
    if rc != 0:
        raise ValueError(f"oracle_qkv_rope failed ({rc})")
    return q, k, v
