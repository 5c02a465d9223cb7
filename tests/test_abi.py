"""C-ABI checks that need no GPU: the library builds and loads, exports every
symbol include/attn.h declares, and rejects invalid arguments with the
documented status before touching the device (no compute call is made)."""
import ctypes
import os
import re

import pytest

import tensor_attn_fwd_gb300 as attn
from tensor_attn_fwd_gb300 import build as attn_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    attn_build.build()
    return attn.load_library()


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", text)


def test_header_declares_entry_points():
    names = set(declared_symbols())
    assert {"attn_fwd", "attn_decode_splitkv", "attn_combine", "attn_status_string",
            "attn_debug_status", "attn_version"} <= names


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert names
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"


def test_status_strings(lib):
    for code in range(7):
        s = attn.attn_status_string(code)
        assert s and isinstance(s, str)
    assert "unknown" in attn.attn_status_string(99)
    assert lib.attn_version() >> 16 == 1


# Fake, never-dereferenced device addresses: validation fails before any launch.
A = 0x10000000       # 16-byte aligned
M = 0x10000004       # misaligned


def fwd(lib, q=A, k=A, v=A, o=A, lse=A, B=1, Hq=2, Hkv=1, Sq=8, Sk=8, D=64, causal=0,
        scale=0.125):
    return lib.attn_fwd(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, None)


def dec(lib, q=A, k=A, v=A, op=A, lp=A, B=1, Hq=4, Hkv=1, Sk=64, D=128, ns=4, scale=0.1):
    return lib.attn_decode_splitkv(q, k, v, op, lp, B, Hq, Hkv, Sk, D, ns, scale, None)


def decv(lib, q=A, k=A, v=A, sl=A, op=A, lp=A, B=1, Hq=4, Hkv=1, Sk=64, D=128, ns=4, scale=0.1):
    return lib.attn_decode_splitkv_varlen(q, k, v, sl, op, lp, B, Hq, Hkv, Sk, D, ns, scale,
                                          None)


@pytest.mark.parametrize("kw,code", [
    (dict(sl=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(sl=A + 2), attn.ATTN_ERR_MISALIGNED),
    (dict(q=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(ns=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(D=96), attn.ATTN_ERR_UNSUPPORTED),
    (dict(v=M), attn.ATTN_ERR_MISALIGNED),
])
def test_decode_varlen_rejects(lib, kw, code):
    assert decv(lib, **kw) == code


def decp(lib, q=A, k=A, v=A, bt=A, sl=A, op=A, lp=A, B=1, Hq=4, Hkv=1, num_pages=8, page=64,
         max_pages=4, D=128, ns=4, scale=0.1):
    return lib.attn_decode_splitkv_paged(q, k, v, bt, sl, op, lp, B, Hq, Hkv, num_pages, page,
                                         max_pages, D, ns, scale, None)


@pytest.mark.parametrize("kw,code", [
    (dict(bt=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(sl=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(bt=A + 2), attn.ATTN_ERR_MISALIGNED),
    (dict(sl=A + 1), attn.ATTN_ERR_MISALIGNED),
    (dict(page=48), attn.ATTN_ERR_UNSUPPORTED),      # not a multiple of 32
    (dict(page=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(num_pages=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(max_pages=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(ns=257), attn.ATTN_ERR_INVALID_ARG),      # more splits than the capacity
    (dict(max_pages=1 << 25, page=64), attn.ATTN_ERR_UNSUPPORTED),
    (dict(Hq=6, Hkv=4), attn.ATTN_ERR_INVALID_ARG),
    (dict(D=96), attn.ATTN_ERR_UNSUPPORTED),
    (dict(k=M), attn.ATTN_ERR_MISALIGNED),
    (dict(q=None), attn.ATTN_ERR_INVALID_ARG),
])
def test_decode_paged_rejects(lib, kw, code):
    assert decp(lib, **kw) == code


def noalloc(lib, q=A, k=A, v=A, o=A, lse=A, B=1, Hq=4, Hkv=1, Sk=64, D=128, ns=4, scale=0.1):
    f = lib.attn_decode_noalloc
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 6 + [ctypes.c_float, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f(q, k, v, o, lse, B, Hq, Hkv, Sk, D, ns, scale, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(o=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(lse=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(ns=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(ns=65), attn.ATTN_ERR_INVALID_ARG),     # more splits than keys
    (dict(Hq=6, Hkv=4), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), attn.ATTN_ERR_INVALID_ARG),
    (dict(D=80), attn.ATTN_ERR_UNSUPPORTED),
    (dict(B=70000), attn.ATTN_ERR_UNSUPPORTED),
    # Sequences past 2^30 keys would overflow the kernels' int split arithmetic;
    # the allocating decode rejects them and so must this one.
    (dict(Sk=(1 << 30) + 1, ns=8), attn.ATTN_ERR_UNSUPPORTED),
    (dict(Sk=2147483647, ns=8), attn.ATTN_ERR_UNSUPPORTED),
    # partials beyond the 4 Mi-float scratch array: 8 * 4096 * (128 + 1) floats
    (dict(B=1024, Hq=4, ns=8), attn.ATTN_ERR_UNSUPPORTED),
    (dict(k=M), attn.ATTN_ERR_MISALIGNED),
    (dict(o=M), attn.ATTN_ERR_MISALIGNED),
    (dict(lse=M), attn.ATTN_ERR_MISALIGNED),
])
def test_decode_noalloc_rejects(lib, kw, code):
    assert noalloc(lib, **kw) == code


def test_decode_noalloc_matches_decode_checks(lib):
    # Every input the allocating decode rejects, the allocation-free one rejects
    # with the same status (partials pointers aside).
    for kw in (dict(Sk=(1 << 30) + 1, ns=8), dict(D=96), dict(Hq=6, Hkv=4), dict(ns=0),
               dict(q=M), dict(scale=0.0)):
        assert noalloc(lib, **kw) == dec(lib, **kw)


def fused(lib, q=A, k=A, v=A, sl=None, o=A, lse=A, op=A, lp=A, cnt=A, B=1, Hq=4, Hkv=1, Sk=64,
          D=128, ns=4, scale=0.1):
    return lib.attn_decode_fused(q, k, v, sl, o, lse, op, lp, cnt, B, Hq, Hkv, Sk, D, ns, scale,
                                 None)


@pytest.mark.parametrize("kw,code", [
    (dict(cnt=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(o=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(lse=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(op=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(q=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(ns=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(ns=65), attn.ATTN_ERR_INVALID_ARG),   # more splits than keys
    (dict(Hq=6, Hkv=4), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), attn.ATTN_ERR_INVALID_ARG),
    (dict(D=80), attn.ATTN_ERR_UNSUPPORTED),
    (dict(B=70000), attn.ATTN_ERR_UNSUPPORTED),
    (dict(Sk=(1 << 30) + 1, ns=8), attn.ATTN_ERR_UNSUPPORTED),
    (dict(k=M), attn.ATTN_ERR_MISALIGNED),
    (dict(o=M), attn.ATTN_ERR_MISALIGNED),
    (dict(lse=M), attn.ATTN_ERR_MISALIGNED),
    (dict(cnt=A + 2), attn.ATTN_ERR_MISALIGNED),
    (dict(sl=A + 2), attn.ATTN_ERR_MISALIGNED),
])
def test_decode_fused_rejects(lib, kw, code):
    assert fused(lib, **kw) == code


def test_decode_fused_matches_decode_checks(lib):
    # The fused decode rejects every input the two-launch decode rejects, with
    # the same status.
    for kw in (dict(Sk=(1 << 30) + 1, ns=8), dict(D=96), dict(Hq=6, Hkv=4), dict(ns=0),
               dict(q=M), dict(scale=0.0), dict(B=70000)):
        assert fused(lib, **kw) == dec(lib, **kw)


def fusedp(lib, q=A, k=A, v=A, bt=A, sl=A, o=A, lse=A, op=A, lp=A, cnt=A, B=1, Hq=4, Hkv=1,
           num_pages=8, page=64, max_pages=4, D=128, ns=4, scale=0.1):
    return lib.attn_decode_fused_paged(q, k, v, bt, sl, o, lse, op, lp, cnt, B, Hq, Hkv, num_pages,
                                       page, max_pages, D, ns, scale, None)


def test_decode_fused_paged_matches_paged_checks(lib):
    # Every cache description or argument the two-launch paged decode rejects,
    # the fused one rejects with the same status.
    for kw in (dict(bt=None), dict(sl=None), dict(num_pages=0), dict(page=48), dict(bt=A + 2),
               dict(max_pages=1 << 25, page=64), dict(D=96), dict(Hq=6, Hkv=4), dict(ns=0),
               dict(q=M), dict(scale=0.0), dict(op=M)):
        assert fusedp(lib, **kw) == decp(lib, **kw), kw
    assert fusedp(lib, cnt=None) == attn.ATTN_ERR_INVALID_ARG
    assert fusedp(lib, o=None) == attn.ATTN_ERR_INVALID_ARG
    assert fusedp(lib, lse=M) == attn.ATTN_ERR_MISALIGNED
    assert fusedp(lib, cnt=A + 2) == attn.ATTN_ERR_MISALIGNED


def test_decode_fused_counters(lib):
    n = ctypes.c_int(0)
    assert lib.attn_decode_fused_counters(64, 32, 8, ctypes.byref(n)) == attn.ATTN_OK
    assert n.value == 64 * 8          # group of 4 query heads: one 16-head slice
    assert lib.attn_decode_fused_counters(2, 64, 2, ctypes.byref(n)) == attn.ATTN_OK
    assert n.value == 2 * 2 * 2       # group of 32: two slices
    assert lib.attn_decode_fused_counters(1, 17, 1, ctypes.byref(n)) == attn.ATTN_OK
    assert n.value == 2
    assert lib.attn_decode_fused_counters(1, 6, 4, ctypes.byref(n)) == attn.ATTN_ERR_INVALID_ARG
    assert lib.attn_decode_fused_counters(0, 4, 1, ctypes.byref(n)) == attn.ATTN_ERR_INVALID_ARG
    assert lib.attn_decode_fused_counters(1, 4, 1, None) == attn.ATTN_ERR_INVALID_ARG


def comb(lib, op=A, lp=A, o=A, lse=A, B=1, Hq=4, D=128, ns=4):
    return lib.attn_combine(op, lp, o, lse, B, Hq, D, ns, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(o=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(lse=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(B=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(Sq=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(Sk=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(Hq=3, Hkv=2), attn.ATTN_ERR_INVALID_ARG),
    (dict(causal=2), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=0.0), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=-1.0), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("inf")), attn.ATTN_ERR_INVALID_ARG),
    (dict(D=96), attn.ATTN_ERR_UNSUPPORTED),
    (dict(D=192), attn.ATTN_ERR_UNSUPPORTED),
    (dict(D=512), attn.ATTN_ERR_UNSUPPORTED),
    (dict(Sq=(1 << 30) + 1), attn.ATTN_ERR_UNSUPPORTED),
    (dict(q=M), attn.ATTN_ERR_MISALIGNED),
    (dict(v=M), attn.ATTN_ERR_MISALIGNED),
    (dict(lse=M), attn.ATTN_ERR_MISALIGNED),
])
def test_fwd_rejects(lib, kw, code):
    assert fwd(lib, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(op=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(ns=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(ns=65), attn.ATTN_ERR_INVALID_ARG),   # more splits than keys
    (dict(Hq=6, Hkv=4), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=0.0), attn.ATTN_ERR_INVALID_ARG),
    (dict(D=80), attn.ATTN_ERR_UNSUPPORTED),
    (dict(B=70000), attn.ATTN_ERR_UNSUPPORTED),
    (dict(k=M), attn.ATTN_ERR_MISALIGNED),
    (dict(lp=M), attn.ATTN_ERR_MISALIGNED),
])
def test_decode_rejects(lib, kw, code):
    assert dec(lib, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(op=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(ns=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(B=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(D=32), attn.ATTN_ERR_UNSUPPORTED),
    (dict(o=M), attn.ATTN_ERR_MISALIGNED),
])
def test_combine_rejects(lib, kw, code):
    assert comb(lib, **kw) == code


def test_python_binding_checks_without_gpu():
    import torch
    q = torch.zeros(1, 2, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        attn.attn_fwd(q, q, q)  # CPU tensors are rejected before any call


def test_binding_has_no_fallback_import():
    # The product binding must not reach the oracle.
    src = open(os.path.join(ROOT, "tensor_attn_fwd_gb300", "__init__.py")).read()
    assert "oracle" not in src.replace("no CPU or PyTorch fallback", "")


def qkv(lib, x=A, w=A, t=A, pos=A, q=A, k=A, v=A, B=1, S=16, hidden=64, Hq=2, Hkv=1, D=64,
        max_pos=16, style=0):
    return lib.attn_qkv_rope(x, w, t, pos, q, k, v, B, S, hidden, Hq, Hkv, D, max_pos, style, None)


@pytest.mark.parametrize("kw,code", [
    (dict(x=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(t=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(v=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(S=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(Hq=3, Hkv=2), attn.ATTN_ERR_INVALID_ARG),
    (dict(style=2), attn.ATTN_ERR_INVALID_ARG),
    (dict(pos=None, max_pos=8), attn.ATTN_ERR_INVALID_ARG),   # positions s need max_pos >= S
    (dict(D=96), attn.ATTN_ERR_UNSUPPORTED),
    (dict(hidden=60), attn.ATTN_ERR_UNSUPPORTED),
    (dict(w=M), attn.ATTN_ERR_MISALIGNED),
    (dict(pos=A + 2), attn.ATTN_ERR_MISALIGNED),
])
def test_qkv_rope_rejects(lib, kw, code):
    assert qkv(lib, **kw) == code


@pytest.mark.parametrize("args,code", [
    ((None, 16, 64, 10000.0), attn.ATTN_ERR_INVALID_ARG),
    ((A, 0, 64, 10000.0), attn.ATTN_ERR_INVALID_ARG),
    ((A, 16, 63, 10000.0), attn.ATTN_ERR_INVALID_ARG),
    ((A, 16, 64, 1.0), attn.ATTN_ERR_INVALID_ARG),
    ((A, 16, 64, float("nan")), attn.ATTN_ERR_INVALID_ARG),
    ((M, 16, 64, 10000.0), attn.ATTN_ERR_MISALIGNED),
])
def test_rope_table_rejects(lib, args, code):
    assert lib.attn_rope_table(*args, None) == code


def test_decode_num_splits_rejects(lib):
    n = ctypes.c_int(0)
    assert lib.attn_decode_num_splits(1, 4, 1, 64, 128, None) == attn.ATTN_ERR_INVALID_ARG
    assert lib.attn_decode_num_splits(0, 4, 1, 64, 128, ctypes.byref(n)) == \
        attn.ATTN_ERR_INVALID_ARG
    assert lib.attn_decode_num_splits(1, 6, 4, 64, 128, ctypes.byref(n)) == \
        attn.ATTN_ERR_INVALID_ARG
    assert lib.attn_decode_num_splits(1, 4, 1, 64, 0, ctypes.byref(n)) == \
        attn.ATTN_ERR_INVALID_ARG


def bwdc(lib, B=1, Hq=2, Hkv=1, Sq=64, Sk=64, D=64, causal=0, scale=0.125, q=A):
    return lib.attn_bwd(q, A, A, A, A, A, A, A, A, A, B, Hq, Hkv, Sq, Sk, D, causal, scale, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(Sq=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(Hq=3, Hkv=2), attn.ATTN_ERR_INVALID_ARG),
    (dict(causal=3), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=0.0), attn.ATTN_ERR_INVALID_ARG),
    (dict(D=256), attn.ATTN_ERR_UNSUPPORTED),
    (dict(B=1024, Hq=1024, Sq=1025), attn.ATTN_ERR_UNSUPPORTED),   # > 2^30 Delta rows
    (dict(q=M), attn.ATTN_ERR_MISALIGNED),
])
def test_bwd_rejects(lib, kw, code):
    assert bwdc(lib, **kw) == code


def test_decode_rejects_too_many_rows(lib):
    # B * Hq above 2^30 output rows
    # (every other limit holds: B*Hkv*Sk*D and ns*B*Hq*D are small, Hkv*slices <= 65535)
    assert dec(lib, B=65535, Hq=32768, Hkv=1, Sk=1, D=64, ns=1) == attn.ATTN_ERR_UNSUPPORTED
    assert dec(lib, B=32768, Hq=32768, Hkv=1, Sk=1, D=64, ns=1, q=None) == attn.ATTN_ERR_INVALID_ARG


def test_wait_selftest_rejects(lib):
    """The bounded-wait self-test checks its limit and its output pointer
    before launching anything."""
    ull = ctypes.c_ulonglong
    lib.attn_wait_selftest.argtypes = [ull, ctypes.c_void_p, ctypes.c_void_p]
    assert lib.attn_wait_selftest(ull(0), None, None) == attn.ATTN_ERR_INVALID_ARG
    assert lib.attn_wait_selftest(ull(999), None, None) == attn.ATTN_ERR_INVALID_ARG
    assert lib.attn_wait_selftest(ull(1_000_000_001), None, None) == attn.ATTN_ERR_INVALID_ARG
    assert lib.attn_wait_selftest(ull(1_000_000), ctypes.c_void_p(4), None) == \
        attn.ATTN_ERR_MISALIGNED


def test_fwd_splitkv_rejects(lib):
    """attn_fwd_splitkv validates before launching: split count within
    [1, ceil(Sk/128)], D 64 or 128, non-null outputs."""
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.attn_fwd_splitkv.argtypes = [vp] * 5 + [i] * 8 + [f, vp]
    ptr = vp(256)

    def call(ns=2, D=128, o_part=ptr, Sk=1000):
        return lib.attn_fwd_splitkv(ptr, ptr, ptr, o_part, ptr, 1, 4, 2, 64, Sk, D, 1, ns,
                                    f(0.1), None)
    assert call(ns=0) == attn.ATTN_ERR_INVALID_ARG
    assert call(ns=9, Sk=1000) == attn.ATTN_ERR_INVALID_ARG   # 8 tiles of 128 keys
    assert call(D=256) == attn.ATTN_ERR_UNSUPPORTED
    assert call(o_part=None) == attn.ATTN_ERR_INVALID_ARG


def test_fwd_num_splits_rejects(lib):
    n = ctypes.c_int(0)
    lib.attn_fwd_num_splits.argtypes = [ctypes.c_int] * 6 + [ctypes.POINTER(ctypes.c_int)]
    assert lib.attn_fwd_num_splits(0, 4, 2, 64, 1000, 128, ctypes.byref(n)) == \
        attn.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_num_splits(1, 4, 3, 64, 1000, 128, ctypes.byref(n)) == \
        attn.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_num_splits(1, 4, 2, 64, 1000, 128, None) == attn.ATTN_ERR_INVALID_ARG
