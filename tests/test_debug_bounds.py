"""The debug build (-DATTN_DEBUG_BOUNDS): every prefill, decode and backward output store is checked
against its buffer, and a store outside it would be skipped and reported as
ATTN_ERR_BOUNDS.  On ragged shapes, every head dimension, both output types and
an output that is only 16-byte aligned, the debug library reports ATTN_OK and
writes exactly what the release library writes."""
import ctypes
import math

import pytest
import torch

import tensor_attn_fwd_gb300 as attn
from tensor_attn_fwd_gb300 import build as attn_build
from attn_inputs import make_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dbg():
    lib = ctypes.CDLL(attn_build.build(debug=True))
    for fn in (lib.attn_fwd, lib.attn_fwd_bf16o):
        fn.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 7 + [ctypes.c_float, ctypes.c_void_p]
        fn.restype = ctypes.c_int
    lib.attn_decode_splitkv.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 6 + [ctypes.c_float, ctypes.c_void_p]
    lib.attn_decode_splitkv.restype = ctypes.c_int
    lib.attn_bwd.argtypes = [ctypes.c_void_p] * 10 + [ctypes.c_int] * 7 + [ctypes.c_float, ctypes.c_void_p]
    lib.attn_bwd.restype = ctypes.c_int
    lib.attn_debug_status.argtypes = [ctypes.c_void_p]
    lib.attn_debug_status.restype = ctypes.c_int
    return lib


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D,causal,bf16o,offset", [
    (2, 4, 2, 301, 301, 64, True, False, False),
    (1, 4, 1, 129, 777, 128, True, True, False),
    (2, 8, 2, 300, 129, 128, False, False, True),
    (1, 2, 2, 7, 7, 128, True, False, False),
    (1, 4, 2, 333, 333, 256, True, False, False),
    (1, 2, 1, 200, 640, 256, False, True, True),
])
def test_debug_build_matches_release(dbg, B, Hq, Hkv, Sq, Sk, D, causal, bf16o, offset):
    q, k, v = (t.cuda() for t in make_qkv(B, Hq, Hkv, Sq, Sk, D, seed=Sq + 3 * Sk + D))
    fwd = attn.attn_fwd_bf16o if bf16o else attn.attn_fwd
    o_ref, lse_ref = fwd(q, k, v, causal=causal)
    dtype = torch.bfloat16 if bf16o else torch.float32
    off = (16 // torch.tensor([], dtype=dtype).element_size()) if offset else 0
    numel = B * Hq * Sq * D
    buf = torch.full((numel + off,), 3.0, dtype=dtype, device="cuda")
    o = buf[off:].view(B, Hq, Sq, D)
    lse = torch.full((B, Hq, Sq), 3.0, device="cuda")
    fn = dbg.attn_fwd_bf16o if bf16o else dbg.attn_fwd
    st = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, Hq, Hkv,
            Sq, Sk, D, int(causal), 1.0 / math.sqrt(D), torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK
    assert dbg.attn_debug_status(None) == attn.ATTN_OK
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


@pytest.mark.parametrize("B,Hq,Hkv,Sk,D,ns", [(3, 8, 2, 1000, 128, 5), (2, 32, 8, 777, 64, 3),
                                              (2, 16, 4, 2048, 256, 4)])
def test_debug_build_decode_matches_release(dbg, B, Hq, Hkv, Sk, D, ns):
    q, k, v = (t.cuda() for t in make_qkv(B, Hq, Hkv, 1, Sk, D, seed=Sk + D + ns))
    op_ref, lp_ref = attn.attn_decode_splitkv(q, k, v, ns)
    op = torch.full_like(op_ref, 3.0)
    lp = torch.full_like(lp_ref, 3.0)
    st = dbg.attn_decode_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), op.data_ptr(),
                                 lp.data_ptr(), B, Hq, Hkv, Sk, D, ns, 1.0 / math.sqrt(D),
                                 torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK
    assert dbg.attn_debug_status(None) == attn.ATTN_OK
    assert torch.equal(op, op_ref) and torch.equal(lp, lp_ref)


@pytest.mark.parametrize("B,Hq,Hkv,S,D,causal", [(1, 4, 2, 301, 64, True), (2, 4, 1, 200, 128, False)])
def test_debug_build_backward_matches_release(dbg, B, Hq, Hkv, S, D, causal):
    q, k, v = (t.cuda() for t in make_qkv(B, Hq, Hkv, S, S, D, seed=S + D))
    g = torch.Generator().manual_seed(S)
    do = torch.randn((B, Hq, S, D), generator=g).to(torch.bfloat16).cuda()
    o, lse = attn.attn_fwd(q, k, v, causal=causal)
    ref = attn.attn_bwd(q, k, v, o, lse, do, causal=causal)
    dq, dk, dv = (torch.full_like(t, 3.0) for t in ref)
    ws = torch.empty((B, Hq, S), device="cuda")
    st = dbg.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                      do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), ws.data_ptr(),
                      B, Hq, Hkv, S, S, D, int(causal), 1.0 / math.sqrt(D),
                      torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK
    assert dbg.attn_debug_status(None) == attn.ATTN_OK
    for got, want in zip((dq, dk, dv), ref):
        assert torch.equal(got, want)


@pytest.mark.parametrize("i", range(0, 120, 4))
def test_debug_build_random_forward_shapes(dbg, i):
    # Every fourth shape of the random sweep (odd lengths, Sq > Sk causal, all
    # head dimensions and groupings), one pass, fp32 or bf16 output.
    from test_fuzz import fwd_case
    c = fwd_case(i)
    q, k, v = (t.cuda() for t in make_qkv(c["B"], c["Hq"], c["Hkv"], c["Sq"], c["Sk"], c["D"],
                                          c["seed"], q_std=c["std"], k_std=c["std"]))
    bf16o = c["out"] == "bf16"
    fwd = attn.attn_fwd_bf16o if bf16o else attn.attn_fwd
    o_ref, lse_ref = fwd(q, k, v, causal=c["causal"], scale=c["scale"])
    o = torch.full_like(o_ref, 3.0)
    lse = torch.full_like(lse_ref, 3.0)
    fn = dbg.attn_fwd_bf16o if bf16o else dbg.attn_fwd
    st = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), c["B"],
            c["Hq"], c["Hkv"], c["Sq"], c["Sk"], c["D"], int(c["causal"]), c["scale"],
            torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK
    assert dbg.attn_debug_status(None) == attn.ATTN_OK, c
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref), c
