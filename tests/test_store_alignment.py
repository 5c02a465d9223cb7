"""Outputs in buffers that are 16- but not 32-byte aligned.

The C-ABI asks for 16-byte aligned pointers.  The kernels write whole 32-byte
segments of an output row when the buffer allows it and two 16-byte stores
otherwise; both paths must write the same bytes to the same places.  Each case
runs once into freshly allocated (aligned) tensors and once into views that
start 16 bytes into a NaN-filled buffer, then checks that the results are
bit-identical and that no element outside the view was written.
"""
import math

import pytest
import torch

import tensor_attn_fwd_gb300 as attn
from attn_inputs import make_qkv

pytestmark = pytest.mark.gpu


def offset_view(shape, dtype):
    """A contiguous view of `shape` whose first element is 16 bytes past a
    32-byte boundary, inside a NaN-filled buffer with guard elements on both
    sides.  Returns (view, buffer, offset, numel)."""
    numel = math.prod(shape)
    off = 16 // torch.tensor([], dtype=dtype).element_size()
    buf = torch.full((off + numel + 16,), float("nan"), dtype=dtype, device="cuda")
    view = buf[off:off + numel].view(shape)
    assert view.data_ptr() % 32 == 16
    return view, buf, off, numel


def assert_guards_untouched(buf, off, numel):
    assert torch.isnan(buf[:off].float()).all()
    assert torch.isnan(buf[off + numel:].float()).all()


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("bf16_out", [False, True])
@pytest.mark.parametrize("Sq,causal", [(301, True), (129, False)])
def test_fwd_output_16_byte_aligned(D, bf16_out, Sq, causal):
    B, Hq, Hkv = 2, 4, 2
    q, k, v = (t.cuda() for t in make_qkv(B, Hq, Hkv, Sq, Sq, D, seed=7 * Sq + D))
    fwd = attn.attn_fwd_bf16o if bf16_out else attn.attn_fwd
    o_ref, lse_ref = fwd(q, k, v, causal=causal)
    dtype = torch.bfloat16 if bf16_out else torch.float32
    o, buf, off, numel = offset_view((B, Hq, Sq, D), dtype)
    o_got, lse_got = fwd(q, k, v, causal=causal, o=o)
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    assert o_got.data_ptr() == o.data_ptr()
    assert torch.equal(o, o_ref)
    assert torch.equal(lse_got, lse_ref)
    assert_guards_untouched(buf, off, numel)


@pytest.mark.parametrize("D", [64, 128])
def test_fwd_splitkv_partials_16_byte_aligned(D):
    B, Hq, Hkv, Sq, Sk, ns = 1, 4, 2, 77, 1000, 3
    q, k, v = (t.cuda() for t in make_qkv(B, Hq, Hkv, Sq, Sk, D, seed=D + 5))
    op_ref, lp_ref = attn.attn_fwd_splitkv(q, k, v, ns, causal=True)
    op, buf, off, numel = offset_view((ns, B, Hq, Sq, D), torch.float32)
    attn.attn_fwd_splitkv(q, k, v, ns, causal=True, o_part=op)
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    assert torch.equal(op, op_ref)
    assert_guards_untouched(buf, off, numel)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("S,causal", [(301, True), (200, False)])
def test_bwd_gradients_16_byte_aligned(D, S, causal):
    B, Hq, Hkv = 1, 4, 2
    q, k, v = (t.cuda() for t in make_qkv(B, Hq, Hkv, S, S, D, seed=S + D))
    g = torch.Generator().manual_seed(S)
    do = torch.randn((B, Hq, S, D), generator=g).to(torch.bfloat16).cuda()
    o, lse = attn.attn_fwd(q, k, v, causal=causal)
    ref = attn.attn_bwd(q, k, v, o, lse, do, causal=causal)
    dq, bq, oq, nq = offset_view((B, Hq, S, D), torch.float32)
    dk, bk, ok_, nk = offset_view((B, Hkv, S, D), torch.float32)
    dv, bv, ov, nv = offset_view((B, Hkv, S, D), torch.float32)
    attn.attn_bwd(q, k, v, o, lse, do, causal=causal, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    for got, want in zip((dq, dk, dv), ref):
        assert torch.equal(got, want)
    for b, o_, n in ((bq, oq, nq), (bk, ok_, nk), (bv, ov, nv)):
        assert_guards_untouched(b, o_, n)
