"""The decode with its LSE combine fused into the split kernel (attn_decode_fused):
its O and LSE against the oracle, its partials and its combined O and LSE bit
for bit against the two-launch decode's (the same code writes the partials and
the merge follows the combine kernel's order), its counters back at
zero after every call, repeated calls on one counter array, per-sequence
lengths with empty sequences, query groups wider than one 16-head slice,
split counts past one warp's 32, and a CUDA graph replayed on new inputs."""
import math

import numpy as np
import pytest
import torch

import oracle
import tensor_attn_fwd_gb300 as attn
from attn_inputs import make_qkv
from test_paged import build_paged
from test_parity import assert_close

pytestmark = pytest.mark.gpu


def check_against_oracle(q, k, v, o, lse, scale, lens=None, what=""):
    o = o.cpu().numpy()
    lse = lse.cpu().numpy()
    B = q.shape[0]
    for b in range(B):
        n = k.shape[2] if lens is None else lens[b]
        if n == 0:
            assert np.all(o[b] == 0) and np.all(lse[b] == -np.inf), f"{what} b{b}: empty sequence"
            continue
        o_ref, lse_ref = oracle.attn_fwd(q[b:b + 1], k[b:b + 1, :, :n], v[b:b + 1, :, :n], False,
                                         scale)
        assert_close(o[b:b + 1], lse[b:b + 1], o_ref[:, :, 0], lse_ref[:, :, 0], f"{what} b{b}")


@pytest.mark.parametrize("B,Hq,Hkv,Sk,D,ns", [
    (4, 32, 8, 1000, 128, 8),     # GQA, ragged tail
    (2, 8, 1, 777, 64, 3),        # MQA
    (3, 16, 4, 600, 256, 5),      # D = 256
    (1, 64, 2, 2048, 128, 16),    # a group of 32 query heads: two head slices
    (2, 8, 8, 4000, 64, 40),      # more splits than one warp of the combine
    (1, 4, 1, 50, 128, 50),       # one key per split
    (5, 32, 8, 300, 128, 1),      # one split: the combine is a copy
])
def test_fused_against_oracle_and_split_path(B, Hq, Hkv, Sk, D, ns):
    scale = 1.0 / math.sqrt(D)
    q, k, v = make_qkv(B, Hq, Hkv, 1, Sk, D, seed=B * 1000 + Sk + ns)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = attn.attn_decode_fused(qd, kd, vd, ns, scale)
    op2, lp2 = attn.attn_decode_splitkv(qd, kd, vd, ns, scale)
    o_part = torch.empty_like(op2)
    lse_part = torch.empty_like(lp2)
    o3, lse3 = attn.attn_decode_fused(qd, kd, vd, ns, scale, o_part=o_part, lse_part=lse_part)
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    check_against_oracle(q, k, v, o, lse, scale, what=f"B{B} Hq{Hq} Hkv{Hkv} Sk{Sk} D{D} ns{ns}")
    # The partials come from the same code path as attn_decode_splitkv's.
    assert torch.equal(o_part, op2) and torch.equal(lse_part, lp2)
    # A second call on the (self-resetting) counters gives the same result.
    assert torch.equal(o3, o) and torch.equal(lse3, lse)
    # The fused merge is the combine kernel's arithmetic in the same order.
    o2, lse2 = attn.attn_combine(op2, lp2)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


def test_fused_varlen_with_empty_sequences():
    B, Hq, Hkv, cap, D, ns = 6, 16, 2, 900, 128, 6
    scale = 0.1
    q, k, v = make_qkv(B, Hq, Hkv, 1, cap, D, seed=77)
    lens = [900, 0, 1, 450, 17, 0]
    seqlens = torch.tensor(lens, dtype=torch.int32, device="cuda")
    o, lse = attn.decode(q.cuda(), k.cuda(), v.cuda(), ns, scale, seqlens=seqlens)
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    check_against_oracle(q, k, v, o, lse, scale, lens=lens, what="varlen")


def test_fused_counters_return_to_zero():
    B, Hq, Hkv, Sk, D, ns = 3, 32, 4, 512, 128, 4
    q, k, v = (t.cuda() for t in make_qkv(B, Hq, Hkv, 1, Sk, D, seed=5))
    n = B * Hkv * ((Hq // Hkv + 15) // 16)
    counters = torch.zeros(n + 8, dtype=torch.int32, device="cuda")
    for _ in range(3):
        attn.attn_decode_fused(q, k, v, ns, counters=counters)
        torch.cuda.synchronize()
        assert attn.attn_debug_status() == attn.ATTN_OK
        assert int(counters.abs().sum()) == 0
    # Too small an array is rejected by the binding.
    with pytest.raises(ValueError):
        attn.attn_decode_fused(q, k, v, ns, counters=counters[: n - 1])


def test_fused_default_split_rule():
    # decode() with no split count takes attn_decode_num_splits and runs fused.
    B, Hq, Hkv, Sk, D = 1, 32, 8, 4096, 128
    q, k, v = make_qkv(B, Hq, Hkv, 1, Sk, D, seed=11)
    o, lse = attn.decode(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    check_against_oracle(q, k, v, o, lse, 1.0 / math.sqrt(D), what="rule")


def test_fused_graph_replay():
    B, Hq, Hkv, Sk, D, ns = 4, 16, 4, 1024, 64, 8
    scale = 1.0 / math.sqrt(D)
    qd = torch.empty((B, Hq, 1, D), dtype=torch.bfloat16, device="cuda")
    kd = torch.empty((B, Hkv, Sk, D), dtype=torch.bfloat16, device="cuda")
    vd = torch.empty_like(kd)
    o = torch.empty((B, Hq, D), device="cuda")
    lse = torch.empty((B, Hq), device="cuda")
    op = torch.empty((ns, B, Hq, D), device="cuda")
    lp = torch.empty((ns, B, Hq), device="cuda")
    counters = torch.zeros(B * Hkv, dtype=torch.int32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        attn.attn_decode_fused(qd.zero_(), kd.zero_(), vd.zero_(), ns, scale, o_part=op,
                               lse_part=lp, o=o, lse=lse, counters=counters)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        attn.attn_decode_fused(qd, kd, vd, ns, scale, o_part=op, lse_part=lp, o=o, lse=lse,
                               counters=counters, stream=side)
    for rep in range(3):
        q, k, v = make_qkv(B, Hq, Hkv, 1, Sk, D, seed=300 + rep)
        qd.copy_(q)
        kd.copy_(k)
        vd.copy_(v)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert attn.attn_debug_status() == attn.ATTN_OK
        assert int(counters.abs().sum()) == 0
        check_against_oracle(q, k, v, o, lse, scale, what=f"replay {rep}")


@pytest.mark.parametrize("B,Hq,Hkv,cap,D,page,ns", [
    (6, 32, 8, 1024, 128, 64, 8),
    (5, 4, 4, 300, 64, 32, 3),
    (3, 16, 2, 700, 256, 128, 5),
])
def test_fused_paged_equals_two_launches(B, Hq, Hkv, cap, D, page, ns):
    scale = 1.0 / math.sqrt(D)
    q, k, v = make_qkv(B, Hq, Hkv, 1, cap, D, seed=B + cap + page)
    lens_t = torch.tensor([cap] + [int(x) for x in torch.randint(
        0, cap + 1, (B - 1,), generator=torch.Generator().manual_seed(cap))], dtype=torch.int32)
    kc, vc, table = build_paged(k, v, lens_t, page, spare_pages=2, seed=cap + 1)
    qd, kcd, vcd, td, ld = q.cuda(), kc.cuda(), vc.cuda(), table.cuda(), lens_t.cuda()
    o, lse = attn.decode_paged(qd, kcd, vcd, td, ld, ns, scale)
    op, lp = attn.attn_decode_splitkv_paged(qd, kcd, vcd, td, ld, ns, scale)
    o2, lse2 = attn.attn_combine(op, lp)
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    check_against_oracle(q, k, v, o, lse, scale, lens=[int(x) for x in lens_t],
                         what=f"paged B{B} page{page} ns{ns}")
