"""GPU parity of the split-KV decode over a paged KV cache.

Each sequence's keys are scattered over shuffled pages of a shared cache whose
unused pages, and unused rows of partly filled pages, hold NaN.  The oracle
gathers each sequence through the same block table (pure indexing) and runs
the plain definition on it: per-split partials with the paged split rule
(whole 32-key blocks) and the full attention after the combine.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import tensor_attn_fwd_gb300 as attn
from attn_inputs import make_qkv
from test_parity import assert_close

pytestmark = pytest.mark.gpu


def build_paged(k, v, lens, page, spare_pages, seed):
    """Scatter contiguous k/v [B,Hkv,Sk,D] into a shuffled paged cache."""
    B, Hkv, Sk, D = k.shape
    max_pages = -(-Sk // page)
    used = [-(-int(n) // page) for n in lens]
    num_pages = sum(used) + spare_pages
    perm = torch.randperm(num_pages, generator=torch.Generator().manual_seed(seed))
    kc = torch.full((num_pages, Hkv, page, D), float("nan")).to(torch.bfloat16)
    vc = kc.clone()
    table = torch.full((B, max_pages), 0, dtype=torch.int32)
    nxt = 0
    for b in range(B):
        for p in range(used[b]):
            pid = int(perm[nxt])
            nxt += 1
            lo, hi = p * page, min((p + 1) * page, int(lens[b]))
            kc[pid, :, :hi - lo] = k[b, :, lo:hi]
            vc[pid, :, :hi - lo] = v[b, :, lo:hi]
            table[b, p] = pid
    return kc, vc, table


@pytest.mark.parametrize("B,Hq,Hkv,cap,D,page,ns", [
    (4, 8, 2, 256, 128, 32, 1),
    (6, 32, 8, 1024, 128, 64, 8),
    (5, 4, 4, 300, 64, 32, 3),
    (3, 16, 1, 2048, 128, 256, 5),
    (4, 32, 8, 4096, 64, 128, 16),
    (3, 8, 2, 1000, 256, 64, 4),   # D = 256
])
def test_decode_paged(B, Hq, Hkv, cap, D, page, ns):
    q, k, v = make_qkv(B, Hq, Hkv, 1, cap, D, seed=B * 11 + cap + page)
    g = torch.Generator().manual_seed(cap + page)
    lens = torch.randint(0, cap + 1, (B,), generator=g, dtype=torch.int32)
    lens[0] = 0            # empty sequence
    lens[1] = cap          # full capacity
    lens[2] = 33 if cap > 33 else 1
    kc, vc, table = build_paged(k, v, lens, page, spare_pages=3, seed=page)
    scale = 1.0 / math.sqrt(D)
    op, lp = attn.attn_decode_splitkv_paged(q.cuda(), kc.cuda(), vc.cuda(), table.cuda(),
                                            lens.cuda(), ns, scale)
    o, lse = attn.attn_combine(op, lp)
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    op, lp, o, lse = (t.cpu().numpy() for t in (op, lp, o, lse))
    for b in range(B):
        n = int(lens[b])
        qb = q[b:b + 1].contiguous()
        kb = oracle.gather_paged(kc, table, lens, b)
        vb = oracle.gather_paged(vc, table, lens, b)
        op_ref, lp_ref = oracle.decode_split(qb, kb, vb, ns, scale, align=32)
        assert_close(op[:, b:b + 1], lp[:, b:b + 1], op_ref, lp_ref, f"partials b={b} len={n}")
        o_ref, lse_ref = oracle.attn_fwd(qb, kb, vb, False, scale)
        assert_close(o[b:b + 1], lse[b:b + 1], o_ref[:, :, 0], lse_ref[:, :, 0], f"b={b} len={n}")


def test_decode_paged_matches_contiguous_varlen():
    """The same keys through a page table or a contiguous cache: the combined
    results agree (the split rules differ, so to rounding only)."""
    B, Hq, Hkv, cap, D, page = 8, 32, 8, 2048, 128, 64
    q, k, v = make_qkv(B, Hq, Hkv, 1, cap, D, seed=77)
    lens = torch.randint(1, cap + 1, (B,), generator=torch.Generator().manual_seed(78),
                         dtype=torch.int32)
    kc, vc, table = build_paged(k, v, lens, page, spare_pages=0, seed=79)
    qd = q.cuda()
    o1, l1 = attn.decode_paged(qd, kc.cuda(), vc.cuda(), table.cuda(), lens.cuda(), 8)
    o2, l2 = attn.decode(qd, k.cuda(), v.cuda(), 8, seqlens=lens.cuda())
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    assert float((o1 - o2).abs().max()) <= 2.0 ** -9 * float(v.float().abs().max())
    assert float((l1 - l2).abs().max()) <= 1e-4


def test_decode_paged_bad_table_entry_reported():
    """A table entry outside [0, num_pages) that a sequence reaches is reported
    in the status word; the kernel reads page 0 in its place and finishes."""
    B, Hq, Hkv, cap, D, page = 2, 8, 2, 128, 64, 32
    q, k, v = make_qkv(B, Hq, Hkv, 1, cap, D, seed=5)
    lens = torch.tensor([cap, 40], dtype=torch.int32)
    kc, vc, table = build_paged(k, v, lens, page, spare_pages=0, seed=6)
    table[1, 1] = kc.shape[0]       # reached: sequence 1 has 40 keys (pages 0 and 1)
    table[1, 3] = -5                # not reached
    o, lse = attn.decode_paged(q.cuda(), kc.cuda(), vc.cuda(), table.cuda(), lens.cuda(), 2)
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_debug_status() == attn.ATTN_OK   # read-and-clear
    # sequence 0 never touches the bad entries
    kb = oracle.gather_paged(kc, table, lens, 0)
    vb = oracle.gather_paged(vc, table, lens, 0)
    o_ref, lse_ref = oracle.attn_fwd(q[0:1].contiguous(), kb, vb, False, 1.0 / math.sqrt(D))
    assert_close(o[0:1].cpu().numpy(), lse[0:1].cpu().numpy(), o_ref[:, :, 0], lse_ref[:, :, 0])
