"""Seeded random shapes against the oracle: the forward (fp32 and bf16 output,
one pass and split-KV + combine), the decode (contiguous, per-sequence lengths,
paged) and the backward, each case drawn from a fixed seed so that a failure
reproduces.  The shapes cover what the fixed cases do not reach together:
odd lengths on both axes, Sq > Sk under the causal mask (rows that see no
key), GQA/MQA groupings of 1-8, D = 64/128/256, scales other than 1/sqrt(D)
and peakier inputs (std up to 2); and, on sampled rows, shapes large enough for
the launch-wide work-item orders and head pairing.  Tolerances are the parity
tolerances (for a bf16 O, plus its rounding to bf16)."""
import math

import numpy as np
import pytest
import torch

import oracle
import tensor_attn_fwd_gb300 as attn
from attn_inputs import make_qkv, sample_rows
from test_parity import assert_close
from test_paged import build_paged

pytestmark = pytest.mark.gpu


def fwd_case(i):
    r = np.random.default_rng(1000 + i)
    D = int(r.choice([64, 128, 256]))
    Hkv = int(r.integers(1, 5))
    group = int(r.choice([1, 2, 3, 4, 8]))
    B = int(r.integers(1, 4))
    Sk = int(r.integers(1, 800))
    Sq = int(r.integers(1, 600)) if r.random() < 0.8 else int(Sk + r.integers(1, 200))
    causal = bool(r.random() < 0.6)
    std = float(r.choice([1.0, math.sqrt(2.0), 2.0]))
    scale = float(r.uniform(0.5, 1.5)) / math.sqrt(D)
    out = "bf16" if r.random() < 0.25 else "fp32"
    splits = 1
    if D <= 128 and out == "fp32" and r.random() < 0.35:
        # at most one split per 128-key tile (the split-KV entry point's limit)
        splits = min(int(r.integers(2, 5)), -(-Sk // 128)) if r.random() < 0.7 else "auto"
    return dict(B=B, Hq=Hkv * group, Hkv=Hkv, Sq=Sq, Sk=Sk, D=D, causal=causal, std=std,
                scale=scale, out=out, splits=splits, seed=2000 + i)


@pytest.mark.parametrize("i", range(120))
def test_fwd_random(i):
    c = fwd_case(i)
    q, k, v = make_qkv(c["B"], c["Hq"], c["Hkv"], c["Sq"], c["Sk"], c["D"], c["seed"],
                       q_std=c["std"], k_std=c["std"])
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    if c["out"] == "bf16":
        o, lse = attn.attn_fwd_bf16o(qd, kd, vd, causal=c["causal"], scale=c["scale"])
    else:
        o, lse = attn.attn_fwd(qd, kd, vd, causal=c["causal"], scale=c["scale"],
                               num_splits=c["splits"])
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, c["causal"], c["scale"])
    assert_close(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, str(c),
                 o_bf16=c["out"] == "bf16")


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D,causal,out,splits", [
    (4, 32, 8, 4096, 4096, 256, True, "fp32", 1),     # D = 256, chunked KV-head order
    (2, 16, 16, 4096, 4096, 256, False, "fp32", 1),   # D = 256, KV-head order
    (8, 16, 16, 2048, 2048, 128, False, "fp32", 1),   # D = 128, KV-head order
    (8, 16, 16, 2048, 2048, 64, False, "bf16", 1),    # D = 64, KV-head order, bf16 O
    (2, 32, 8, 100, 8192, 128, True, "fp32", 1),      # head pairs: a chunk against a cache
    (2, 32, 8, 100, 8192, 128, True, "fp32", 8),      # head pairs with split-KV
    (1, 64, 8, 128, 16384, 64, True, "fp32", "auto"),
    (3, 24, 8, 3000, 5000, 128, True, "fp32", 1),     # Sq != Sk, groups of 3
    (2, 8, 1, 6000, 6000, 256, True, "bf16", 1),      # MQA at D = 256
])
def test_fwd_large_sampled(B, Hq, Hkv, Sq, Sk, D, causal, out, splits):
    # Sizes at which the launch-wide work-item orders and head pairing take
    # effect; 400 random rows plus every head's edge rows against the oracle.
    seed = B * 7 + Sq + Sk + D
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Sk, D, seed)
    scale = 1.0 / math.sqrt(D)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    if out == "bf16":
        o, lse = attn.attn_fwd_bf16o(qd, kd, vd, causal=causal, scale=scale)
    else:
        o, lse = attn.attn_fwd(qd, kd, vd, causal=causal, scale=scale, num_splits=splits)
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    rows = sample_rows(B, Hq, Sq, 400, seed)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, scale, rows=rows.numpy())
    assert_close(o.float().reshape(-1, D)[rows].cpu().numpy(), lse.reshape(-1)[rows].cpu().numpy(),
                 o_ref, lse_ref, f"B{B} Hq{Hq} Hkv{Hkv} Sq{Sq} Sk{Sk} D{D} c{causal} {out}",
                 o_bf16=out == "bf16")


@pytest.mark.parametrize("i", range(48))
def test_decode_random(i):
    r = np.random.default_rng(3000 + i)
    D = int(r.choice([64, 128, 256]))
    Hkv = int(r.integers(1, 9))
    group = int(r.choice([1, 2, 4, 8]))
    Hq = Hkv * group
    B = int(r.integers(1, 7))
    cap = int(r.integers(1, 3000))
    ns = int(r.integers(1, min(cap, 20) + 1))
    kind = ["contiguous", "varlen", "paged"][i % 3]
    scale = float(r.uniform(0.5, 1.5)) / math.sqrt(D)
    q, k, v = make_qkv(B, Hq, Hkv, 1, cap, D, seed=4000 + i)
    qd = q.cuda()
    if kind == "contiguous":
        o, lse = attn.decode(qd, k.cuda(), v.cuda(), ns, scale)
        lens = [cap] * B
    else:
        lens_t = torch.from_numpy(r.integers(0, cap + 1, B).astype(np.int32))
        if B > 1:
            lens_t[0] = cap
        if kind == "varlen":
            o, lse = attn.decode(qd, k.cuda(), v.cuda(), ns, scale, seqlens=lens_t.cuda())
        else:
            page = int(r.choice([32, 64, 128]))
            kc, vc, table = build_paged(k, v, lens_t, page, spare_pages=2, seed=5000 + i)
            o, lse = attn.decode_paged(qd, kc.cuda(), vc.cuda(), table.cuda(), lens_t.cuda(), ns,
                                       scale)
        lens = [int(x) for x in lens_t]
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    o = o.cpu().numpy()
    lse = lse.cpu().numpy()
    for b in range(B):
        n = lens[b]
        if n == 0:
            assert np.all(o[b] == 0) and np.all(lse[b] == -np.inf), f"{kind} b{b}: empty sequence"
            continue
        o_ref, lse_ref = oracle.attn_fwd(q[b:b + 1], k[b:b + 1, :, :n], v[b:b + 1, :, :n], False,
                                         scale)
        assert_close(o[b:b + 1], lse[b:b + 1], o_ref[:, :, 0], lse_ref[:, :, 0],
                     f"{kind} B{B} Hq{Hq} Hkv{Hkv} cap{cap} D{D} ns{ns} b{b} n{n}")


@pytest.mark.parametrize("i", range(24))
def test_bwd_random(i):
    r = np.random.default_rng(6000 + i)
    D = int(r.choice([64, 128]))
    Hkv = int(r.integers(1, 4))
    Hq = Hkv * int(r.choice([1, 2, 4]))
    B = int(r.integers(1, 3))
    Sq = int(r.integers(1, 420))
    Sk = int(r.integers(1, 420))
    causal = bool(r.random() < 0.6)
    scale = float(r.uniform(0.5, 1.5)) / math.sqrt(D)
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Sk, D, seed=7000 + i)
    do = torch.randn((B, Hq, Sq, D), generator=torch.Generator().manual_seed(8000 + i)).to(
        torch.bfloat16)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = attn.attn_fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = attn.attn_bwd(qd, kd, vd, o, lse, do.cuda(), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    refs = oracle.attn_bwd(q, k, v, do, causal, scale)
    what = f"B{B} Hq{Hq} Hkv{Hkv} Sq{Sq} Sk{Sk} D{D} c{causal}"
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        got = got.cpu().double().numpy()
        assert np.all(np.isfinite(got)), f"{what} {name}: non-finite"
        err = float(np.max(np.abs(got - ref))) / max(float(np.max(np.abs(ref))), 1.0)
        assert err <= 2e-2, f"{what} {name}: relative max error {err:.3e}"
