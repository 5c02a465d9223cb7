"""GPU parity of the attention backward against the fp64 oracle.

Tolerance: P and dS are rounded to bf16 before the tensor-core products
(as P is in the forward), with fp32 accumulation.  Each gradient is compared
in the max norm: max|g_gpu - g_ref| <= 2e-2 * max(1, max|g_ref|) -- relative
to the gradient's scale, absolute where the exact gradient vanishes (e.g. a
single visible key makes dS, hence dQ and dK, exactly zero).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import tensor_attn_fwd_gb300 as attn
from attn_inputs import make_qkv

pytestmark = pytest.mark.gpu

REL_TOL = 2e-2


def run_bwd_case(B, Hq, Hkv, Sq, Sk, D, causal, seed):
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Sk, D, seed)
    g = torch.Generator().manual_seed(seed + 1)
    do = torch.randn((B, Hq, Sq, D), generator=g).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(D)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = attn.attn_fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = attn.attn_bwd(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    dq_ref, dk_ref, dv_ref = oracle.attn_bwd(q, k, v, do, causal, scale)
    for name, got, ref in (("dq", dq, dq_ref), ("dk", dk, dk_ref), ("dv", dv, dv_ref)):
        got = got.cpu().double().numpy()
        assert np.all(np.isfinite(got)), name
        denom = max(float(np.max(np.abs(ref))), 1.0)
        err = float(np.max(np.abs(got - ref))) / denom
        assert err <= REL_TOL, f"{name}: relative max error {err:.3e}"


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_small(D, causal):
    run_bwd_case(1, 2, 1, 256, 256, D, causal, seed=D + causal)


@pytest.mark.parametrize("Sq,Sk", [(1, 1), (7, 7), (130, 300), (300, 130), (129, 129)])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_ragged(Sq, Sk, causal):
    run_bwd_case(2, 4, 2, Sq, Sk, 128, causal, seed=Sq * 3 + Sk)


@pytest.mark.parametrize("Hq,Hkv", [(8, 1), (8, 8), (8, 2)])
def test_bwd_heads(Hq, Hkv):
    run_bwd_case(1, Hq, Hkv, 384, 384, 64, True, seed=Hq + Hkv)


def test_bwd_longer():
    run_bwd_case(1, 4, 1, 1024, 1024, 128, True, seed=99)


def test_bwd_full_size_sampled():
    """Causal GQA B2 Hq32 Hkv8 S8192 D128 (the prefill workload), as the benchmark
    runs it; dQ on sampled query rows, dK/dV on sampled keys of two KV heads."""
    from attn_inputs import WORKLOADS, sample_rows, workload_inputs
    w = WORKLOADS[3]
    q, k, v = workload_inputs(w)
    g = torch.Generator().manual_seed(w.seed + 7)
    do = torch.randn(q.shape, generator=g).to(torch.bfloat16)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = attn.attn_fwd(qd, kd, vd, causal=w.causal, scale=w.scale)
    dq, dk, dv = attn.attn_bwd(qd, kd, vd, o, lse, dod, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    del qd, kd, vd, dod, o, lse
    rows = sample_rows(w.B, w.Hq, w.Sq, n_random=48, seed=w.seed)
    pick = torch.randperm(rows.numel(), generator=torch.Generator().manual_seed(5))[:96]
    rows = rows[pick].sort().values
    S = w.Sk
    keys = []
    for bg in (0 * w.Hkv + 3, 1 * w.Hkv + 6):
        keys += [bg * S + j for j in (0, 1, 127, 128, 4095, 4096, S - 129, S - 1)]
    keys = torch.tensor(keys + [bg * S + int(j) for j in
                                torch.randint(0, S, (8,), generator=torch.Generator().manual_seed(6))])
    dq_ref, dk_ref, dv_ref = oracle.attn_bwd_sampled(q, k, v, do, w.causal, w.scale,
                                                     rows.numpy(), keys.numpy())
    got = {"dq": dq.reshape(-1, w.D)[rows.cuda()], "dk": dk.reshape(-1, w.D)[keys.cuda()],
           "dv": dv.reshape(-1, w.D)[keys.cuda()]}
    for name, ref in (("dq", dq_ref), ("dk", dk_ref), ("dv", dv_ref)):
        g_np = got[name].cpu().double().numpy()
        assert np.all(np.isfinite(g_np)), name
        err = float(np.max(np.abs(g_np - ref))) / max(float(np.max(np.abs(ref))), 1.0)
        assert err <= REL_TOL, f"{name}: relative max error {err:.3e}"
