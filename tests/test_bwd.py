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
