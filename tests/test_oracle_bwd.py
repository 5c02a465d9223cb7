"""Pins for the fp64 oracle of the attention backward (CPU only).

The backward oracle is checked against central finite differences of the
fp64 forward (L = sum(dO * O)), against PyTorch fp64 autograd of
scaled-dot-product attention, and against closed forms: zero upstream gradient,
column sums of P (sum_j dV_j = sum_i dO_i), and dK = 0 when Q = 0.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from attn_inputs import make_qkv


def _dout(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def test_f64_forward_matches_bf16_forward():
    for causal in (False, True):
        q, k, v = make_qkv(2, 4, 2, 9, 13, 8, seed=3)
        o1, l1 = oracle.attn_fwd(q, k, v, causal, 0.3)
        o2, l2 = oracle.attn_fwd_f64(q, k, v, causal, 0.3)
        np.testing.assert_array_equal(o1, o2)
        np.testing.assert_array_equal(l1, l2)


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D,causal", [
    (1, 1, 1, 3, 4, 2, False),
    (1, 2, 1, 4, 4, 3, True),
    (1, 4, 2, 3, 5, 2, True),    # GQA, Sq < Sk
    (1, 2, 2, 5, 3, 2, True),    # Sq > Sk: leading rows fully masked
])
def test_finite_differences(B, Hq, Hkv, Sq, Sk, D, causal):
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Sk, D, seed=Sq * 10 + Sk)
    do = _dout(q.shape, seed=5).double().numpy()
    qd, kd, vd = (t.double().numpy() for t in (q, k, v))
    scale = 0.45
    dq, dk, dv = oracle.attn_bwd(qd, kd, vd, do, causal, scale)

    def loss(qx, kx, vx):
        o, _ = oracle.attn_fwd_f64(qx, kx, vx, causal, scale)
        return float(np.sum(o * do))

    eps = 1e-6
    for name, x, grad in (("q", qd, dq), ("k", kd, dk), ("v", vd, dv)):
        num = np.zeros_like(x)
        flat = x.reshape(-1)
        for idx in range(flat.size):
            old = flat[idx]
            flat[idx] = old + eps
            lp = loss(qd, kd, vd)
            flat[idx] = old - eps
            lm = loss(qd, kd, vd)
            flat[idx] = old
            num.reshape(-1)[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(grad, num, rtol=0, atol=2e-8, err_msg=f"d{name}")


def test_library_autograd_fp64():
    B, Hq, Hkv, Sq, Sk, D = 2, 6, 3, 11, 17, 8
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Sk, D, seed=21)
    do = _dout(q.shape, seed=22)
    scale = 1.0 / math.sqrt(D)
    grp = Hq // Hkv
    for causal in (False, True):
        dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal, scale)
        qq = q.double().requires_grad_(True)
        kk = k.double().requires_grad_(True)
        vv = v.double().requires_grad_(True)
        i = torch.arange(Sq)[:, None]
        j = torch.arange(Sk)[None, :]
        mask = (j <= i + Sk - Sq) if causal else torch.ones(Sq, Sk, dtype=torch.bool)
        o = torch.nn.functional.scaled_dot_product_attention(
            qq, kk.repeat_interleave(grp, dim=1), vv.repeat_interleave(grp, dim=1),
            attn_mask=mask, scale=scale)
        o.backward(do.double())
        np.testing.assert_allclose(dq, qq.grad.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dk, kk.grad.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dv, vv.grad.numpy(), rtol=0, atol=1e-12)


def test_zero_upstream_gradient():
    q, k, v = make_qkv(1, 4, 2, 10, 10, 8, seed=2)
    do = np.zeros(tuple(q.shape))
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, True, 0.3)
    assert not dq.any() and not dk.any() and not dv.any()


def test_dv_column_sums_and_zero_query():
    B, Hq, Hkv, Sq, Sk, D = 1, 4, 2, 12, 12, 8
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Sk, D, seed=4)
    do = _dout(q.shape, seed=6)
    grp = Hq // Hkv
    for causal in (False, True):
        _, _, dv = oracle.attn_bwd(q, k, v, do, causal, 0.3)
        # every row of P sums to one, so sum_j dV_j = sum over the group's rows of dO
        want = do.double().numpy().reshape(B, Hkv, grp, Sq, D).sum(axis=(2, 3))
        np.testing.assert_allclose(dv.sum(axis=2), want, rtol=0, atol=1e-12)
    qz = torch.zeros_like(q)
    _, dk, _ = oracle.attn_bwd(qz, k, v, do, True, 0.3)
    np.testing.assert_allclose(dk, 0.0, rtol=0, atol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Sq,Sk", [(13, 13), (9, 17), (17, 9)])
def test_sampled_matches_full(causal, Sq, Sk):
    """The sampled form on bf16 inputs gives the full oracle's values at its rows and keys."""
    B, Hq, Hkv, D = 2, 6, 2, 8
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Sk, D, seed=40 + Sq + Sk)
    do = _dout(q.shape, seed=41)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal, 0.35)
    qrows = np.array([0, 5, B * Hq * Sq - 1, Sq + 3, 3 * Sq])
    keys = np.array([0, Sk - 1, Sk + 2, 3 * Sk + 1, B * Hkv * Sk - 1, 1])
    sq, sk, sv = oracle.attn_bwd_sampled(q, k, v, do, causal, 0.35, qrows, keys)
    np.testing.assert_allclose(sq, dq.reshape(-1, D)[qrows], rtol=0, atol=1e-13)
    np.testing.assert_allclose(sk, dk.reshape(-1, D)[keys], rtol=0, atol=1e-13)
    np.testing.assert_allclose(sv, dv.reshape(-1, D)[keys], rtol=0, atol=1e-13)
