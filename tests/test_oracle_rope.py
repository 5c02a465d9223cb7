"""Pins for the fp64 QKV-projection + RoPE oracle (CPU only).

Checked against: a library matmul (at position 0 RoPE is the identity), the
closed form of a single rotated pair, norm preservation per pair, RoPE's
relative-position property (q(m).k(n) depends on m - n only), and the
equivalence of the two pair conventions under a permutation of the weights.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _bf16(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(torch.bfloat16)


def _proj_ref(x, w):
    return x.double().numpy() @ w.double().numpy().T


@pytest.mark.parametrize("style", [0, 1])
def test_position_zero_is_plain_projection(style):
    T, hidden, Hq, Hkv, D = 9, 40, 4, 2, 16
    x = _bf16((T, hidden), 1)
    w = _bf16(((Hq + 2 * Hkv) * D, hidden), 2, std=0.2)
    q, k, v = oracle.qkv_rope(x, w, np.zeros(T, np.int32), Hq, Hkv, D, style=style)
    y = _proj_ref(x, w)
    np.testing.assert_allclose(q.reshape(T, -1), y[:, :Hq * D], rtol=0, atol=1e-12)
    np.testing.assert_allclose(k.reshape(T, -1), y[:, Hq * D:(Hq + Hkv) * D], rtol=0, atol=1e-12)
    np.testing.assert_allclose(v.reshape(T, -1), y[:, (Hq + Hkv) * D:], rtol=0, atol=1e-12)


@pytest.mark.parametrize("style", [0, 1])
def test_single_pair_closed_form(style):
    # hidden = D = 2, identity projections: x = (1, 0) rotates to (cos p, sin p).
    eye = torch.eye(2)
    w = torch.cat([eye, eye, eye]).to(torch.bfloat16)          # Q, K, V heads
    pos = np.array([0, 1, 5, 1000, 8191], dtype=np.int32)
    x = torch.tensor([[1.0, 0.0]] * pos.size).to(torch.bfloat16)
    q, k, v = oracle.qkv_rope(x, w, pos, 1, 1, 2, base=10000.0, style=style)
    want = np.stack([np.cos(pos.astype(np.float64)), np.sin(pos.astype(np.float64))], axis=1)
    np.testing.assert_allclose(q[:, 0], want, rtol=0, atol=1e-12)
    np.testing.assert_allclose(k[:, 0], want, rtol=0, atol=1e-12)
    np.testing.assert_allclose(v[:, 0], np.tile([1.0, 0.0], (pos.size, 1)), rtol=0, atol=0)


@pytest.mark.parametrize("style", [0, 1])
def test_rotation_preserves_pair_norms(style):
    T, hidden, Hq, Hkv, D = 6, 32, 2, 1, 8
    x = _bf16((T, hidden), 3)
    w = _bf16(((Hq + 2 * Hkv) * D, hidden), 4, std=0.3)
    pos = np.array([3, 17, 100, 4095, 7, 0], np.int32)
    q, k, _ = oracle.qkv_rope(x, w, pos, Hq, Hkv, D, style=style)
    q0, k0, _ = oracle.qkv_rope(x, w, np.zeros(T, np.int32), Hq, Hkv, D, style=style)

    def pair_norms(a):
        if style == 0:
            return a[..., 0::2] ** 2 + a[..., 1::2] ** 2
        return a[..., :D // 2] ** 2 + a[..., D // 2:] ** 2
    np.testing.assert_allclose(pair_norms(q), pair_norms(q0), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(pair_norms(k), pair_norms(k0), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("style", [0, 1])
def test_relative_position_property(style):
    T, hidden, Hq, Hkv, D = 2, 24, 2, 1, 16
    x = _bf16((T, hidden), 5)
    w = _bf16(((Hq + 2 * Hkv) * D, hidden), 6, std=0.3)

    def score(m, n):
        q, k, _ = oracle.qkv_rope(x, w, np.array([m, n], np.int32), Hq, Hkv, D, style=style)
        return q[0] @ k[1, 0]          # both query heads against the KV head
    base = score(40, 13)
    for c in (1, 100, 3000):
        np.testing.assert_allclose(score(40 + c, 13 + c), base, rtol=1e-9, atol=1e-9)
    assert not np.allclose(score(41, 13), base)   # but it does depend on m - n


def test_styles_equivalent_under_permutation():
    T, hidden, Hq, Hkv, D = 5, 16, 2, 2, 8
    x = _bf16((T, hidden), 7)
    w = _bf16(((Hq + 2 * Hkv) * D, hidden), 8, std=0.3)
    # Permute the rows of every Q/K head so that y'[2i] = y[i], y'[2i+1] = y[i + D/2].
    perm_head = np.empty(D, dtype=np.int64)
    perm_head[0::2] = np.arange(D // 2)
    perm_head[1::2] = np.arange(D // 2) + D // 2
    rows = []
    for h in range(Hq + 2 * Hkv):
        rows.append(h * D + (perm_head if h < Hq + Hkv else np.arange(D)))
    wp = w[torch.from_numpy(np.concatenate(rows))]
    pos = np.array([0, 9, 250, 77, 1], np.int32)
    q1, k1, v1 = oracle.qkv_rope(x, w, pos, Hq, Hkv, D, style=1)
    q0, k0, v0 = oracle.qkv_rope(x, wp, pos, Hq, Hkv, D, style=0)
    np.testing.assert_allclose(q0, q1[..., perm_head], rtol=0, atol=1e-12)
    np.testing.assert_allclose(k0, k1[..., perm_head], rtol=0, atol=1e-12)
    np.testing.assert_allclose(v0, v1, rtol=0, atol=0)


def test_token_subset_and_invalid_arguments():
    T, hidden, Hq, Hkv, D = 7, 16, 2, 1, 4
    x = _bf16((T, hidden), 9)
    w = _bf16(((Hq + 2 * Hkv) * D, hidden), 10)
    pos = np.arange(T, dtype=np.int32) * 3
    q, k, v = oracle.qkv_rope(x, w, pos, Hq, Hkv, D)
    qs, ks, vs = oracle.qkv_rope(x, w, pos, Hq, Hkv, D, tokens=[6, 0, 3])
    np.testing.assert_array_equal(qs, q[[6, 0, 3]])
    np.testing.assert_array_equal(ks, k[[6, 0, 3]])
    np.testing.assert_array_equal(vs, v[[6, 0, 3]])
    with pytest.raises(ValueError):
        oracle.qkv_rope(x, w, pos, Hq, Hkv, D, tokens=[T])
    with pytest.raises(ValueError):
        oracle.qkv_rope(x, w, pos, Hq, Hkv, D, style=2)


@pytest.mark.parametrize("style", [0, 1])
def test_second_pair_frequency(style):
    # D = 4: pair 1 turns at theta_1 = base^(-2/4) = 1/100 for base 10000.
    eye = torch.eye(4)
    w = torch.cat([eye, eye, eye]).to(torch.bfloat16)
    pos = np.array([0, 1, 50, 314, 8000], dtype=np.int32)
    a, b = (2, 3) if style == 0 else (1, 3)
    xr = torch.zeros((pos.size, 4))
    xr[:, a] = 1.0
    q, _, _ = oracle.qkv_rope(xr.to(torch.bfloat16), w, pos, 1, 1, 4, base=10000.0, style=style)
    ang = pos.astype(np.float64) / 100.0
    np.testing.assert_allclose(q[:, 0, a], np.cos(ang), rtol=0, atol=1e-12)
    np.testing.assert_allclose(q[:, 0, b], np.sin(ang), rtol=0, atol=1e-12)
    other = [d for d in range(4) if d not in (a, b)]
    np.testing.assert_allclose(q[:, 0, other], 0.0, rtol=0, atol=0)
