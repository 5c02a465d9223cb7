"""Pins for the fp64 CPU oracle (CPU only).

Each test checks the oracle against something other than itself: brute force
in 50-digit arithmetic without the max shift, closed forms the definition
fixes (uniform attention, identical value rows, causal row 0, the two-key
logistic), invariants (rows of P sum to one, linearity in V, key permutation,
GQA = MHA with repeated KV heads, split invariance of the LSE combine) and an
independent library routine (PyTorch's fp64 scaled-dot-product attention plus
SciPy's logsumexp).  Together they catch a dropped term, a wrong sign or index,
a transposed operand, a wrong head mapping or a wrong causal alignment.
"""
import math

import mpmath
import numpy as np
import pytest
import torch

import oracle
from attn_inputs import make_qkv

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def f64(x):
    return x.to(torch.float64).numpy()


def visible(i, Sq, Sk, causal):
    if not causal:
        return Sk
    return max(0, min(Sk, i + Sk - Sq + 1))


def brute_force(q, k, v, causal, scale):
    """Explicit score matrix, exp without max shift, normalise, multiply (mpmath)."""
    mpmath.mp.dps = 50
    B, Hq, Sq, D = q.shape
    _, Hkv, Sk, _ = k.shape
    grp = Hq // Hkv
    qd, kd, vd = f64(q), f64(k), f64(v)
    O = np.zeros((B, Hq, Sq, D))
    L = np.zeros((B, Hq, Sq))
    for b in range(B):
        for h in range(Hq):
            g = h // grp
            for i in range(Sq):
                n = visible(i, Sq, Sk, causal)
                if n == 0:
                    O[b, h, i] = 0.0
                    L[b, h, i] = -math.inf
                    continue
                e = []
                for j in range(n):
                    s = mpmath.mpf(0)
                    for d in range(D):
                        s += mpmath.mpf(qd[b, h, i, d]) * mpmath.mpf(kd[b, g, j, d])
                    e.append(mpmath.exp(mpmath.mpf(scale) * s))
                tot = mpmath.fsum(e)
                for d in range(D):
                    O[b, h, i, d] = float(mpmath.fsum(e[j] * mpmath.mpf(vd[b, g, j, d])
                                                      for j in range(n)) / tot)
                L[b, h, i] = float(mpmath.log(tot))
    return O, L


TINY = [
    # B, Hq, Hkv, Sq, Sk, D, causal
    (1, 1, 1, 1, 1, 1, False),
    (1, 2, 1, 5, 5, 4, True),
    (2, 4, 2, 3, 7, 8, False),
    (1, 2, 2, 4, 6, 3, True),     # Sq < Sk, bottom-right causal
    (1, 3, 1, 6, 4, 5, True),     # Sq > Sk: leading rows fully masked
    (2, 2, 1, 8, 8, 8, True),
]


@pytest.mark.parametrize("shape", TINY)
def test_brute_force_tiny(shape):
    B, Hq, Hkv, Sq, Sk, D, causal = shape
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Sk, D, seed=7 + Sq * 13 + D)
    scale = 0.37
    O, L = oracle.attn_fwd(q, k, v, causal, scale)
    Ob, Lb = brute_force(q, k, v, causal, scale)
    finite = np.isfinite(Lb)
    assert np.array_equal(np.isfinite(L), finite)
    assert np.all(L[~finite] == -np.inf)
    np.testing.assert_allclose(O, Ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L[finite], Lb[finite], rtol=0, atol=1e-12)


def test_library_sdpa_fp64():
    """Independent library routine: torch SDPA (fp64, CPU) + scipy logsumexp."""
    from scipy.special import logsumexp
    B, Hq, Hkv, Sq, Sk, D = 2, 6, 3, 33, 47, 16
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Sk, D, seed=11)
    scale = 1.0 / math.sqrt(D)
    for causal in (False, True):
        O, L = oracle.attn_fwd(q, k, v, causal, scale)
        grp = Hq // Hkv
        kq = k.to(torch.float64).repeat_interleave(grp, dim=1)
        vq = v.to(torch.float64).repeat_interleave(grp, dim=1)
        qq = q.to(torch.float64)
        i = torch.arange(Sq)[:, None]
        j = torch.arange(Sk)[None, :]
        mask = (j <= i + Sk - Sq) if causal else torch.ones(Sq, Sk, dtype=torch.bool)
        ref = torch.nn.functional.scaled_dot_product_attention(
            qq, kq, vq, attn_mask=mask, scale=scale)
        np.testing.assert_allclose(O, ref.numpy(), rtol=0, atol=1e-12)
        s = (qq @ kq.transpose(-1, -2)).numpy() * scale
        s = np.where(mask.numpy()[None, None], s, -np.inf)
        np.testing.assert_allclose(L, logsumexp(s, axis=-1), rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_rows_of_p_sum_to_one(causal):
    B, Hq, Hkv, S, D = 1, 4, 2, 40, 32
    q, k, _ = make_qkv(B, Hq, Hkv, S, S, D, seed=3)
    v = torch.ones((B, Hkv, S, D), dtype=torch.bfloat16)
    O, _ = oracle.attn_fwd(q, k, v, causal, 0.5)
    np.testing.assert_allclose(O, 1.0, rtol=0, atol=1e-14)


def test_linearity_in_v():
    B, Hq, Hkv, S, D = 1, 2, 2, 24, 8
    q, k, _ = make_qkv(B, Hq, Hkv, S, S, D, seed=5)
    g = torch.Generator().manual_seed(9)
    # small integers: 2*V1 + V2 stays exact in bf16
    v1 = torch.randint(-8, 9, (B, Hkv, S, D), generator=g).to(torch.bfloat16)
    v2 = torch.randint(-8, 9, (B, Hkv, S, D), generator=g).to(torch.bfloat16)
    v12 = (2 * v1.float() + v2.float()).to(torch.bfloat16)
    for causal in (False, True):
        O1, _ = oracle.attn_fwd(q, k, v1, causal, 0.3)
        O2, _ = oracle.attn_fwd(q, k, v2, causal, 0.3)
        O12, L12 = oracle.attn_fwd(q, k, v12, causal, 0.3)
        np.testing.assert_allclose(O12, 2 * O1 + O2, rtol=0, atol=1e-12)


@pytest.mark.parametrize("Sq,Sk,causal", [(16, 16, False), (16, 16, True),
                                          (5, 12, True), (12, 5, True)])
def test_zero_query_is_mean_of_visible_rows(Sq, Sk, causal):
    B, Hq, Hkv, D = 2, 4, 1, 16
    _, k, v = make_qkv(B, Hq, Hkv, Sq, Sk, D, seed=21)
    q = torch.zeros((B, Hq, Sq, D), dtype=torch.bfloat16)
    O, L = oracle.attn_fwd(q, k, v, causal, 0.125)
    vd = f64(v)
    for i in range(Sq):
        n = visible(i, Sq, Sk, causal)
        if n == 0:
            assert np.all(O[:, :, i] == 0.0) and np.all(L[:, :, i] == -np.inf)
            continue
        mean = vd[:, 0, :n, :].mean(axis=1)  # [B, D]
        np.testing.assert_allclose(O[:, :, i], np.broadcast_to(mean[:, None], (B, Hq, D)),
                                   rtol=0, atol=1e-13)
        np.testing.assert_allclose(L[:, :, i], math.log(n), rtol=0, atol=1e-13)


def test_scale_zero_is_uniform():
    B, Hq, Hkv, S, D = 1, 2, 2, 20, 8
    q, k, v = make_qkv(B, Hq, Hkv, S, S, D, seed=4)
    O, L = oracle.attn_fwd(q, k, v, False, 0.0)
    np.testing.assert_allclose(O, f64(v).mean(axis=2, keepdims=True).repeat(S, axis=2),
                               rtol=0, atol=1e-13)
    np.testing.assert_allclose(L, math.log(S), rtol=0, atol=1e-13)


def test_identical_value_rows():
    B, Hq, Hkv, S, D = 2, 4, 2, 30, 16
    q, k, _ = make_qkv(B, Hq, Hkv, S, S, D, seed=8)
    row = torch.randn(D, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    v = row.expand(B, Hkv, S, D).contiguous()
    for causal in (False, True):
        O, _ = oracle.attn_fwd(q, k, v, causal, 0.2)
        np.testing.assert_allclose(O, np.broadcast_to(f64(row), O.shape), rtol=0,
                                   atol=1e-13)


def test_causal_row_zero():
    B, Hq, Hkv, S, D = 2, 4, 2, 17, 32
    q, k, v = make_qkv(B, Hq, Hkv, S, S, D, seed=12)
    scale = 1 / math.sqrt(D)
    O, L = oracle.attn_fwd(q, k, v, True, scale)
    qd, kd, vd = f64(q), f64(k), f64(v)
    for b in range(B):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            np.testing.assert_array_equal(O[b, h, 0], vd[b, g, 0])
            assert L[b, h, 0] == pytest.approx(scale * float(qd[b, h, 0] @ kd[b, g, 0]),
                                               abs=1e-13)


def test_two_key_logistic():
    """Two visible keys: P = logistic(s0 - s1); LSE = s1 + log1p(exp(s0 - s1))."""
    q, k, v = make_qkv(1, 1, 1, 1, 2, 4, seed=31)
    scale = 0.7
    O, L = oracle.attn_fwd(q, k, v, False, scale)
    qd, kd, vd = f64(q)[0, 0, 0], f64(k)[0, 0], f64(v)[0, 0]
    s0, s1 = scale * qd @ kd[0], scale * qd @ kd[1]
    p0 = 1.0 / (1.0 + math.exp(s1 - s0))
    np.testing.assert_allclose(O[0, 0, 0], p0 * vd[0] + (1 - p0) * vd[1], atol=1e-14)
    assert L[0, 0, 0] == pytest.approx(s1 + math.log1p(math.exp(s0 - s1)), abs=1e-14)


def test_gqa_equals_mha_with_repeated_kv():
    B, Hq, Hkv, S, D = 2, 8, 2, 21, 16
    q, k, v = make_qkv(B, Hq, Hkv, S, S, D, seed=13)
    grp = Hq // Hkv
    kr = k.repeat_interleave(grp, dim=1).contiguous()
    vr = v.repeat_interleave(grp, dim=1).contiguous()
    for causal in (False, True):
        O1, L1 = oracle.attn_fwd(q, k, v, causal, 0.25)
        O2, L2 = oracle.attn_fwd(q, kr, vr, causal, 0.25)
        np.testing.assert_array_equal(O1, O2)
        np.testing.assert_array_equal(L1, L2)


def test_key_permutation_invariance():
    B, Hq, Hkv, S, D = 1, 4, 2, 25, 16
    q, k, v = make_qkv(B, Hq, Hkv, S, S, D, seed=14)
    perm = torch.randperm(S, generator=torch.Generator().manual_seed(3))
    O1, L1 = oracle.attn_fwd(q, k, v, False, 0.25)
    O2, L2 = oracle.attn_fwd(q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous(),
                             False, 0.25)
    np.testing.assert_allclose(O1, O2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(L1, L2, rtol=0, atol=1e-13)


def test_causal_alignment_is_bottom_right():
    """Sq < Sk: the last query row sees every key, row i sees i + Sk - Sq + 1."""
    B, Hq, Hkv, Sq, Sk, D = 1, 2, 1, 4, 9, 8
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Sk, D, seed=15)
    Oc, Lc = oracle.attn_fwd(q, k, v, True, 0.3)
    On, Ln = oracle.attn_fwd(q, k, v, False, 0.3)
    np.testing.assert_array_equal(Oc[:, :, -1], On[:, :, -1])
    for i in range(Sq):
        n = i + Sk - Sq + 1
        Oi, Li = oracle.attn_fwd(q[:, :, i:i + 1].contiguous(), k[:, :, :n].contiguous(),
                                 v[:, :, :n].contiguous(), False, 0.3)
        np.testing.assert_array_equal(Oc[:, :, i:i + 1], Oi)
        np.testing.assert_array_equal(Lc[:, :, i:i + 1], Li)


def test_row_selection_matches_full():
    B, Hq, Hkv, S, D = 2, 4, 2, 50, 16
    q, k, v = make_qkv(B, Hq, Hkv, S, S, D, seed=16)
    O, L = oracle.attn_fwd(q, k, v, True, 0.25)
    rows = np.array([0, 7, 49, 50, 123, B * Hq * S - 1])
    Or, Lr = oracle.attn_fwd(q, k, v, True, 0.25, rows=rows)
    np.testing.assert_array_equal(Or, O.reshape(-1, D)[rows])
    np.testing.assert_array_equal(Lr, L.reshape(-1)[rows])


@pytest.mark.parametrize("align", [1, 32])
@pytest.mark.parametrize("Sk", [1, 7, 10, 64, 100])
def test_split_invariance(Sk, align):
    B, Hq, Hkv, D = 2, 8, 2, 16
    q, k, v = make_qkv(B, Hq, Hkv, 1, Sk, D, seed=17 + Sk)
    O, L = oracle.attn_fwd(q, k, v, False, 0.25)
    for ns in sorted({1, 2, 3, 8, Sk}):
        if ns > Sk:
            continue
        op, lp = oracle.decode_split(q, k, v, ns, 0.25, align=align)
        chunk = -(-(-(-Sk // ns)) // align) * align
        for s in range(ns):  # empty splits carry -inf and zeros
            if s * chunk >= Sk:
                assert np.all(lp[s] == -np.inf) and np.all(op[s] == 0.0)
        Oc, Lc = oracle.combine(op, lp)
        np.testing.assert_allclose(Oc, O[:, :, 0], rtol=0, atol=1e-13)
        np.testing.assert_allclose(Lc, L[:, :, 0], rtol=0, atol=1e-13)


def test_combine_all_empty_and_single():
    op = np.zeros((3, 2, 4))
    lp = np.full((3, 2), -np.inf)
    o, l = oracle.combine(op, lp)
    assert np.all(o == 0) and np.all(l == -np.inf)
    rng = np.random.default_rng(0)
    op1 = rng.standard_normal((1, 5, 8))
    lp1 = rng.standard_normal((1, 5))
    o, l = oracle.combine(op1, lp1)
    np.testing.assert_array_equal(o, op1[0])
    np.testing.assert_array_equal(l, lp1[0])


def test_invalid_arguments_rejected():
    q, k, v = make_qkv(1, 3, 2, 4, 4, 8, seed=1)  # Hq % Hkv != 0
    with pytest.raises(ValueError):
        oracle.attn_fwd(q, k, v, False, 1.0)


def test_aligned_split_boundaries():
    """align=32: split s holds exactly keys [32*ceil(ceil(Sk/ns)/32)*s, ...)."""
    B, Hq, Hkv, Sk, D = 1, 2, 1, 100, 8
    q, k, v = make_qkv(B, Hq, Hkv, 1, Sk, D, seed=5)
    op, lp = oracle.decode_split(q, k, v, 3, 0.5, align=32)   # chunk 34 -> 64
    o0, l0 = oracle.attn_fwd(q, k[:, :, :64], v[:, :, :64], False, 0.5)
    o1, l1 = oracle.attn_fwd(q, k[:, :, 64:], v[:, :, 64:], False, 0.5)
    np.testing.assert_array_equal(op[0], o0[:, :, 0])
    np.testing.assert_array_equal(lp[0], l0[:, :, 0])
    np.testing.assert_array_equal(op[1], o1[:, :, 0])
    np.testing.assert_array_equal(lp[1], l1[:, :, 0])
    assert np.all(lp[2] == -np.inf) and np.all(op[2] == 0.0)


def test_gather_paged_recovers_sequences():
    """A cache built from contiguous K with shuffled pages gathers back to each
    sequence's prefix, bit for bit; unused pages (NaN) are never read."""
    B, Hkv, Sk, D, page = 3, 2, 96, 8, 32
    _, k, _ = make_qkv(B, Hkv, Hkv, 1, Sk, D, seed=9)
    npp = Sk // page
    num_pages = B * npp + 2
    perm = torch.randperm(num_pages, generator=torch.Generator().manual_seed(3))
    cache = torch.full((num_pages, Hkv, page, D), float("nan")).to(torch.bfloat16)
    table = torch.zeros((B, npp), dtype=torch.int32)
    for b in range(B):
        for p in range(npp):
            pid = int(perm[b * npp + p])
            cache[pid] = k[b, :, p * page:(p + 1) * page]
            table[b, p] = pid
    lens = torch.tensor([0, 33, 96], dtype=torch.int32)
    for b in range(B):
        got = oracle.gather_paged(cache, table, lens, b)
        n = int(lens[b])
        assert got.shape == (1, Hkv, n, D)
        assert torch.equal(got.view(torch.int16), k[b:b + 1, :, :n].contiguous().view(torch.int16))
    bad = table.clone()
    bad[1, 1] = num_pages
    with pytest.raises(ValueError):
        oracle.gather_paged(cache, bad, lens, 1)
