"""GPU parity of the CUDA library against the fp64 CPU oracle.

Tolerances (bf16 inputs, fp32 accumulation, P rounded to bf16 before P*V):
  O:   max |O_gpu - O_ref| <= 2e-2
  LSE: |LSE_gpu - LSE_ref| <= 1e-3 * max(1, |LSE_ref|)
Rows with no visible key must match exactly (O = 0, LSE = -inf).
A bf16 O is the fp32 O rounded to nearest even (checked bit for bit), so it may
also differ by that rounding, at most 2^-8 of its magnitude: per element
|O_gpu - O_ref| <= 2e-2 + 2^-8 * (|O_ref| + 2e-2).
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

import oracle
import tensor_attn_fwd_gb300 as attn
from attn_inputs import WORKLOADS, make_qkv, sample_rows, workload_inputs

pytestmark = pytest.mark.gpu

O_TOL = 2e-2
LSE_TOL = 1e-3
BF16_REL = 2.0 ** -8  # round to nearest even into bf16's 8-bit significand


def assert_close(o_gpu, lse_gpu, o_ref, lse_ref, what="", o_bf16=False):
    """O within O_TOL (plus the bf16 rounding of the output when o_bf16), LSE
    within LSE_TOL relative to max(1, |LSE_ref|), the -inf pattern exact."""
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
    assert o_gpu.shape == o_ref.shape and lse_gpu.shape == lse_ref.shape
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite O"
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse_gpu), fin), f"{what}: -inf pattern differs"
    assert np.all(lse_gpu[~fin] == -np.inf)
    err_o = float(np.max(np.abs(o_gpu - o_ref))) if o_gpu.size else 0.0
    if o_bf16:
        excess = np.abs(o_gpu - o_ref) - (O_TOL + BF16_REL * (np.abs(o_ref) + O_TOL))
        worst = float(np.max(excess)) if o_gpu.size else -1.0
        assert worst <= 0.0, (f"{what}: bf16 O error {err_o:.3e} beyond 2e-2 plus the output "
                              f"rounding (by {worst:.3e})")
    else:
        assert err_o <= O_TOL, f"{what}: O max-abs error {err_o:.3e} > {O_TOL}"
    if np.any(fin):
        d = np.abs(lse_gpu[fin] - lse_ref[fin]) / np.maximum(1.0, np.abs(lse_ref[fin]))
        assert float(d.max()) <= LSE_TOL, f"{what}: LSE error {float(d.max()):.3e} > {LSE_TOL}"
    return err_o


def gpu_fwd(q, k, v, causal, scale):
    o, lse = attn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    return o.cpu().numpy(), lse.cpu().numpy()


def run_fwd_case(B, Hq, Hkv, Sq, Sk, D, causal, seed, q_std=1.0, k_std=1.0, v_dist="normal"):
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Sk, D, seed, q_std=q_std, k_std=k_std, v_dist=v_dist)
    scale = 1.0 / math.sqrt(D)
    o, lse = gpu_fwd(q, k, v, causal, scale)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, scale)
    return assert_close(o, lse, o_ref, lse_ref, f"B{B} Hq{Hq} Hkv{Hkv} Sq{Sq} Sk{Sk} D{D} c{causal}")


@pytest.mark.parametrize("cfg", [1, 2])
def test_workload_full(cfg):
    w = WORKLOADS[cfg]
    q, k, v = workload_inputs(w)
    o, lse = gpu_fwd(q, k, v, w.causal, w.scale)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, w.causal, w.scale)
    assert_close(o, lse, o_ref, lse_ref, w.name)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S", [1, 7, 127, 129, 300])
def test_odd_lengths(S, causal, D):
    run_fwd_case(1, 2, 1, S, S, D, causal, seed=100 + S)


@pytest.mark.parametrize("Sq,Sk", [(64, 300), (129, 1000), (300, 129), (1, 513), (200, 77)])
@pytest.mark.parametrize("causal", [False, True])
def test_unequal_lengths(Sq, Sk, causal):
    # Sq > Sk with causal masking leaves leading rows with no visible key.
    run_fwd_case(2, 4, 2, Sq, Sk, 128, causal, seed=Sq * 7 + Sk)


@pytest.mark.parametrize("Hq,Hkv", [(8, 1), (8, 8), (8, 2), (12, 3)])
def test_head_grouping(Hq, Hkv):
    run_fwd_case(2, Hq, Hkv, 256, 384, 64, True, seed=Hq * 10 + Hkv)


@pytest.mark.parametrize("Hq,Hkv,causal,S", [
    (4, 4, True, 700),     # causal MHA, D=128: single-CTA kernel
    (6, 2, True, 300),     # causal, group of 3: single-CTA kernel
    (6, 2, False, 777),    # non-causal, group of 3: CTA pairs over row blocks
    (3, 1, False, 1100),   # odd head count, row-block pairs, odd number of blocks
    (8, 2, True, 1500),    # group of 4: CTA pairs over heads
])
def test_d128_kernel_forms(Hq, Hkv, causal, S):
    run_fwd_case(2, Hq, Hkv, S, S, 128, causal, seed=Hq * 31 + S)


def test_multi_item_per_cta():
    # More 256-row work items than SMs, so CTAs walk several items each.
    run_fwd_case(2, 48, 8, 1024, 1024, 64, True, seed=77)


def test_peaky_scores_rescale_path():
    # Large score range forces the lazy O rescale on most rows.
    run_fwd_case(1, 4, 4, 640, 640, 128, False, seed=5, q_std=3.0, k_std=3.0, v_dist="uniform")


def test_invariants_on_gpu():
    B, Hq, Hkv, S, D = 1, 4, 2, 384, 128
    q, k, _ = make_qkv(B, Hq, Hkv, S, S, D, seed=9)
    ones = torch.ones((B, Hkv, S, D), dtype=torch.bfloat16)
    o, _ = gpu_fwd(q, k, ones, True, 0.1)
    assert np.max(np.abs(o - 1.0)) <= O_TOL  # rows of P sum to one
    qz = torch.zeros_like(q)
    _, k2, v2 = make_qkv(B, Hq, Hkv, S, S, D, seed=10)
    o, lse = gpu_fwd(qz, k2, v2, True, 0.1)
    vd = v2.double().numpy()
    for i in (0, 1, 200, S - 1):  # uniform over visible keys
        ref = vd[:, :, : i + 1].mean(axis=2).repeat(Hq // Hkv, axis=1)
        assert np.max(np.abs(o[:, :, i] - ref)) <= O_TOL
        assert np.max(np.abs(lse[:, :, i] - math.log(i + 1))) <= LSE_TOL * max(1, math.log(i + 1))
    o, _ = gpu_fwd(q, k, v2, True, 0.1)  # causal row 0 returns V row 0
    ref0 = vd[:, :, 0].repeat(Hq // Hkv, axis=1)
    assert np.max(np.abs(o[:, :, 0] - ref0)) <= 1e-6


@pytest.mark.parametrize("cfg", [3, 4])
def test_workload_full_size_sampled_rows(cfg):
    w = WORKLOADS[cfg]
    q, k, v = workload_inputs(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = attn.attn_fwd(qd, kd, vd, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    rows = sample_rows(w.B, w.Hq, w.Sq, n_random=256, seed=w.seed)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, w.causal, w.scale, rows=rows.numpy())
    o_s = o.reshape(-1, w.D)[rows.cuda()].cpu().numpy()
    lse_s = lse.reshape(-1)[rows.cuda()].cpu().numpy()
    assert_close(o_s, lse_s, o_ref, lse_ref, w.name)
    # Every output row is finite and normalised (|O| <= max |V|).
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    assert float(o.abs().max()) <= float(v.float().abs().max()) + 1e-3


@pytest.mark.parametrize("cfg,std", [(3, None), (4, None), (4, 2.0)])
def test_workload_full_size_every_row(cfg, std):
    # Every element of O and LSE at the full workload sizes against the oracle.
    # Workload 4's "N(0,2)" is read as variance 2 (std sqrt 2); std = 2 is the
    # other reading, whose scores are peakier still.
    w = WORKLOADS[cfg]
    if std is not None:
        w = dataclasses.replace(w, name=f"{w.name}_std{std:g}", q_std=std, k_std=std)
    q, k, v = workload_inputs(w)
    o, lse = gpu_fwd(q, k, v, w.causal, w.scale)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, w.causal, w.scale)
    assert_close(o, lse, o_ref, lse_ref, w.name)


# ---------------------------------------------------------------- decode

def gpu_decode(q, k, v, ns, scale):
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    op, lp = attn.attn_decode_splitkv(qd, kd, vd, ns, scale)
    o, lse = attn.attn_combine(op, lp)
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    return op.cpu().numpy(), lp.cpu().numpy(), o.cpu().numpy(), lse.cpu().numpy()


def test_decode_workload_full():
    w = WORKLOADS[5]
    q, k, v = workload_inputs(w)
    op, lp, o, lse = gpu_decode(q, k, v, w.num_splits, w.scale)
    op_ref, lp_ref = oracle.decode_split(q, k, v, w.num_splits, w.scale)
    assert_close(op, lp, op_ref, lp_ref, "partials")
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, False, w.scale)
    assert_close(o, lse, o_ref[:, :, 0], lse_ref[:, :, 0], w.name)


@pytest.mark.parametrize("B,Hq,Hkv,Sk,D,ns", [
    (2, 8, 2, 1, 128, 1),
    (3, 4, 4, 7, 64, 3),
    (2, 8, 1, 100, 128, 8),     # MQA, ragged blocks, empty splits
    (1, 16, 2, 1000, 64, 5),    # group of 8 -> two 4-head slices
    (2, 6, 2, 333, 128, 7),     # group of 3 (partial slice)
    (1, 32, 8, 4096, 128, 1),
    (1, 4, 1, 64, 128, 64),     # one key per split
    (2, 8, 2, 500, 256, 4),     # D = 256
    (1, 16, 1, 2000, 256, 7),   # D = 256, MQA, group of 16
    (3, 6, 2, 33, 256, 5),      # D = 256, ragged, empty splits
])
def test_decode_shapes(B, Hq, Hkv, Sk, D, ns):
    q, k, v = make_qkv(B, Hq, Hkv, 1, Sk, D, seed=B * 1000 + Sk + ns)
    scale = 1.0 / math.sqrt(D)
    op, lp, o, lse = gpu_decode(q, k, v, ns, scale)
    op_ref, lp_ref = oracle.decode_split(q, k, v, ns, scale)
    assert_close(op, lp, op_ref, lp_ref, "partials")
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, False, scale)
    assert_close(o, lse, o_ref[:, :, 0], lse_ref[:, :, 0], "combined")


@pytest.mark.parametrize("D", [64, 128, 256])
def test_combine_alone_against_oracle(D):
    # Feed the same partials (including empty splits) to both combines.
    g = torch.Generator().manual_seed(3)
    ns, B, Hq = 6, 3, 8
    op = torch.randn(ns, B, Hq, D, generator=g)
    lp = torch.randn(ns, B, Hq, generator=g) * 4
    lp[1] = -math.inf
    lp[:, 0, 0] = -math.inf  # a row whose splits are all empty
    op[:, 0, 0] = 0.0
    o, lse = attn.attn_combine(op.cuda(), lp.cuda())
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.combine(op.double().numpy(), lp.double().numpy())
    assert_close(o.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "combine")


def test_decode_split_invariance_on_gpu():
    # P is rounded to bf16 before P*V relative to each split's own reference
    # maximum, so different splittings round differently: |dO| <= 2^-9 * max|V|
    # bounds the difference; the LSE sums stay in fp32.
    q, k, v = make_qkv(2, 8, 2, 1, 777, 128, seed=42)
    outs = [gpu_decode(q, k, v, ns, 0.1)[2:] for ns in (1, 2, 3, 8, 16)]
    vmax = float(v.float().abs().max())
    for o, lse in outs[1:]:
        assert np.max(np.abs(o - outs[0][0])) <= 2.0 ** -9 * vmax
        assert np.max(np.abs(lse - outs[0][1])) <= 1e-4


def test_decode_matches_prefill_kernel():
    q, k, v = make_qkv(2, 8, 2, 1, 640, 128, seed=43)
    _, _, o, lse = gpu_decode(q, k, v, 4, 0.09)
    of, lf = gpu_fwd(q, k, v, False, 0.09)
    assert np.max(np.abs(o - of[:, :, 0])) <= O_TOL
    assert np.max(np.abs(lse - lf[:, :, 0])) <= LSE_TOL * 10


@pytest.mark.parametrize("B,Hq,Hkv,Sk,D,ns", [
    (6, 8, 2, 700, 128, 4),
    (5, 4, 4, 300, 64, 3),
    (4, 32, 8, 2048, 128, 8),
    (4, 8, 2, 900, 256, 3),     # D = 256
])
def test_decode_varlen(B, Hq, Hkv, Sk, D, ns):
    q, k, v = make_qkv(B, Hq, Hkv, 1, Sk, D, seed=B * 7 + Sk)
    g = torch.Generator().manual_seed(Sk)
    lens = torch.randint(0, Sk + 1, (B,), generator=g, dtype=torch.int32)
    lens[0] = 0            # empty sequence
    lens[1] = Sk           # full capacity
    lens[2] = 1            # a single key
    kd, vd = k.cuda(), v.cuda()
    # Cache slots past each sequence's length hold NaN: they must not leak in.
    for b in range(B):
        kd[b, :, int(lens[b]):] = float("nan")
        vd[b, :, int(lens[b]):] = float("nan")
    scale = 1.0 / math.sqrt(D)
    op, lp = attn.attn_decode_splitkv_varlen(q.cuda(), kd, vd, lens.cuda(), ns, scale)
    o, lse = attn.attn_combine(op, lp)
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    op, lp, o, lse = (t.cpu().numpy() for t in (op, lp, o, lse))
    for b in range(B):
        n = int(lens[b])
        qb = q[b:b + 1].contiguous()
        kb = k[b:b + 1, :, :n].contiguous()
        vb = v[b:b + 1, :, :n].contiguous()
        op_ref, lp_ref = oracle.decode_split(qb, kb, vb, ns, scale)
        assert_close(op[:, b:b + 1], lp[:, b:b + 1], op_ref, lp_ref, f"partials b={b} len={n}")
        o_ref, lse_ref = oracle.attn_fwd(qb, kb, vb, False, scale)
        assert_close(o[b:b + 1], lse[b:b + 1], o_ref[:, :, 0], lse_ref[:, :, 0], f"b={b} len={n}")


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D,causal", [
    (1, 2, 2, 128, 128, 64, False),
    (2, 8, 2, 700, 700, 128, True),
    (1, 4, 1, 300, 900, 128, True),
])
def test_bf16_output(B, Hq, Hkv, Sq, Sk, D, causal):
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Sk, D, seed=Sq + Sk)
    scale = 1.0 / math.sqrt(D)
    o16, lse = attn.attn_fwd_bf16o(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    o32, lse32 = attn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    assert o16.dtype == torch.bfloat16
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, scale)
    assert_close(o16.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "bf16 O",
                 o_bf16=True)
    # exactly the fp32 result rounded to nearest even
    assert torch.equal(o16, o32.to(torch.bfloat16))
    assert torch.equal(lse, lse32)


@pytest.mark.parametrize("B,Hq,Hkv,Sk,D,want", [
    (64, 32, 8, 4096, 128, 1),     # 512 CTAs already fill the SMs
    (4, 32, 8, 8192, 128, None),   # 32 CTAs: several splits
    (8, 32, 4, 32768, 256, None),  # D = 256: one CTA per SM, so one wave
    (1, 32, 8, 2048, 128, 8),      # capped at Sk / 256 (128 KB of K and V a split)
    (1, 32, 8, 4096, 128, None),   # 8 CTAs a split: 152 SMs -> 16 splits
    (4, 32, 4, 32768, 64, None),   # D = 64: two CTAs per SM
    (1, 32, 8, 8192, 64, 16),      # D = 64: capped at Sk / 512
    (1, 8, 1, 16384, 128, 32),     # one CTA a split: at most 32 splits
    (1, 4, 1, 500, 128, 1),        # too short to split
])
def test_decode_num_splits_rule(B, Hq, Hkv, Sk, D, want):
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    ns = attn.attn_decode_num_splits(B, Hq, Hkv, Sk, D)
    base = B * Hkv * (((Hq // Hkv) + 15) // 16)
    if D == 256:
        per_sm = max(1, n_sm // base)
    else:
        t = -(-(2 if D == 64 else 1) * n_sm // base)
        per_sm = min(32, 1 << int(math.floor(math.log2(t) + 0.5)))
    expect = want if want is not None else min(per_sm, max(1, Sk // (32768 // D)))
    assert ns == expect
    # and the default decode path uses it and matches the oracle
    q, k, v = make_qkv(B, Hq, Hkv, 1, Sk, D, seed=B + Sk)
    o, lse = attn.decode(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, False, 1.0 / math.sqrt(D))
    assert_close(o.cpu().numpy(), lse.cpu().numpy(), o_ref[:, :, 0], lse_ref[:, :, 0], "auto splits")
