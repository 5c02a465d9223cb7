"""GPU parity of the head-dimension-256 forward (one query tile per CTA,
double-buffered S) against the fp64 oracle, with the tolerances of the
D = 64 / 128 kernel."""
import math

import numpy as np
import pytest
import torch

import oracle
import tensor_attn_fwd_gb300 as attn
from attn_inputs import make_qkv, sample_rows
from test_parity import assert_close, gpu_fwd, run_fwd_case

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S", [1, 7, 128, 129, 300])
def test_d256_odd_lengths(S, causal):
    run_fwd_case(1, 2, 1, S, S, 256, causal, seed=300 + S)


@pytest.mark.parametrize("Sq,Sk", [(64, 300), (129, 1000), (300, 129), (1, 513), (200, 77)])
@pytest.mark.parametrize("causal", [False, True])
def test_d256_unequal_lengths(Sq, Sk, causal):
    run_fwd_case(2, 4, 2, Sq, Sk, 256, causal, seed=Sq * 5 + Sk)


@pytest.mark.parametrize("Hq,Hkv", [(8, 1), (8, 8), (8, 2)])
def test_d256_head_grouping(Hq, Hkv):
    run_fwd_case(1, Hq, Hkv, 384, 384, 256, True, seed=Hq * 3 + Hkv)


def test_d256_multi_item_per_cta():
    # 2*16*16 = 512 query tiles: every CTA walks several items, and each
    # item's first scores are issued during the previous item's last step.
    run_fwd_case(2, 16, 4, 2048, 2048, 256, True, seed=81)


def test_d256_peaky_scores_rescale_path():
    # Large score range: the lazy rescale of O runs while the previous step's
    # product may still be in flight (the kernel waits for it).
    run_fwd_case(1, 4, 4, 1024, 1024, 256, False, seed=6, q_std=3.0, k_std=3.0,
                 v_dist="uniform")


def test_d256_bf16_output():
    q, k, v = make_qkv(2, 4, 2, 500, 700, 256, seed=12)
    scale = 1.0 / 16.0
    o16, lse16 = attn.attn_fwd_bf16o(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=scale)
    o32, lse32 = attn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=scale)
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, True, scale)
    assert_close(o16.float().cpu().numpy(), lse16.cpu().numpy(), o_ref, lse_ref, "bf16 O",
                 o_bf16=True)
    assert torch.equal(o16, o32.to(torch.bfloat16))
    assert torch.equal(lse16, lse32)


def test_d256_large_sampled():
    """Causal GQA B2 Hq16 Hkv4 S8192 D256 on sampled rows."""
    B, Hq, Hkv, S, D = 2, 16, 4, 8192, 256
    q, k, v = make_qkv(B, Hq, Hkv, S, S, D, seed=2561)
    scale = 1.0 / 16.0
    o, lse = attn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=scale)
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    rows = sample_rows(B, Hq, S, n_random=192, seed=2562)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, True, scale, rows=rows.numpy())
    o_s = o.reshape(-1, D)[rows.cuda()].cpu().numpy()
    lse_s = lse.reshape(-1)[rows.cuda()].cpu().numpy()
    assert_close(o_s, lse_s, o_ref, lse_ref, "D256 S8192 sampled")


def test_d256_chunked_order_every_row():
    """Causal multi-head B8 H16 S2048 D256: 268 MB of K/V, so the kernel walks
    the items in chunks of 24 KV heads (the last chunk holds 8), longest first
    within each; every row against the oracle."""
    B, H, S, D = 8, 16, 2048, 256
    q, k, v = make_qkv(B, H, H, S, S, D, seed=2563)
    scale = 1.0 / 16.0
    o, lse = attn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=scale)
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, True, scale)
    assert_close(o.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "D256 chunked order")


def test_d256_chunked_order_gqa_sampled():
    """Causal GQA B4 Hq32 Hkv8 S4096 D256: 134 MB of K/V, chunks of 12 KV heads
    (the last holds 8), on sampled rows (every head's edge rows included)."""
    B, Hq, Hkv, S, D = 4, 32, 8, 4096, 256
    q, k, v = make_qkv(B, Hq, Hkv, S, S, D, seed=2564)
    scale = 1.0 / 16.0
    o, lse = attn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=scale)
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    rows = sample_rows(B, Hq, S, n_random=256, seed=2565)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, True, scale, rows=rows.numpy())
    o_s = o.reshape(-1, D)[rows.cuda()].cpu().numpy()
    lse_s = lse.reshape(-1)[rows.cuda()].cpu().numpy()
    assert_close(o_s, lse_s, o_ref, lse_ref, "D256 chunked order GQA sampled")


def test_d256_backward_and_split_prefill_unsupported():
    """D = 256 has the one-pass forward and split-KV decode (parity in
    test_parity); the backward and the split-KV prefill report
    ATTN_ERR_UNSUPPORTED."""
    q, k, v = (t.cuda() for t in make_qkv(1, 2, 1, 64, 300, 256, seed=1))
    o, lse = attn.attn_fwd(q, k, v)
    with pytest.raises(attn.AttnError) as e:
        attn.attn_bwd(q, k, v, o, lse, q)
    assert e.value.status == attn.ATTN_ERR_UNSUPPORTED
    with pytest.raises(attn.AttnError) as e:
        attn.attn_fwd_splitkv(q, k, v, 2)
    assert e.value.status == attn.ATTN_ERR_UNSUPPORTED
