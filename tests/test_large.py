"""Long sequences: the decode, chunked-prefill and prefill paths against the
fp64 oracle on caches of 2^18 - 2^20 keys (sampled rows where the oracle would
take too long on all of them), tolerances as in test_parity."""
import math

import numpy as np
import pytest
import torch

import oracle
import tensor_attn_fwd_gb300 as attn
from attn_inputs import make_qkv, sample_rows

pytestmark = pytest.mark.gpu

O_TOL = 2e-2
LSE_TOL = 1e-3


def check(o_gpu, lse_gpu, o_ref, lse_ref, what):
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
    assert np.all(np.isfinite(o_gpu)) and np.all(np.isfinite(lse_gpu)), what
    err_o = float(np.max(np.abs(o_gpu - o_ref)))
    err_l = float(np.max(np.abs(lse_gpu - lse_ref) / np.maximum(1.0, np.abs(lse_ref))))
    assert err_o <= O_TOL, f"{what}: O max-abs error {err_o:.3e}"
    assert err_l <= LSE_TOL, f"{what}: LSE error {err_l:.3e}"


def test_decode_million_keys():
    """One query row per head against 2^20 keys (split count from the rule)."""
    B, Hq, Hkv, Sk, D = 1, 8, 1, 1 << 20, 128
    q, k, v = make_qkv(B, Hq, Hkv, 1, Sk, D, seed=2024)
    scale = 1.0 / math.sqrt(D)
    o, lse = attn.decode(q.cuda(), k.cuda(), v.cuda(), scale=scale)
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, False, scale)
    check(o.cpu().numpy(), lse.cpu().numpy(), o_ref[:, :, 0], lse_ref[:, :, 0], "decode 2^20")


def test_chunk_against_long_cache():
    """A 100-row causal chunk against 2^18 keys: paired heads, KV splits."""
    B, Hq, Hkv, Sq, Sk, D = 1, 4, 1, 100, 1 << 18, 128
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Sk, D, seed=77)
    scale = 1.0 / math.sqrt(D)
    o, lse = attn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=scale,
                           num_splits="auto")
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    rows = sample_rows(B, Hq, Sq, n_random=24, seed=5)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, True, scale, rows=rows.numpy())
    og = o.reshape(-1, D)[rows.cuda()].cpu().numpy()
    lg = lse.reshape(-1)[rows.cuda()].cpu().numpy()
    check(og, lg, o_ref, lse_ref, "chunk vs 2^18")


def test_long_prefill():
    """A 65536 x 65536 non-causal prefill (one pass), sampled rows."""
    B, H, S, D = 1, 2, 1 << 16, 64
    q, k, v = make_qkv(B, H, H, S, S, D, seed=99)
    scale = 1.0 / math.sqrt(D)
    o, lse = attn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=False, scale=scale)
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    rows = sample_rows(B, H, S, n_random=32, seed=6)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, False, scale, rows=rows.numpy())
    og = o.reshape(-1, D)[rows.cuda()].cpu().numpy()
    lg = lse.reshape(-1)[rows.cuda()].cpu().numpy()
    check(og, lg, o_ref, lse_ref, "prefill 2^16")
