"""Prefill over KV splits (attn_fwd_splitkv + attn_combine, i.e. attn_fwd with
num_splits > 1) against the fp64 oracle, with the tolerances of test_parity:
the combined O and LSE are the full attention whatever the split count."""
import math

import numpy as np
import pytest
import torch

import oracle
import tensor_attn_fwd_gb300 as attn
from attn_inputs import make_qkv

pytestmark = pytest.mark.gpu

O_TOL = 2e-2
LSE_TOL = 1e-3


def assert_close(o_gpu, lse_gpu, o_ref, lse_ref, what):
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite O"
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse_gpu), fin), f"{what}: -inf pattern differs"
    err_o = float(np.max(np.abs(o_gpu - o_ref)))
    assert err_o <= O_TOL, f"{what}: O max-abs error {err_o:.3e}"
    if np.any(fin):
        d = np.abs(lse_gpu[fin] - lse_ref[fin]) / np.maximum(1.0, np.abs(lse_ref[fin]))
        assert float(d.max()) <= LSE_TOL, f"{what}: LSE error {float(d.max()):.3e}"


CASES = [
    # B, Hq, Hkv, Sq, Sk, D, causal, num_splits
    (1, 4, 2, 64, 1000, 128, True, 3),      # a short chunk, ragged last key tile
    (2, 8, 2, 200, 2048, 64, True, 4),
    (1, 4, 4, 300, 300, 128, True, 2),      # Sq = Sk
    (1, 2, 1, 128, 4096, 128, False, 32),   # one 128-key tile per split
    (1, 4, 4, 500, 100, 64, True, 1),       # Sq > Sk: leading rows see no key
    (1, 4, 4, 500, 300, 64, True, 3),       # ... with splits
    (2, 4, 1, 256, 1536, 128, True, 5),     # MQA, splits of 3 tiles (the last one 0)
    (1, 3, 3, 1, 777, 128, False, 7),       # one query row
]


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D,causal,ns", CASES)
def test_splitkv_matches_oracle(B, Hq, Hkv, Sq, Sk, D, causal, ns):
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Sk, D, seed=B * 1000 + Sq * 7 + Sk + ns)
    scale = 1.0 / math.sqrt(D)
    o, lse = attn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale,
                           num_splits=ns)
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, scale)
    assert_close(o.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref,
                 f"B{B} Hq{Hq} Sq{Sq} Sk{Sk} D{D} c{causal} ns{ns}")


def test_one_split_is_the_plain_forward():
    """With one split the partial is attn_fwd's output, bit for bit."""
    q, k, v = make_qkv(2, 4, 2, 300, 700, 128, seed=5)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o, lse = attn.attn_fwd(q, k, v, causal=True)
    o_part, lse_part = attn.attn_fwd_splitkv(q, k, v, 1, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o_part[0], o) and torch.equal(lse_part[0], lse)


def test_partials_of_keyless_splits():
    """A split that holds no key a row may see leaves O = 0 and LSE = -inf for it:
    with Sq = Sk causal, split s (keys from 128*t*s) is empty for every row
    below that key."""
    S, ns = 512, 4
    q, k, v = make_qkv(1, 2, 2, S, S, 64, seed=9)
    o_part, lse_part = attn.attn_fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), ns, causal=True)
    torch.cuda.synchronize()
    o_part, lse_part = o_part.cpu(), lse_part.cpu()
    t = 128 * (((S + 127) // 128 + ns - 1) // ns)  # keys per split
    for s in range(ns):
        rows = torch.arange(S) < s * t  # rows whose last visible key precedes the split
        assert torch.all(lse_part[s][..., rows] == -math.inf)
        assert torch.all(o_part[s][:, :, rows] == 0)
        assert torch.all(torch.isfinite(lse_part[s][..., ~rows]))


def test_auto_split_count():
    # Few work items (B * Hq * ceil(Sq/256) = 4) against a long cache: splits.
    ns = attn.attn_fwd_num_splits(1, 4, 2, 200, 8192, 128)
    assert 1 < ns <= 8192 // 128 // 4
    assert 4 * ns <= torch.cuda.get_device_properties(0).multi_processor_count
    # Enough items to fill the GPU: one pass.
    assert attn.attn_fwd_num_splits(4, 32, 8, 8192, 8192, 128) == 1
    assert attn.attn_fwd_num_splits(1, 4, 2, 200, 8192, 256) == 1
    # Short caches against comparable chunks: the combine would cost more.
    assert attn.attn_fwd_num_splits(1, 16, 16, 1024, 1024, 64) == 1
    assert attn.attn_fwd_num_splits(1, 32, 8, 512, 1024, 128) == 1
    # ... but a long cache, or 16+ KV tiles, still splits.
    assert attn.attn_fwd_num_splits(1, 32, 8, 256, 1024, 128) > 1
    assert attn.attn_fwd_num_splits(1, 8, 8, 2048, 2048, 128) > 1
    q, k, v = make_qkv(1, 4, 2, 200, 3000, 128, seed=11)
    o, lse = attn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, num_splits="auto")
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, True, 128 ** -0.5)
    assert_close(o.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "auto")


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D,causal,ns", [
    (1, 8, 2, 128, 1000, 128, True, 1),    # Sq = 128, groups of 4: heads paired per item
    (2, 8, 1, 16, 700, 64, False, 1),      # MQA, a few query rows
    (1, 8, 4, 100, 100, 128, True, 1),     # Sq = Sk
    (1, 8, 2, 77, 2000, 128, True, 4),     # paired heads over KV splits
    (1, 6, 2, 100, 300, 128, True, 1),     # groups of 3: no pairing
])
def test_short_chunks_match_oracle(B, Hq, Hkv, Sq, Sk, D, causal, ns):
    """Sq <= 128 with an even number of query heads per KV group: an item holds
    rows [0,128) of two heads of one group (both tiles have rows)."""
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Sk, D, seed=31 * Sq + Sk + Hq)
    scale = 1.0 / math.sqrt(D)
    o, lse = attn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale,
                           num_splits=ns)
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, scale)
    assert_close(o.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref,
                 f"B{B} Hq{Hq} Hkv{Hkv} Sq{Sq} Sk{Sk} ns{ns}")
