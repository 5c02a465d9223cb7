"""GPU parity of the fused QKV projection + rotary embedding against the fp64
oracle.

Tolerance: the kernel accumulates in fp32 (hidden terms) and rounds each
output to bf16 (relative error <= 2^-9); rotation uses an fp32 (cos, sin)
table (error <= 2^-24).  Each element must satisfy
|out - ref| <= 2^-8 |ref| + 1e-4 rms(ref).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import tensor_attn_fwd_gb300 as attn

pytestmark = pytest.mark.gpu


def _inputs(B, S, hidden, Hq, Hkv, D, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((B, S, hidden), generator=g).to(torch.bfloat16)
    w = (torch.randn(((Hq + 2 * Hkv) * D, hidden), generator=g) / math.sqrt(hidden)).to(torch.bfloat16)
    return x, w


def _check(got, ref, what):
    got = got.double().cpu().numpy()
    assert np.all(np.isfinite(got)), what
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    err = np.abs(got - ref) - (2.0 ** -8 * np.abs(ref) + 1e-4 * rms)
    assert float(err.max()) <= 0.0, f"{what}: worst excess {float(err.max()):.3e}"


def run_case(B, S, hidden, Hq, Hkv, D, style, seed, positions=None, max_pos=None, base=10000.0):
    x, w = _inputs(B, S, hidden, Hq, Hkv, D, seed)
    T = B * S
    if positions is None:
        pos = np.tile(np.arange(S, dtype=np.int32), B)
        max_pos = max_pos or S
        pos_dev = None
    else:
        pos = np.asarray(positions, dtype=np.int32).reshape(T)
        pos_dev = torch.from_numpy(pos).cuda()
    table = attn.attn_rope_table(max_pos, D, base)
    q, k, v = attn.attn_qkv_rope(x.cuda(), w.cuda(), table, Hq, Hkv, positions=pos_dev,
                                 style=style)
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    qr, kr, vr = oracle.qkv_rope(x.reshape(T, hidden), w, pos, Hq, Hkv, D, base=base, style=style)
    # oracle [T, H, D] -> [B, H, S, D]
    for name, got, ref, H in (("q", q, qr, Hq), ("k", k, kr, Hkv), ("v", v, vr, Hkv)):
        ref = ref.reshape(B, S, H, D).transpose(0, 2, 1, 3)
        _check(got, ref, name)


@pytest.mark.parametrize("style", [0, 1])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_qkv_rope_small(D, style):
    run_case(2, 200, 512, 4, 2, D, style, seed=D + style)


def test_qkv_rope_ragged_sizes():
    # T = 3*77 (not a multiple of 128), hidden 200 (not a multiple of 64),
    # N = (3 + 2) * 64 = 320 (not a multiple of 256).
    run_case(3, 77, 200, 3, 1, 64, 0, seed=11)
    run_case(1, 1, 8, 1, 1, 128, 1, seed=12)
    # CTA-pair form (T >= 512): T = 700 (2 x 256 + 188), hidden 200, N = 320.
    run_case(1, 700, 200, 3, 1, 64, 1, seed=13)
    # hidden 64: the second 64-wide box of every K = 128 stage lies wholly past
    # hidden and must arrive as zeros.
    run_case(2, 300, 64, 2, 1, 128, 0, seed=14)


def test_qkv_rope_positions_and_gqa():
    B, S = 2, 300
    g = torch.Generator().manual_seed(13)
    pos = torch.randint(0, 32768, (B, S), generator=g, dtype=torch.int32).numpy()
    run_case(B, S, 256, 8, 1, 128, 1, seed=14, positions=pos, max_pos=32768, base=500000.0)


def test_rope_table_values():
    max_pos, D, base = 9000, 128, 10000.0
    t = attn.attn_rope_table(max_pos, D, base).cpu().double().numpy()
    i = np.arange(D // 2, dtype=np.float64)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * base ** (-2.0 * i / D)[None, :]
    np.testing.assert_allclose(t[..., 0], np.cos(ang), rtol=0, atol=1.2e-7)
    np.testing.assert_allclose(t[..., 1], np.sin(ang), rtol=0, atol=1.2e-7)


def test_position_out_of_range_reported():
    B, S, hidden, Hq, Hkv, D = 1, 64, 64, 2, 1, 64
    x, w = _inputs(B, S, hidden, Hq, Hkv, D, seed=15)
    table = attn.attn_rope_table(64, D)
    pos = torch.arange(S, dtype=torch.int32).cuda()
    pos[5] = 64
    attn.attn_qkv_rope(x.cuda(), w.cuda(), table, Hq, Hkv, positions=pos)
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_debug_status() == attn.ATTN_OK


def test_qkv_rope_llama_shape_sampled():
    """B2 S8192 hidden 4096, Hq32 Hkv8 D128 (the projection in front of the
    causal GQA prefill workload), on sampled tokens."""
    B, S, hidden, Hq, Hkv, D = 2, 8192, 4096, 32, 8, 128
    x, w = _inputs(B, S, hidden, Hq, Hkv, D, seed=16)
    table = attn.attn_rope_table(S, D)
    q, k, v = attn.attn_qkv_rope(x.cuda(), w.cuda(), table, Hq, Hkv, style=0)
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    T = B * S
    g = torch.Generator().manual_seed(17)
    toks = torch.unique(torch.cat([torch.tensor([0, 1, 127, 128, S - 1, S, T - 1]),
                                   torch.randint(0, T, (40,), generator=g)])).numpy()
    pos = np.tile(np.arange(S, dtype=np.int32), B)
    qr, kr, vr = oracle.qkv_rope(x.reshape(T, hidden), w, pos, Hq, Hkv, D, style=0, tokens=toks)
    b, s = toks // S, toks % S
    for name, got, ref in (("q", q, qr), ("k", k, kr), ("v", v, vr)):
        sel = got[torch.from_numpy(b).cuda(), :, torch.from_numpy(s).cuda()]   # [n, H, D]
        _check(sel, ref, name)
