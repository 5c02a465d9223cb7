"""The prefill and decode kernels launch as programmatic dependents: their CTAs
may start while the previous kernel in the stream still runs, and must not
touch global memory before it has completed.  These tests chain calls whose
inputs are the previous call's outputs, with grids smaller than the GPU so
that the dependent CTAs really do start early on idle SMs, and check that the
chained results equal the same chain run with a device synchronisation between
calls (bit for bit) and the oracle's chain (within the parity tolerances)."""
import math

import numpy as np
import pytest
import torch

import oracle
import tensor_attn_fwd_gb300 as attn
from attn_inputs import make_qkv

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D,causal", [(64, False), (128, True), (256, True)])
def test_prefill_chain_reads_previous_output(D, causal):
    # 2 x 4 heads x 384 rows: 16 items (D 64/128) or 24 tiles (D 256), far fewer
    # CTAs than SMs; q of call i+1 is the bf16 O of call i.
    B, H, S, steps = 2, 4, 384, 4
    scale = 1.0 / math.sqrt(D)
    q0, k, v = make_qkv(B, H, H, S, S, D, seed=70 + D)
    qd, kd, vd = q0.cuda(), k.cuda(), v.cuda()

    def chain(sync):
        x = qd
        outs = []
        for _ in range(steps):
            o, lse = attn.attn_fwd_bf16o(x, kd, vd, causal=causal, scale=scale)
            if sync:
                torch.cuda.synchronize()
            outs.append((o, lse))
            x = o
        torch.cuda.synchronize()
        return outs

    ref = chain(sync=True)
    for rep in range(3):
        got = chain(sync=False)
        assert attn.attn_debug_status() == attn.ATTN_OK
        for i, ((o1, l1), (o2, l2)) in enumerate(zip(got, ref)):
            assert torch.equal(o1, o2), f"rep {rep} step {i}: O differs from the synchronised chain"
            assert torch.equal(l1, l2), f"rep {rep} step {i}: LSE differs"

    # the oracle's chain, with O rounded to bf16 between calls as the kernel does
    x = q0
    for i in range(steps):
        o_ref, lse_ref = oracle.attn_fwd(x, k, v, causal, scale)
        o_gpu = ref[i][0].float().cpu().double().numpy()
        err = float(np.max(np.abs(o_gpu - o_ref)))
        # 2e-2, plus the rounding of the bf16 output (2^-8 of its magnitude)
        excess = float(np.max(np.abs(o_gpu - o_ref) - (2e-2 + 2.0 ** -8 * (np.abs(o_ref) + 2e-2))))
        assert excess <= 0.0, f"step {i}: O max-abs error {err:.3e} against the oracle chain"
        dl = np.abs(ref[i][1].cpu().double().numpy() - lse_ref) / np.maximum(1.0, np.abs(lse_ref))
        assert float(dl.max()) <= 1e-3, f"step {i}: LSE error {float(dl.max()):.3e}"
        x = ref[i][0].cpu()  # continue from the GPU's own bf16 O (same bits on both sides)


def test_decode_chain_reads_previous_partials():
    # split kernel i+1 may start while combine i still reads the shared
    # partials workspace; the split kernel must wait before writing it.
    B, Hq, Hkv, Sk, D, ns = 2, 8, 2, 3000, 128, 6
    scale = 1.0 / math.sqrt(D)
    qs = [make_qkv(B, Hq, Hkv, 1, Sk, D, seed=90 + i)[0].cuda() for i in range(4)]
    _, k, v = make_qkv(B, Hq, Hkv, 1, Sk, D, seed=89)
    kd, vd = k.cuda(), v.cuda()
    op = torch.empty((ns, B, Hq, D), device="cuda")
    lp = torch.empty((ns, B, Hq), device="cuda")

    def run(sync):
        outs = []
        for q in qs:
            o, lse = attn.decode(q, kd, vd, ns, scale, workspace=(op, lp))
            if sync:
                torch.cuda.synchronize()
            outs.append((o, lse))
        torch.cuda.synchronize()
        return outs

    ref = run(sync=True)
    for rep in range(3):
        got = run(sync=False)
        assert attn.attn_debug_status() == attn.ATTN_OK
        for i, ((o1, l1), (o2, l2)) in enumerate(zip(got, ref)):
            assert torch.equal(o1, o2) and torch.equal(l1, l2), f"rep {rep} call {i} differs"
    for i, q in enumerate(qs):
        o_ref, lse_ref = oracle.attn_fwd(q.cpu(), k, v, False, scale)
        err = float(np.max(np.abs(ref[i][0].cpu().double().numpy() - o_ref[:, :, 0])))
        assert err <= 2e-2, f"call {i}: O max-abs error {err:.3e}"
