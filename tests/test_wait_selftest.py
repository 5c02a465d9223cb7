"""Failure detection without a fault: the bounded wait every kernel uses gives
up on an mbarrier that nothing arrives on, records ATTN_ERR_TIMEOUT in the
device status word, and leaves the context usable for the next call."""
import numpy as np
import pytest
import torch

import oracle
import tensor_attn_fwd_gb300 as attn
from attn_inputs import make_qkv

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_ns", [20_000, 10_000_000])
def test_bounded_wait_expires_and_reports(limit_ns):
    assert attn.attn_debug_status() == attn.ATTN_OK
    status, waited = attn.attn_wait_selftest(limit_ns)
    assert status == attn.ATTN_ERR_TIMEOUT
    # The wait lasted at least its limit and gave up soon after it.
    assert limit_ns <= waited < limit_ns + 50_000_000
    # Reading the status cleared it.
    assert attn.attn_debug_status() == attn.ATTN_OK


def test_context_usable_after_timeout():
    status, _ = attn.attn_wait_selftest(1_000_000)
    assert status == attn.ATTN_ERR_TIMEOUT
    q, k, v = make_qkv(1, 2, 2, 200, 200, 64, seed=77)
    o, lse = attn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, True, 64 ** -0.5)
    assert float(np.max(np.abs(o.cpu().double().numpy() - o_ref))) <= 2e-2
    fin = np.isfinite(lse_ref)
    err = np.abs(lse.cpu().double().numpy()[fin] - lse_ref[fin]) / np.maximum(1, np.abs(lse_ref[fin]))
    assert float(np.max(err)) <= 1e-3
