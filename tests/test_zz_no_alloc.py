"""attn_decode_noalloc: the decode entry point for callers that cannot allocate.

Some callers cannot allocate device memory when they call in (a plug-in whose
host framework owns all device memory and hands it no allocator, or a
latency-critical loop that may not call cudaMalloc/cudaFree).  For them the
library offers attn_decode_noalloc, which keeps the split partials in a static
device array instead of caller-supplied workspace.  These tests call it
through the C ABI and check it against the allocating path
(attn_decode_splitkv + attn_combine), within the parity tolerances, on two
calls in a row (the second call runs on the scratch the first one left).
This file is named to be collected last.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import tensor_attn_fwd_gb300 as attn
from attn_inputs import WORKLOADS, make_qkv, workload_inputs

pytestmark = pytest.mark.gpu

O_TOL = 2e-2
LSE_TOL = 1e-3
CAPACITY = 4 * 1024 * 1024  # ATTN_NOALLOC_SCRATCH_FLOATS


def noalloc_fn():
    f = attn.load_library().attn_decode_noalloc
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 6 + [ctypes.c_float, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f


def call_noalloc(q, k, v, num_splits, scale):
    B, Hq, _, D = q.shape
    _, Hkv, Sk, _ = k.shape
    o = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device=q.device)
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=q.device)
    st = noalloc_fn()(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                      B, Hq, Hkv, Sk, D, num_splits, scale,
                      torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK, attn.attn_status_string(st)
    return o, lse


def compare(o1, l1, o2, l2):
    o1, l1, o2, l2 = (x.double().cpu().numpy() for x in (o1, l1, o2, l2))
    assert np.all(np.isfinite(o1))
    fin = np.isfinite(l2)
    assert np.array_equal(np.isfinite(l1), fin)
    assert float(np.max(np.abs(o1 - o2))) <= O_TOL
    if np.any(fin):
        d = np.abs(l1[fin] - l2[fin]) / np.maximum(1.0, np.abs(l2[fin]))
        assert float(d.max()) <= LSE_TOL


def test_noalloc_matches_allocating_decode_two_calls_in_a_row():
    w = WORKLOADS[5]
    cases = [workload_inputs(w) + (w.num_splits, w.scale),
             make_qkv(3, 8, 2, 1, 1000, 64, seed=11) + (5, 1.0 / math.sqrt(64))]
    for q, k, v, ns, scale in cases:
        q, k, v = q.cuda(), k.cuda(), v.cuda()
        ref_o, ref_l = attn.decode(q, k, v, ns, scale)
        o1, l1 = call_noalloc(q, k, v, ns, scale)
        o2, l2 = call_noalloc(q, k, v, ns, scale)   # second call in a row
        torch.cuda.synchronize()
        assert attn.attn_debug_status() == attn.ATTN_OK
        compare(o1, l1, ref_o, ref_l)
        compare(o2, l2, ref_o, ref_l)


def test_noalloc_rejects_requests_beyond_scratch():
    q, k, v = (t.cuda() for t in make_qkv(1, 8, 8, 1, 64, 128, seed=3))
    B, Hq, D = 1, 8, 128
    ns = CAPACITY // (B * Hq * (D + 1)) + 1   # one split too many
    k = torch.zeros((1, 8, ns, 128), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    o = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    st = noalloc_fn()(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                      B, Hq, 8, ns, D, ns, 0.1, torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_ERR_UNSUPPORTED
