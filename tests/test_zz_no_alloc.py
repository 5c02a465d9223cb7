"""attn_decode_noalloc: the decode entry point for callers that cannot allocate.

Some callers cannot allocate device memory when they call in (a plug-in whose
host framework owns all device memory and hands it no allocator, or a
latency-critical loop that may not call cudaMalloc/cudaFree).  For them the
library offers attn_decode_noalloc, which keeps the split partials in a static
device array instead of caller-supplied workspace.  These tests call it
through the C ABI and check it against the fp64 oracle and against the
allocating path (attn_decode_splitkv + attn_combine), within the parity
tolerances, on two calls in a row (the second call runs on the scratch the
first one left).  The cases cover D = 64, 128 and 256, more than 32 splits
(the combine's outer loop over groups of 32), partials that fill the scratch
array to within one split (the LSE partials at its far end), and a small call
right after a large one (no stale partial may leak in).
This file is named to be collected last.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
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


def compare(o1, l1, o2, l2, what):
    o1, l1 = (x.double().cpu().numpy() if torch.is_tensor(x) else x for x in (o1, l1))
    o2, l2 = (x.double().cpu().numpy() if torch.is_tensor(x) else x for x in (o2, l2))
    assert np.all(np.isfinite(o1)), f"{what}: non-finite O"
    fin = np.isfinite(l2)
    assert np.array_equal(np.isfinite(l1), fin), f"{what}: -inf pattern differs"
    err = float(np.max(np.abs(o1 - o2)))
    assert err <= O_TOL, f"{what}: O max-abs error {err:.3e}"
    if np.any(fin):
        d = np.abs(l1[fin] - l2[fin]) / np.maximum(1.0, np.abs(l2[fin]))
        assert float(d.max()) <= LSE_TOL, f"{what}: LSE error {float(d.max()):.3e}"


def near_capacity_case():
    # B=4, Hq=32, D=128: one split's partials are 4*32*(128+1) = 16512 floats;
    # 254 splits take 4,194,048 of the 4,194,304 floats (256 to spare, less
    # than one split), so the LSE partials sit at the far end of the array.
    B, Hq, Hkv, D = 4, 32, 8, 128
    ns = CAPACITY // (B * Hq * (D + 1))
    assert ns == 254 and CAPACITY - ns * B * Hq * (D + 1) < B * Hq * (D + 1)
    return make_qkv(B, Hq, Hkv, 1, 8192, D, seed=254) + (ns, 1.0 / math.sqrt(D))


def cases():
    w = WORKLOADS[5]
    return [
        ("near capacity, 254 splits", near_capacity_case()),
        ("workload 5 (D=128, 8 splits)", workload_inputs(w) + (w.num_splits, w.scale)),
        ("D=256, 40 splits", make_qkv(2, 16, 4, 1, 3000, 256, seed=256) + (40, 1.0 / 16.0)),
        ("D=64, 5 splits, small after large", make_qkv(3, 8, 2, 1, 1000, 64, seed=11)
         + (5, 1.0 / math.sqrt(64))),
    ]


def test_noalloc_matches_oracle_and_allocating_decode_two_calls_in_a_row():
    # The largest case runs first and fills the scratch array; every later,
    # smaller case must read only the partials it wrote itself.
    for what, (q, k, v, ns, scale) in cases():
        o_ref, lse_ref = oracle.attn_fwd(q, k, v, False, scale)
        o_ref, lse_ref = o_ref[:, :, 0], lse_ref[:, :, 0]
        q, k, v = q.cuda(), k.cuda(), v.cuda()
        o1, l1 = call_noalloc(q, k, v, ns, scale)
        o2, l2 = call_noalloc(q, k, v, ns, scale)   # second call in a row
        ref_o, ref_l = attn.decode(q, k, v, ns, scale)
        torch.cuda.synchronize()
        assert attn.attn_debug_status() == attn.ATTN_OK
        for o, l, n in ((o1, l1, "first call"), (o2, l2, "second call")):
            compare(o, l, o_ref, lse_ref, f"{what}, {n} vs oracle")
            compare(o, l, ref_o, ref_l, f"{what}, {n} vs allocating decode")


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
