"""Calls from several host threads at once, each on its own CUDA stream (the
C ABI releases the GIL through ctypes): forward, decode and backward give the
same results as the same calls made one at a time."""
import math
import threading

import pytest
import torch

import tensor_attn_fwd_gb300 as attn
from attn_inputs import make_qkv

pytestmark = pytest.mark.gpu


def _problem(i):
    q, k, v = (t.cuda() for t in make_qkv(1, 8, 2, 256 + 64 * i, 256 + 64 * i, 128, seed=60 + i))
    g = torch.Generator().manual_seed(70 + i)
    do = torch.randn(q.shape, generator=g).to(torch.bfloat16).cuda()
    return q, k, v, do


def _run(q, k, v, do, stream):
    with torch.cuda.stream(stream):
        o, lse = attn.attn_fwd(q, k, v, causal=True)
        od, ld = attn.decode(q[:, :, -1:].contiguous(), k, v, 3)
        dq, dk, dv = attn.attn_bwd(q, k, v, o, lse, do, causal=True)
    return o, lse, od, ld, dq, dk, dv


def test_concurrent_host_threads():
    probs = [_problem(i) for i in range(4)]
    serial = []
    for pr in probs:
        serial.append(_run(*pr, torch.cuda.current_stream()))
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    results = [None] * len(probs)
    errors = []
    start = threading.Barrier(len(probs))

    def worker(i):
        try:
            s = torch.cuda.Stream()
            start.wait()
            for _ in range(3):
                out = _run(*probs[i], s)
            s.synchronize()
            results[i] = out
        except Exception as exc:  # reported below
            errors.append(exc)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(probs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors
    torch.cuda.synchronize()
    assert attn.attn_debug_status() == attn.ATTN_OK
    for i, (a, b) in enumerate(zip(results, serial)):
        assert a is not None, f"thread {i} did not finish"
        for x, y in zip(a, b):
            assert torch.equal(x, y), f"thread {i}: results differ from the serial run"
