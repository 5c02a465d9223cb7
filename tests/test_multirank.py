"""The bench's multi-rank path (replicas only) on CPU: world_size-2 gloo ranks
exercise the barrier and the max-over-ranks reduction that bench.py uses to
turn per-rank step times into one whole-job figure."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out):
    import sys
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        bench.barrier(True)
        # per-rank "step time": rank r reports 1.5 + r ms
        t = bench.max_over_ranks(1.5 + rank, True, torch.device("cpu"))
        out[rank] = t
        bench.barrier(True)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_single_rank_helpers_are_noops():
    import bench
    bench.barrier(False)
    assert bench.max_over_ranks(3.25, False, torch.device("cpu")) == 3.25
