"""The sm_103a microbenchmarks: they build without a GPU, and on a GB300 they
report the rates the kernels' design relies on (one 128x128x16 MMA per ~64
cycles, twice that at N = 256; the prefill MMA warp's step sequence above its
2048 MMA cycles; TMEM load/store bandwidth; a TMA stage ring that streams HBM
near the copy bandwidth and L2 well above it)."""
import os
import subprocess

import pytest

from tensor_attn_fwd_gb300 import microbench


def test_microbench_compiles(tmp_path):
    out = str(tmp_path / "mb")
    subprocess.run(microbench.nvcc_command(out), check=True)
    assert os.path.getsize(out) > 0


@pytest.mark.gpu
def test_microbench_rates():
    recs = microbench.run()
    assert not any("error" in r for r in recs), recs
    mma = {r["shape"]: r["cycles_per_mma"] for r in recs if r["bench"] == "mma_cycles"}
    assert 50 <= mma["SS M128 N128 K16"] <= 90
    assert 100 <= mma["SS M128 N256 K16"] <= 180
    assert 50 <= mma["TS M128 N128 K16"] <= 90
    # M = 64 does a quarter of the N = 256, M = 128 work but takes longer than half
    assert 64 <= mma["SS M64 N256 K16"] <= 300
    # N = 64: half the N = 128 time with A in TMEM; with both operands in shared
    # memory the 6 KB of operands per MMA take longer than the tensor work
    assert 25 <= mma["TS M128 N64 K16"] <= 50
    assert mma["TS M128 N64 K16"] < mma["SS M128 N64 K16"] <= 80
    (wait,) = [r for r in recs if r["bench"] == "wait_latency"]
    assert 5 <= wait["cycles_per_try_wait"] <= 500
    (step,) = [r for r in recs if r["bench"] == "step_sequence"]
    assert 2000 <= step["cycles_per_step"] <= 4000
    assert step["cycles_per_step_waits_x4"] > step["cycles_per_step"]
    (ex2,) = [r for r in recs if r["bench"] == "ex2_rate"]
    assert ex2["results_per_clock_per_sm"] > 0
    tmem = {(r["op"].split()[0], r["warps"]): r["bytes_per_clock_per_sm"]
            for r in recs if r["bench"] == "tmem_bw"}
    assert set(tmem) == {("ld", 4), ("st", 4), ("ld", 8), ("st", 8)}
    # 128 lanes x 4 bytes = 512 bytes per TMEM column: a softmax row pass of
    # 128 columns must take far fewer cycles than the 2048-cycle MMA step
    assert all(100 <= v <= 4096 for v in tmem.values()), tmem
    assert tmem[("ld", 8)] >= tmem[("ld", 4)]
    ring = {r["source"]: r["gb_per_s"] for r in recs if r["bench"] == "tma_ring_bw"}
    assert 3000 <= ring["hbm"] <= 9000, ring   # measured copy peak ~6.7 TB/s
    assert ring["l2"] > ring["hbm"], ring
