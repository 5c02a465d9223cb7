"""Microbenchmarks of the sm_103a mechanisms the kernels are designed around.

``run()`` compiles ``mb.cu`` (nvcc, sm_103a) next to this file on first use,
runs it on the current GPU and returns its measurements as dicts:

- ``mma_cycles``: cycles per tcgen05.mma (bf16 -> fp32) for M128 N128 / N256
  K16 in SS form, M128 N128 in TS form, M64 N256 in SS form and M128 N64 in
  both forms, issued back to back by one warp.
- ``wait_latency``: cycles of a dependent mbarrier.try_wait on a completed phase.
- ``step_sequence``: cycles per KV step of the prefill MMA warp's issue
  sequence (32 MMAs, 5 waits, 4 commits) with every barrier complete, with each
  wait repeated four times, and the cost of one extra wait between MMA issues.
- ``ex2_rate``: ex2.approx.f32 results per clock per SM.
- ``tmem_bw``: bytes per clock per SM moved by tcgen05.ld / tcgen05.st
  (32x32b shapes) with 4 and with 8 warps per CTA.
- ``tma_ring_bw``: GB/s of a TMA producer feeding a 6-stage ring of 32 KB
  stages (two 128 x 64 bf16 boxes, 128B swizzle) whose consumer only releases
  them: streamed from HBM (1 GiB) and re-read from L2 (38 MiB).

``python -m tensor_attn_fwd_gb300.microbench`` prints them as JSON lines.
"""
import json
import os
import subprocess

_DIR = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_DIR, "mb.cu")
_EXE = os.path.join(_DIR, "mb")


def nvcc_command(out: str = _EXE) -> list:
    return ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
            "-lineinfo", "-o", out, _SRC]


def build(force: bool = False) -> str:
    if force or not os.path.exists(_EXE) or os.path.getmtime(_EXE) < os.path.getmtime(_SRC):
        subprocess.run(nvcc_command(), check=True)
    return _EXE


def run() -> list:
    exe = build()
    res = subprocess.run([exe], check=True, capture_output=True, text=True)
    return [json.loads(line) for line in res.stdout.splitlines() if line.strip()]
