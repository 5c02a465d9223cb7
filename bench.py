"""Benchmark of the attention forward (prefill) and split-KV decode on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One JSON line is printed by rank 0.  ``value`` is the prefill throughput in
TFLOP/s (counted FLOPs 4*B*Hq*Sq*Sk*D, halved for causal) on the causal GQA
workload B=2, Hq=32, Hkv=8, S=8192, D=128; a step is one attn_fwd launch with
its inputs resident in HBM.  L2 is flushed between steps by writing a 256 MiB
buffer outside the timed events.  The ``decode`` object reports the split-KV
decode + combine (B=64, Hq=32, Hkv=8, Sk=4096, D=128, 8 splits) in GB/s of
algorithmic bytes.  ``backward`` times attn_bwd on the prefill workload
(TFLOP/s at 2.5x the forward's FLOPs) and ``qkv_rope`` the fused QKV
projection + RoPE that produces that workload's Q, K, V from hidden states of
width 4096 (TFLOP/s at 2*T*hidden*N).  ``e2e`` repeats the prefill through the
public API with pinned host buffers, the host<->device copies inside the timed
region.

The ``configs`` object reports each of the five workloads (1-5): its GPU time
(workloads 1 and 2 from a replayed CUDA graph of 50 launches, since a single
launch is shorter than the host's call), throughput against the roofline, and
the max O / LSE error of the timed run's own output against the fp64 CPU
oracle on the same seeded inputs, every query row by default (``--parity
sample`` checks the documented row sample of workloads 3 and 4 instead).  The
oracle's run on workload 3 doubles as the ``cpu_baseline``.  The process exits
with status 3 after printing if any output misses the tolerances.

--impl reference times the fp64 CPU oracle on the same workload (a bounded
sample of query rows per step) and prints the same line with impl=reference.
Multi-GPU (torchrun): every rank runs its own replica (replicas only, no
collective on the data path); value = total FLOPs of all ranks / max time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from attn_inputs import WORKLOADS, sample_rows, workload_inputs  # noqa: E402

METRIC = "attn fwd TFLOP/s & % BF16 TC peak (prefill); decode HBM GB/s & % of peak"
PREFILL = WORKLOADS[3]
DECODE = WORKLOADS[5]
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# DRAM bytes (read + write) per launch of each kernel on the workloads above,
# from `ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum` (one pass) of
# `bench.py --profile prefill|decode`; profiles/ holds the summary.  Reset to
# None whenever the kernel changes until it is captured again.
PREFILL_TRAFFIC_BYTES = 319545344 + 214419968
DECODE_TRAFFIC_BYTES = 1074342656 + 11164928


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while work runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu_index), "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.t is not None:
            self.t.join(timeout=2)

    def summary(self, t0=None, t1=None):
        rows = []
        for ts, line in self.lines:
            if (t0 is not None and ts < t0) or (t1 is not None and ts > t1):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"],
                    "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, _, flags in rows for i, f in enumerate(flags)
                          if f.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def flush_l2(buf):
    if buf is not None:
        buf.add_(1)


def time_launches(fn, steps, warmup, flush_buf, stream):
    """Per-step CUDA-event times (ms) of fn() on `stream`; L2 is flushed in
    between unless flush_buf is None (inputs larger than L2)."""
    for _ in range(warmup):
        flush_l2(flush_buf)
        fn()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush_l2(flush_buf)
        starts[i].record(stream)
        fn()
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def barrier(dist_on):
    if dist_on:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, dist_on: bool, device) -> float:
    if not dist_on:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def oracle_rows_flops(w, rows):
    """Counted FLOPs (4*D per visible key) of a set of flat row ids."""
    i = rows % w.Sq
    if w.causal:
        nvis = torch.clamp(i + w.Sk - w.Sq + 1, 0, w.Sk)
    else:
        nvis = torch.full_like(i, w.Sk)
    return float(4.0 * w.D * nvis.double().sum())


def run_oracle_sample(w, q, k, v, target_s: float, seed: int = 0):
    """Time the oracle on a row sample sized to take about target_s seconds."""
    import oracle  # CPU baseline only
    n = 64
    while True:
        rows = sample_rows(w.B, w.Hq, w.Sq, n_random=n, seed=seed)
        t0 = time.perf_counter()
        oracle.attn_fwd(q, k, v, w.causal, w.scale, rows=rows.numpy())
        dt = time.perf_counter() - t0
        if dt >= target_s or n >= w.B * w.Hq * w.Sq:
            return rows, dt
        n = min(int(n * max(2.0, 1.2 * target_s / max(dt, 1e-3))), w.B * w.Hq * w.Sq)


def omp_threads() -> int:
    env = os.environ.get("OMP_NUM_THREADS")
    if env and env.isdigit():
        return int(env)
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_model() -> str:
    """Host CPU model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


O_TOL = 2e-2    # max |O_gpu - O_ref|
LSE_TOL = 1e-3  # |LSE_gpu - LSE_ref| / max(1, |LSE_ref|)


def parity_errors(o_gpu, lse_gpu, o_ref, lse_ref):
    """Max O error and LSE error of a GPU result against the oracle's, and
    whether they meet the tolerances (rows with no visible key must be O = 0,
    LSE = -inf on both sides)."""
    import numpy as np
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    lse_ref = np.asarray(lse_ref, dtype=np.float64)
    fin = np.isfinite(lse_ref)
    pattern = bool(np.array_equal(np.isfinite(lse_gpu), fin) and np.all(lse_gpu[~fin] == -np.inf))
    finite_o = bool(np.all(np.isfinite(o_gpu)))
    err_o = float(np.max(np.abs(o_gpu - o_ref))) if o_gpu.size else 0.0
    err_l = 0.0
    if np.any(fin) and pattern:
        err_l = float(np.max(np.abs(lse_gpu[fin] - lse_ref[fin])
                             / np.maximum(1.0, np.abs(lse_ref[fin]))))
    ok = pattern and finite_o and err_o <= O_TOL and err_l <= LSE_TOL
    return {"o_max_abs_err": err_o, "lse_max_err": err_l, "pass": bool(ok),
            "tol": f"O max-abs <= {O_TOL}; LSE |d|/max(1,|ref|) <= {LSE_TOL}"}


def graph_launch_ms(fn, launches=50, reps=7):
    """GPU time of one fn() launch: a CUDA graph of `launches` calls replayed
    `reps` times, CUDA events around each replay; the median per launch."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=side):
        for _ in range(launches):
            fn()
    g.replay()
    torch.cuda.synchronize()
    per = []
    for _ in range(reps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        per.append(a.elapsed_time(b) / launches)
    del g
    return statistics.median(per)


def workload_config(w, extra=None):
    cfg = {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq, "Sk": w.Sk,
           "D": w.D, "causal": w.causal, "inputs": "bf16 N(0,1) Q/K/V from seed %d" % w.seed,
           "parallelism": "replicas"}
    if extra:
        cfg.update(extra)
    return cfg


def prefill_config(w):
    """The headline workload's config, the same dict on both arms (the L2
    statement describes how the GPU arm keeps the steps cold)."""
    return workload_config(w, {"l2": "flushed between steps (256 MiB write outside "
                                     "the timed events); inputs+outputs 472 MB > L2"})


def reference_arm(args, rank, world):
    """The fp64 CPU oracle as the reference arm (rank 0 only)."""
    if rank != 0:
        return
    w = PREFILL
    q, k, v = workload_inputs(w)
    total = args.steps + args.warmup
    per_step = max(0.5, min(10.0, 90.0 / max(1, total)))
    rows, _ = run_oracle_sample(w, q, k, v, per_step, seed=w.seed)
    import oracle
    flops = oracle_rows_flops(w, rows)
    for _ in range(args.warmup):
        oracle.attn_fwd(q, k, v, w.causal, w.scale, rows=rows.numpy())
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.attn_fwd(q, k, v, w.causal, w.scale, rows=rows.numpy())
        times.append(time.perf_counter() - t0)
    sec = sum(times) / len(times)
    value = flops / sec / 1e12
    sample = f"{rows.numel()} query rows of the workload per step ({flops / 1e9:.1f} GFLOP counted)"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": prefill_config(w),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": omp_threads(),
                             "cpu_model": cpu_model(), "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def ours_arm(args, rank, world, local_rank, dist_on):
    import tensor_attn_fwd_gb300 as attn
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    stream = torch.cuda.current_stream()
    peaks, peaks_src = load_peaks()
    sampler = ClockSampler(local_rank)
    sampler.start()

    flush_buf = torch.zeros(64 * 1024 * 1024, dtype=torch.float32, device=device)  # 256 MiB

    # ---------------- prefill (value)
    w = PREFILL
    q_h, k_h, v_h = workload_inputs(w)
    q, k, v = q_h.to(device), k_h.to(device), v_h.to(device)
    o = torch.empty((w.B, w.Hq, w.Sq, w.D), dtype=torch.float32, device=device)
    lse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=device)

    def prefill():
        attn.attn_fwd(q, k, v, causal=w.causal, scale=w.scale, o=o, lse=lse, stream=stream)

    prefill()
    torch.cuda.synchronize()
    if attn.attn_debug_status() != attn.ATTN_OK:
        raise RuntimeError("prefill kernel reported a timeout")
    barrier(dist_on)
    torch.cuda.synchronize()
    t_clock0 = time.time()
    times = time_launches(prefill, args.steps, args.warmup, flush_buf, stream)
    torch.cuda.synchronize()
    barrier(dist_on)
    t_clock1 = time.time()
    # The timed launches' own output, checked against the oracle below.
    c3_out = (o.cpu(), lse.cpu())
    ms = sum(times) / len(times)
    ms_max = max_over_ranks(ms, dist_on, device)
    flops = w.flops()
    value = flops * world / (ms_max * 1e-3) / 1e12
    achieved = flops / (ms * 1e-3) / 1e12
    # The same launches back to back (no flush: Q+K+V alone exceed L2).  Without
    # the flush's gaps the GPU runs at its power cap, the regime of the measured
    # sustained peak.
    times_bb = time_launches(prefill, args.steps, 3, None, stream)
    ms_bb = sum(times_bb) / len(times_bb)
    back_to_back = {"value": flops / (ms_bb * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "ms_per_step": ms_bb, "steps": len(times_bb),
                    "peak": peaks["bf16_tflops_sustained"],
                    "frac": flops / (ms_bb * 1e-3) / 1e12 / peaks["bf16_tflops_sustained"],
                    "peak_source": f"{peaks_src} cuBLAS bf16 sustained (4 s back to back)",
                    "l2": "no flush: Q+K+V 201 MB > L2"}

    # ---------------- decode (split-KV + combine)
    d = DECODE
    dq_h, dk_h, dv_h = workload_inputs(d)
    dq, dk, dv = dq_h.to(device), dk_h.to(device), dv_h.to(device)
    op = torch.empty((d.num_splits, d.B, d.Hq, d.D), dtype=torch.float32, device=device)
    lp = torch.empty((d.num_splits, d.B, d.Hq), dtype=torch.float32, device=device)
    do = torch.empty((d.B, d.Hq, d.D), dtype=torch.float32, device=device)
    dl = torch.empty((d.B, d.Hq), dtype=torch.float32, device=device)

    def decode_split():
        attn.attn_decode_splitkv(dq, dk, dv, d.num_splits, d.scale, op, lp, stream=stream)

    def decode_combine():
        attn.attn_combine(op, lp, do, dl, stream=stream)

    def decode_both():
        decode_split()
        decode_combine()

    fo = torch.empty_like(do)
    fl = torch.empty_like(dl)
    fop = torch.empty_like(op)
    flp = torch.empty_like(lp)
    fcnt = torch.zeros(d.B * d.Hkv * ((d.Hq // d.Hkv + 15) // 16), dtype=torch.int32,
                       device=device)

    def decode_fused():  # the same decode with the combine in the split kernel
        attn.attn_decode_fused(dq, dk, dv, d.num_splits, d.scale, o_part=fop, lse_part=flp,
                               o=fo, lse=fl, counters=fcnt, stream=stream)

    decode_both()
    decode_fused()
    torch.cuda.synchronize()
    # K+V (1.07 GB) exceed L2 eightfold: no flush between decode steps (a flush
    # would leave dirty lines whose write-back competes with the K/V stream).
    t_both = time_launches(decode_both, args.steps, args.warmup, None, stream)
    t_split = time_launches(decode_split, args.steps, args.warmup, None, stream)
    t_comb = time_launches(decode_combine, args.steps, args.warmup, None, stream)
    t_fused = time_launches(decode_fused, args.steps, args.warmup, None, stream)
    t_clock2 = time.time()
    c5_out = (op.cpu(), lp.cpu(), do.cpu(), dl.cpu())
    dbytes = d.algorithmic_bytes()
    d_ms = sum(t_both) / len(t_both)
    d_split_ms = sum(t_split) / len(t_split)
    decode = {
        "workload": d.name, "metric": "decode HBM GB/s (algorithmic bytes)",
        "l2": "no flush: K+V 1.07 GB > L2",
        "value": dbytes / (d_ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": d_ms,
        "split_kernel_ms": d_split_ms, "combine_kernel_ms": sum(t_comb) / len(t_comb),
        "fused_one_launch_ms": sum(t_fused) / len(t_fused),
        "fused_equals_two_launches": bool(torch.equal(fo, do) and torch.equal(fl, dl)),
        "algorithmic_bytes": dbytes,
        "frac_of_measured_hbm": dbytes / (d_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
        "frac_of_nominal_8tbs": dbytes / (d_ms * 1e-3) / 1e9 / 8000.0,
        "roofline": {"bound": "hbm", "achieved": dbytes / (d_split_ms * 1e-3) / 1e9,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": dbytes / (d_split_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                     "traffic": DECODE_TRAFFIC_BYTES,
                     "peak_source": f"{peaks_src} STREAM-style copy"},
    }

    # ---------------- backward on the prefill workload (Delta + dK/dV + dQ kernels)
    backward = None
    if not args.no_backward:
        g = torch.Generator().manual_seed(w.seed + 7)
        dout = torch.randn(q.shape, generator=g).to(torch.bfloat16).to(device)
        dq = torch.empty(q.shape, dtype=torch.float32, device=device)
        dk = torch.empty(k.shape, dtype=torch.float32, device=device)
        dv = torch.empty(v.shape, dtype=torch.float32, device=device)
        dws = torch.empty(lse.shape, dtype=torch.float32, device=device)
        prefill()

        def bwd():
            attn.attn_bwd(q, k, v, o, lse, dout, causal=w.causal, scale=w.scale, dq=dq, dk=dk,
                          dv=dv, delta_ws=dws, stream=stream)

        b_steps = max(3, min(args.steps, 50))
        b_times = time_launches(bwd, b_steps, 3, flush_buf, stream)
        b_ms = sum(b_times) / len(b_times)
        b_flops = 2.5 * flops  # five GEMM-sized products against the forward's two
        backward = {"workload": w.name, "metric": "attn bwd TFLOP/s (2.5x forward FLOPs)",
                    "value": b_flops / (b_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "ms_per_step": b_ms, "steps": b_steps,
                    "frac_of_measured_bf16_peak": b_flops / (b_ms * 1e-3) / 1e12
                    / peaks["bf16_tflops"],
                    "gpu_launches_per_step": 3}
        del dq, dk, dv, dws, dout

    # ---------------- QKV projection + RoPE producing this workload's Q, K, V
    qkv_rope = None
    if not args.no_qkv_rope:
        hidden = 4096  # Llama-family model width for 32 query heads of 128
        g = torch.Generator().manual_seed(w.seed + 11)
        xq = torch.randn((w.B, w.Sq, hidden), generator=g).to(torch.bfloat16).to(device)
        wq = (torch.randn(((w.Hq + 2 * w.Hkv) * w.D, hidden), generator=g)
              / math.sqrt(hidden)).to(torch.bfloat16).to(device)
        table = attn.attn_rope_table(w.Sq, w.D, 10000.0)
        qo = torch.empty(q.shape, dtype=torch.bfloat16, device=device)
        ko = torch.empty(k.shape, dtype=torch.bfloat16, device=device)
        vo = torch.empty(v.shape, dtype=torch.bfloat16, device=device)

        def qkv():
            attn.attn_qkv_rope(xq, wq, table, w.Hq, w.Hkv, q=qo, k=ko, v=vo, stream=stream)

        r_steps = max(3, min(args.steps, 50))
        r_times = time_launches(qkv, r_steps, 3, flush_buf, stream)
        r_ms = sum(r_times) / len(r_times)
        r_flops = 2.0 * w.B * w.Sq * hidden * (w.Hq + 2 * w.Hkv) * w.D
        qkv_rope = {"workload": f"x [{w.B},{w.Sq},{hidden}] bf16 -> RoPE(x W^T) as Q,K,V of "
                                f"{w.name}",
                    "metric": "QKV projection + RoPE TFLOP/s (2*T*hidden*N)",
                    "value": r_flops / (r_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "ms_per_step": r_ms, "steps": r_steps,
                    "frac_of_measured_bf16_peak": r_flops / (r_ms * 1e-3) / 1e12
                    / peaks["bf16_tflops"],
                    "gpu_launches_per_step": 1}
        del xq, wq, table, qo, ko, vo

    # ---------------- end to end through the public API, host buffers
    # Every step copies its inputs from pinned host memory, runs attn_fwd and
    # copies O and LSE back to pinned host memory.  Steps are pipelined the way
    # a serving loop would run them: host->device copies, compute and
    # device->host copies on three streams, with two device buffer sets, so the
    # copies of one step overlap the compute of its neighbours.  The timed
    # region spans all K steps (first copy in to last copy out).
    e2e = None
    if not args.no_e2e:
        qp, kp, vp = q_h.pin_memory(), k_h.pin_memory(), v_h.pin_memory()
        op_h = torch.empty(o.shape, dtype=torch.float32).pin_memory()
        lp_h = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
        sets = [tuple(torch.empty_like(t, device=device) for t in (q, k, v))
                + (torch.empty_like(o), torch.empty_like(lse)) for _ in range(2)]
        s_in, s_cmp, s_out = (torch.cuda.Stream(device) for _ in range(3))

        def e2e_run(steps):
            ev_in = [torch.cuda.Event() for _ in range(steps)]
            ev_cmp = [torch.cuda.Event() for _ in range(steps)]
            ev_out = [torch.cuda.Event() for _ in range(steps)]
            for i in range(steps):
                qd, kd, vd, od, ld = sets[i % 2]
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(ev_cmp[i - 2])  # set i%2 inputs are free
                    qd.copy_(qp, non_blocking=True)
                    kd.copy_(kp, non_blocking=True)
                    vd.copy_(vp, non_blocking=True)
                    ev_in[i].record(s_in)
                s_cmp.wait_event(ev_in[i])
                if i >= 2:
                    s_cmp.wait_event(ev_out[i - 2])  # set i%2 outputs are read back
                attn.attn_fwd(qd, kd, vd, causal=w.causal, scale=w.scale, o=od, lse=ld,
                              stream=s_cmp)
                ev_cmp[i].record(s_cmp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_cmp[i])
                    op_h.copy_(od, non_blocking=True)
                    lp_h.copy_(ld, non_blocking=True)
                    ev_out[i].record(s_out)
            return ev_out[-1]

        # The host link's own rates on this machine, for reading the e2e number: one
        # timed copy of the step's inputs in and of its outputs back, each alone.
        def link_gbs(copy, nbytes):
            copy()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s_in)
            copy()
            b.record(s_in)
            torch.cuda.synchronize()
            return nbytes / (a.elapsed_time(b) * 1e-3) / 1e9

        def copy_in():
            with torch.cuda.stream(s_in):
                sets[0][0].copy_(qp, non_blocking=True)
                sets[0][1].copy_(kp, non_blocking=True)
                sets[0][2].copy_(vp, non_blocking=True)

        def copy_out():
            with torch.cuda.stream(s_in):
                op_h.copy_(sets[0][3], non_blocking=True)
                lp_h.copy_(sets[0][4], non_blocking=True)

        link = {"h2d_gbs": link_gbs(copy_in, sum(t.numel() * t.element_size() for t in (qp, kp, vp))),
                "d2h_gbs": link_gbs(copy_out, op_h.numel() * 4 + lp_h.numel() * 4)}
        e_steps = max(4, min(args.steps, 20))
        e2e_run(3)  # warm-up
        torch.cuda.synchronize()
        barrier(dist_on)
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(s_in)
        s_cmp.wait_stream(s_in)
        s_out.wait_stream(s_in)
        last = e2e_run(e_steps)
        s_in.wait_event(last)
        t_end.record(s_in)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(t_start.elapsed_time(t_end) / e_steps, dist_on, device)
        h2d = sum(t.numel() * t.element_size() for t in (qp, kp, vp))
        d2h = op_h.numel() * 4 + lp_h.numel() * 4
        e2e = {"value": flops * world / (e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "ms_per_step": e_ms, "steps": e_steps, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "host_link": link,
               "method": "pinned host buffers; H2D, attn_fwd and D2H on three streams, "
                         "two device buffer sets, timed from the first copy in to the "
                         "last copy out; host_link: one copy in and one out, each alone"}
        del sets
    # ---------------- the other workloads (1, 2, 4): GPU time and output
    cfg_runs = {}
    for ci in (1, 2, 4):
        cw = WORKLOADS[ci]
        cq_h, ck_h, cv_h = workload_inputs(cw)
        cq, ck, cv = cq_h.to(device), ck_h.to(device), cv_h.to(device)
        co = torch.empty((cw.B, cw.Hq, cw.Sq, cw.D), dtype=torch.float32, device=device)
        cl = torch.empty((cw.B, cw.Hq, cw.Sq), dtype=torch.float32, device=device)

        def cfn(cq=cq, ck=ck, cv=cv, co=co, cl=cl, cw=cw):
            attn.attn_fwd(cq, ck, cv, causal=cw.causal, scale=cw.scale, o=co, lse=cl)

        if ci in (1, 2):
            # A launch is shorter than the host's call: replay a graph of 50.
            # Inputs and outputs (<= 42 MB) stay in L2 between launches.
            c_ms = graph_launch_ms(cfn)
            timing = "CUDA graph of 50 launches, median of 7 replays (L2 warm: inputs fit)"
        else:
            c_times = time_launches(cfn, max(3, min(args.steps, 100)), 3, flush_buf, stream)
            c_ms = sum(c_times) / len(c_times)
            timing = f"CUDA events, mean of {len(c_times)} launches, L2 flushed between"
        torch.cuda.synchronize()
        if attn.attn_debug_status() != attn.ATTN_OK:
            raise RuntimeError(f"{cw.name}: kernel reported a timeout")
        cfg_runs[ci] = {"ms": c_ms, "timing": timing, "out": (co.cpu(), cl.cpu()),
                        "inputs": (cq_h, ck_h, cv_h)}
        del cq, ck, cv, co, cl
    cfg_runs[3] = {"ms": ms, "timing": "the value's launches (CUDA events, L2 flushed between)",
                   "out": c3_out, "inputs": (q_h, k_h, v_h)}
    sampler.stop()
    clocks = sampler.summary(t_clock0, t_clock2)

    if rank != 0:
        return

    # ---------------- parity of every timed output against the fp64 oracle
    import oracle  # test infrastructure: the check, never the product path
    per_workload = {}
    cpu = None
    parity_ok = True
    for ci in (1, 2, 3, 4):
        cw = WORKLOADS[ci]
        run = cfg_runs[ci]
        cq_h, ck_h, cv_h = run["inputs"]
        o_gpu, l_gpu = run["out"]
        total_rows = cw.B * cw.Hq * cw.Sq
        if args.parity == "sample" and ci in (3, 4):
            rows = sample_rows(cw.B, cw.Hq, cw.Sq, n_random=256, seed=cw.seed)
            t0 = time.perf_counter()
            o_ref, l_ref = oracle.attn_fwd(cq_h, ck_h, cv_h, cw.causal, cw.scale,
                                           rows=rows.numpy())
            o_dt = time.perf_counter() - t0
            o_cmp = o_gpu.reshape(-1, cw.D)[rows].numpy()
            l_cmp = l_gpu.reshape(-1)[rows].numpy()
            n_rows, row_flops = rows.numel(), oracle_rows_flops(cw, rows)
        else:
            t0 = time.perf_counter()
            o_ref, l_ref = oracle.attn_fwd(cq_h, ck_h, cv_h, cw.causal, cw.scale)
            o_dt = time.perf_counter() - t0
            o_cmp, l_cmp = o_gpu.numpy(), l_gpu.numpy()
            n_rows, row_flops = total_rows, cw.flops()
        par = parity_errors(o_cmp, l_cmp, o_ref, l_ref)
        par.update({"rows": n_rows, "rows_total": total_rows, "oracle_s": o_dt})
        parity_ok &= par["pass"]
        del o_ref, l_ref
        cflops = cw.flops()
        c_tf = cflops / (run["ms"] * 1e-3) / 1e12
        per_workload[f"C{ci}"] = {
            "workload": cw.describe(), "gpu_us": run["ms"] * 1e3, "timing": run["timing"],
            "counted_flops": cflops, "value": c_tf, "unit": "TFLOP/s",
            "frac_of_measured_bf16_peak": c_tf / peaks["bf16_tflops"], "parity": par}
        if ci == 3 and n_rows == total_rows and world == 1 and not args.no_cpu_baseline:
            # The oracle's full run on this workload is the CPU baseline.
            cpu = {"value": row_flops / o_dt / 1e12, "unit": "TFLOP/s", "cores": omp_threads(),
                   "cpu_model": cpu_model(), "kind": "oracle",
                   "sample": f"all {n_rows} query rows of {cw.name} ({row_flops / 1e9:.1f} "
                             f"GFLOP counted, {o_dt:.1f} s): the parity check of the timed "
                             f"output"}
    # Workload 5: partials against the oracle's split, combined O/LSE against
    # the unsplit forward.
    t0 = time.perf_counter()
    op_ref, lp_ref = oracle.decode_split(dq_h, dk_h, dv_h, d.num_splits, d.scale)
    o5_ref, l5_ref = oracle.attn_fwd(dq_h, dk_h, dv_h, False, d.scale)
    o_dt = time.perf_counter() - t0
    op_g, lp_g, o5_g, l5_g = c5_out
    par = parity_errors(o5_g.numpy(), l5_g.numpy(), o5_ref[:, :, 0], l5_ref[:, :, 0])
    par_p = parity_errors(op_g.numpy(), lp_g.numpy(), op_ref, lp_ref)
    par.update({"rows": d.B * d.Hq, "rows_total": d.B * d.Hq, "oracle_s": o_dt,
                "partials": {k2: par_p[k2] for k2 in ("o_max_abs_err", "lse_max_err", "pass")}})
    par["pass"] = bool(par["pass"] and par_p["pass"])
    parity_ok &= par["pass"]
    per_workload["C5"] = {
        "workload": d.describe(), "gpu_us": d_ms * 1e3,
        "timing": "split + combine, CUDA events, mean of the decode object's launches",
        "algorithmic_bytes": dbytes, "value": dbytes / (d_ms * 1e-3) / 1e9, "unit": "GB/s",
        "frac_of_measured_hbm": dbytes / (d_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
        "frac_of_nominal_8tbs": dbytes / (d_ms * 1e-3) / 1e9 / 8000.0, "parity": par}

    if cpu is None and world == 1 and not args.no_cpu_baseline:
        rows, dt = run_oracle_sample(w, q_h, k_h, v_h, args.cpu_seconds, seed=w.seed)
        cflops = oracle_rows_flops(w, rows)
        cpu = {"value": cflops / dt / 1e12, "unit": "TFLOP/s", "cores": omp_threads(),
               "cpu_model": cpu_model(), "kind": "oracle",
               "sample": f"{rows.numel()} query rows of {w.name} ({cflops / 1e9:.1f} GFLOP "
                         f"counted, {dt:.1f} s)"}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": prefill_config(w),
        "frac_of_measured_bf16_peak": achieved / peaks["bf16_tflops"],
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                     "traffic": PREFILL_TRAFFIC_BYTES,
                     "peak_source": f"{peaks_src} cuBLAS bf16 burst"},
        "back_to_back": back_to_back,
        "decode": decode,
        "backward": backward,
        "qkv_rope": qkv_rope,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "configs": per_workload,
        "parity_ok": bool(parity_ok),
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if not parity_ok:
        sys.exit(3)


def profile_arm(args):
    """A short run of one path for ncu: `--profile prefill|decode|backward|qkv|d256`, no
    flush, no e2e, no CPU baseline; `--batch` shrinks the workload's batch.
    `backward` runs one forward, then the Delta, dK/dV and dQ kernels per step."""
    import dataclasses

    import tensor_attn_fwd_gb300 as attn
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    w = DECODE if args.profile == "decode" else PREFILL
    if args.batch:
        w = dataclasses.replace(w, B=args.batch)
    if args.profile not in ("d256", "fwd"):
        q, k, v = (t.to(device) for t in workload_inputs(w))
    if args.profile == "prefill":
        def fn():
            attn.attn_fwd(q, k, v, causal=w.causal, scale=w.scale)
    elif args.profile == "qkv":
        import math as _m
        hidden = 4096
        g = torch.Generator().manual_seed(w.seed + 11)
        xq = torch.randn((w.B, w.Sq, hidden), generator=g).to(torch.bfloat16).to(device)
        wq = (torch.randn(((w.Hq + 2 * w.Hkv) * w.D, hidden), generator=g)
              / _m.sqrt(hidden)).to(torch.bfloat16).to(device)
        table = attn.attn_rope_table(w.Sq, w.D, 10000.0)

        def fn():
            attn.attn_qkv_rope(xq, wq, table, w.Hq, w.Hkv)
    elif args.profile == "d256":
        # head dimension 256: causal GQA Hq16 Hkv4 S8192 (batch from --batch, default 2)
        from attn_inputs import make_qkv
        bsz = args.batch or 2
        q, k, v = (t.to(device) for t in make_qkv(bsz, 16, 4, 8192, 8192, 256, seed=2561))
        w = dataclasses.replace(w, name="gqa_hq16_hkv4_s8192_d256_causal", B=bsz, Hq=16, Hkv=4,
                                D=256)

        def fn():
            attn.attn_fwd(q, k, v, causal=True, scale=1.0 / 16.0)
    elif args.profile == "fwd":
        # any forward shape: --shape B,Hq,Hkv,Sq,Sk,D,causal (inputs N(0,1), seed 7)
        from attn_inputs import make_qkv
        B_, Hq_, Hkv_, Sq_, Sk_, D_, c_ = (int(x) for x in args.shape.split(","))
        q, k, v = (t.to(device) for t in make_qkv(B_, Hq_, Hkv_, Sq_, Sk_, D_, seed=7))
        w = dataclasses.replace(w, name=f"fwd_{args.shape.replace(',', '_')}", B=B_, Hq=Hq_,
                                Hkv=Hkv_, Sq=Sq_, Sk=Sk_, D=D_, causal=bool(c_))

        def fn():
            attn.attn_fwd(q, k, v, causal=bool(c_), scale=1.0 / math.sqrt(D_))
    elif args.profile == "backward":
        o, lse = attn.attn_fwd(q, k, v, causal=w.causal, scale=w.scale)
        g = torch.Generator().manual_seed(w.seed + 7)
        dout = torch.randn(q.shape, generator=g).to(torch.bfloat16).to(device)

        def fn():
            attn.attn_bwd(q, k, v, o, lse, dout, causal=w.causal, scale=w.scale)
    else:
        def fn():
            attn.decode(q, k, v, w.num_splits, w.scale)
    for _ in range(args.warmup + args.steps):
        fn()
    torch.cuda.synchronize()
    if attn.attn_debug_status() != attn.ATTN_OK:
        raise RuntimeError("kernel reported a timeout")
    print(json.dumps({"profile": args.profile, "workload": w.describe(),
                      "launches": args.warmup + args.steps}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--no-qkv-rope", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--parity", choices=["all", "sample"], default="all",
                    help="oracle check of workloads 3 and 4: every row, or the row sample")
    ap.add_argument("--profile", choices=["prefill", "decode", "backward", "qkv", "d256", "fwd"],
                    default=None,
                    help="run a few launches of one kernel (for ncu) and exit")
    ap.add_argument("--batch", type=int, default=0, help="override B in --profile mode")
    ap.add_argument("--shape", default="1,32,32,8192,8192,64,0",
                    help="--profile fwd: B,Hq,Hkv,Sq,Sk,D,causal")
    args = ap.parse_args()
    if args.warmup < 3 and not args.profile:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    dist_on = world > 1
    if args.impl == "reference":
        reference_arm(args, rank, world)
        return
    if args.profile:
        profile_arm(args)
        return
    if dist_on:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        ours_arm(args, rank, world, local_rank, dist_on)
    finally:
        if dist_on:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
