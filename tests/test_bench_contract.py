"""bench.py's JSON line: every key the measurement contract names, with values
of the right kind, from a short run on the GPU (and the reference arm's line
from the oracle on the CPU)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args):
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                         check=True, capture_output=True, text=True, timeout=900)
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    return json.loads(lines[0])


@pytest.mark.gpu
def test_bench_line_has_the_contract_keys():
    d = run_bench("--steps", "3", "--warmup", "3", "--no-backward", "--no-qkv-rope",
                  "--parity", "sample")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["value"] > 0 and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == "gqa_b2_hq32_hkv8_s8192_d128_causal"
    r = d["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    assert r["traffic"] is None or r["traffic"] > 0
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["value"] > 0
    e = d["e2e"]
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0 and e["value"] > 0
    assert d["gpu_launches"] >= d["steps"]
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
    dec = d["decode"]
    assert dec["roofline"]["bound"] == "hbm" and dec["value"] > 0
    # one entry per workload, each tied to an oracle check of its own timed output
    assert sorted(d["configs"]) == ["C1", "C2", "C3", "C4", "C5"]
    for name, c in d["configs"].items():
        assert c["gpu_us"] > 0 and c["value"] > 0, name
        p = c["parity"]
        assert p["pass"] is True and p["rows"] >= 1, (name, p)
        assert p["o_max_abs_err"] <= 2e-2 and p["lse_max_err"] <= 1e-3, (name, p)
    for name in ("C1", "C2", "C5"):
        assert d["configs"][name]["parity"]["rows"] == d["configs"][name]["parity"]["rows_total"]
    assert d["parity_ok"] is True
    assert d["cpu_baseline"]["cpu_model"]
