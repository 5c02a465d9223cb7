"""Build libattn.so (the CUDA library behind the C ABI in include/attn.h).

Each translation unit under csrc/ is compiled in parallel with nvcc for
sm_103a only, then linked into ``tensor_attn_fwd_gb300/libattn.so`` (in-tree,
git-ignored).  The build is skipped when the library is newer than every source.

    python -m tensor_attn_fwd_gb300.build [--force] [--verbose]
"""
from __future__ import annotations

import argparse
import glob
import os
import re
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_PATH = os.path.join(PKG_DIR, "libattn.so")
# The debug library: every prefill output store is checked against its buffer
# (ATTN_DEBUG_BOUNDS; a stray store is skipped and reported as ATTN_ERR_BOUNDS).
DEBUG_BUILD_DIR = os.path.join(PKG_DIR, "_build_debug")
DEBUG_LIB_PATH = os.path.join(PKG_DIR, "libattn_debug.so")
DEBUG_FLAGS = ["-DATTN_DEBUG_BOUNDS"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    cuda_home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(cuda_home, "bin", "nvcc")
    if os.path.exists(cand):
        return cand
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found (set CUDA_HOME)")
    return found


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (sources() + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h"))
            + [os.path.abspath(__file__)])


def up_to_date(lib_path: str = LIB_PATH) -> bool:
    if not os.path.exists(lib_path):
        return False
    t = os.path.getmtime(lib_path)
    return all(os.path.getmtime(d) <= t for d in _deps())


# Kernels that rebalance registers with setmaxnreg must be compiled with exactly
# the per-thread count their split assumes (threads x count = the pool that
# setmaxnreg.inc draws from); a smaller count would make .inc wait forever.
EXACT_REGISTERS = {"attn_fwd_kernel": 168}


def check_register_counts(ptxas_log: str):
    """Parse `ptxas -v` output; raise if a kernel in EXACT_REGISTERS deviates."""
    current = None
    seen = set()
    for line in ptxas_log.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            current = m.group(1)
            continue
        m = re.search(r"Used (\d+) registers", line)
        if m and current:
            for name, want in EXACT_REGISTERS.items():
                if name in current:
                    seen.add(name)
                    if int(m.group(1)) != want:
                        raise RuntimeError(
                            f"{current}: ptxas used {m.group(1)} registers, the setmaxnreg "
                            f"split needs exactly {want}")
            current = None
    return seen


def build(force: bool = False, verbose: bool = False, extra_flags=None, debug: bool = False) -> str:
    lib_path = DEBUG_LIB_PATH if debug else LIB_PATH
    build_dir = DEBUG_BUILD_DIR if debug else BUILD_DIR
    if not force and up_to_date(lib_path):
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    flags = NVCC_FLAGS + ["-Xptxas", "-v"] + (DEBUG_FLAGS if debug else []) + list(extra_flags or [])

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, *flags, "-I", INCLUDE, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with ThreadPoolExecutor(max_workers=max(1, min(len(sources()), os.cpu_count() or 1))) as ex:
        results = list(ex.map(compile_one, sources()))
    failed = False
    seen = set()
    for src, _, r in results:
        if verbose or r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode != 0:
            failed = True
            sys.stderr.write(f"nvcc failed for {src}\n")
        else:
            seen |= check_register_counts(r.stdout + r.stderr)
    if failed:
        raise RuntimeError("libattn build failed")
    missing = set(EXACT_REGISTERS) - seen
    if missing:
        raise RuntimeError(f"no ptxas register report for {sorted(missing)}")
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", *[o for _, o, _ in results],
           "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("libattn link failed")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--debug", action="store_true", help="build libattn_debug.so (bounds checks)")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose, debug=a.debug))
