"""The C ABI used from plain C: tests/c_abi/attn_abi_demo.c is compiled with
gcc against include/attn.h and linked with libattn.so and the CUDA runtime
(no Python or PyTorch in the caller).  On a GPU it runs attn_fwd on inputs
written here and its outputs are compared with the oracle."""
import math
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
import tensor_attn_fwd_gb300 as attn
from attn_inputs import make_qkv
from tensor_attn_fwd_gb300 import build as attn_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi", "attn_abi_demo.c")


def _cuda_home():
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    if not os.path.isdir(os.path.join(home, "include")):
        pytest.skip("CUDA toolkit headers not found")
    return home


def build_demo(out_dir):
    attn_build.build()
    home = _cuda_home()
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    lib_dir = os.path.dirname(attn.library_path())
    exe = os.path.join(out_dir, "attn_abi_demo")
    cuda_lib = next((d for d in (os.path.join(home, "lib64"), os.path.join(home, "lib"),
                                 os.path.join(home, "targets", "sbsa-linux", "lib"),
                                 os.path.join(home, "targets", "x86_64-linux", "lib"))
                     if os.path.exists(os.path.join(d, "libcudart.so"))), None)
    if cuda_lib is None:
        pytest.skip("libcudart.so not found")
    cmd = ["gcc", "-std=c11", "-Wall", "-Werror", "-O1", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(home, "include"), SRC, "-o", exe, "-L", lib_dir, "-lattn",
           "-L", cuda_lib, "-lcudart", f"-Wl,-rpath,{lib_dir}", f"-Wl,-rpath,{cuda_lib}"]
    subprocess.run(cmd, check=True)
    return exe


def test_c_header_compiles_and_links(tmp_path):
    exe = build_demo(str(tmp_path))
    assert os.path.exists(exe)


@pytest.mark.gpu
@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D,causal", [
    (1, 2, 2, 128, 128, 64, 0),
    (2, 8, 2, 300, 450, 128, 1),
])
def test_c_caller_matches_oracle(tmp_path, B, Hq, Hkv, Sq, Sk, D, causal):
    exe = build_demo(str(tmp_path))
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Sk, D, seed=Sq + Sk + D)
    bits = [oracle._bf16_bits(t).reshape(-1) for t in (q, k, v)]
    inp, out = tmp_path / "in.bin", tmp_path / "out.bin"
    np.concatenate(bits).astype(np.uint16).tofile(inp)
    scale = 1.0 / math.sqrt(D)
    r = subprocess.run([exe, str(inp), str(out), str(B), str(Hq), str(Hkv), str(Sq), str(Sk),
                        str(D), str(causal), repr(scale)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    res = np.fromfile(out, dtype=np.float32)
    n_o = B * Hq * Sq * D
    o = res[:n_o].reshape(B, Hq, Sq, D)
    lse = res[n_o:].reshape(B, Hq, Sq)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, bool(causal), scale)
    from test_parity import assert_close
    assert_close(o, lse, o_ref, lse_ref, "C caller")
