"""The C ABI from a caller written in plain C (tests/c_abi_ring.c): it
includes only include/rsa.h and the CUDA runtime's C API.  Without a GPU the
program is compiled as C99 with warnings as errors and linked against
librsa.so, so the header is valid C and every symbol it uses resolves.  With
a GPU it runs: the ring and the host-to-host call on its own seeded inputs,
one argument error with its message; its results are compared with the
oracle here."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
import context_attention_rsa_gb300 as rsa
from conftest import ROOT
from gpu_helpers import assert_close, need_cuda

B, H, T, D = 1, 2, 1024, 128   # the shape the program uses


def _cuda_home():
    for c in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if c and os.path.exists(os.path.join(c, "include", "cuda_runtime_api.h")):
            return c
    return None


def _build_caller(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    cuda = _cuda_home()
    if not cc or not cuda:
        pytest.skip("no C compiler or CUDA headers")
    libdir = next((os.path.join(cuda, d) for d in ("lib64", "lib") if os.path.exists(
        os.path.join(cuda, d, "libcudart.so"))), None)
    if libdir is None:
        pytest.skip("no libcudart.so")
    lib = rsa.library_path()
    exe = str(tmp_path / "c_abi_ring")
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-O2", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), os.path.join(ROOT, "tests", "c_abi_ring.c"), "-o", exe,
           "-L", os.path.dirname(lib), "-l:" + os.path.basename(lib), "-L", libdir, "-lcudart",
           "-Wl,-rpath," + os.path.dirname(lib) + ":" + libdir]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-3000:]
    return exe


def test_c_caller_compiles_as_c99_and_links_against_the_library(tmp_path):
    exe = _build_caller(tmp_path)
    assert os.path.exists(exe)


def _read_bf16(path):
    a = np.fromfile(path, dtype=np.uint16).view(np.int16)
    return torch.from_numpy(a.copy()).view(torch.bfloat16).reshape(B, H, T, D)


@pytest.mark.gpu
def test_c_caller_runs_and_matches_the_oracle(tmp_path):
    need_cuda()
    exe = _build_caller(tmp_path)
    out_dir = tmp_path / "out"
    out_dir.mkdir()
    r = subprocess.run([exe, str(out_dir)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, (r.stdout + r.stderr)[-3000:]
    assert "host_call_bit_exact 1" in r.stdout
    q, k, v = (_read_bf16(out_dir / f"{n}.bin") for n in "qkv")
    out = _read_bf16(out_dir / "out.bin")
    lse = torch.from_numpy(np.fromfile(out_dir / "lse.bin", dtype=np.float32).copy()).reshape(B, H, T)
    ro, rl = oracle.attention(q, k, v, True)
    assert_close(out, lse, ro, rl, torch.bfloat16, what="C caller")
