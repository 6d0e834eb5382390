"""In-tree build of librsa.so with nvcc for sm_103a.

Each .cu file is compiled to an object in parallel, then linked into
``context_attention_rsa_gb300/_build/librsa.so``.  A stamp of the sources,
headers and flags makes repeated calls free when nothing changed.
"""
from __future__ import annotations

import concurrent.futures
import hashlib
import os
import shutil
import subprocess
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "librsa.so")
STAMP = os.path.join(BUILD, "librsa.stamp")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xcompiler", "-Wall", "-Xcompiler", "-Wno-unused-function"]

_lock = threading.Lock()


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build librsa")
    return cand


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _inputs():
    files = sources() + sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                               if f.endswith((".h", ".cuh"))) + [os.path.join(INCLUDE, "rsa.h")]
    return files


def _digest(extra_flags) -> str:
    h = hashlib.sha256()
    for f in _inputs():
        h.update(f.encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(ARCH + NVCC_FLAGS + list(extra_flags)).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile librsa.so if stale; returns its path.  Raises on failure."""
    with _lock:
        os.makedirs(BUILD, exist_ok=True)
        dig = _digest(extra_flags)
        if not force and os.path.exists(LIB) and os.path.exists(STAMP):
            with open(STAMP) as f:
                if f.read().strip() == dig:
                    return LIB
        cc = nvcc()
        objs = []
        cmds = []
        for src in sources():
            obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
            objs.append(obj)
            cmds.append([cc, *ARCH, *NVCC_FLAGS, *extra_flags, "-I", INCLUDE, "-c", src, "-o", obj])

        def run(cmd):
            r = subprocess.run(cmd, capture_output=True, text=True)
            return cmd, r

        with concurrent.futures.ThreadPoolExecutor(max_workers=min(8, len(cmds))) as ex:
            results = list(ex.map(run, cmds))
        for cmd, r in results:
            if verbose and (r.stdout or r.stderr):
                print(r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        tmp = LIB + f".tmp{os.getpid()}"
        link = [cc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart=static"]
        r = subprocess.run(link, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + " ".join(link) + "\n" + r.stdout + r.stderr)
        os.replace(tmp, LIB)
        with open(STAMP, "w") as f:
            f.write(dig)
        return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True,
                extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else []))
