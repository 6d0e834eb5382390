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
# The RSA_DEBUG variant: device-side bounds checks on the kernels' computed
# global accesses, which record the first bad index into the device error
# word (no trap) and skip the access.
DEBUG_BUILD = os.path.join(BUILD, "debug")
DEBUG_LIB = os.path.join(DEBUG_BUILD, "librsa.so")

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


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool = False) -> str:
    """Compile librsa.so (or, with debug, its RSA_DEBUG variant) if stale;
    returns its path.  Raises on failure."""
    out_dir, lib = (DEBUG_BUILD, DEBUG_LIB) if debug else (BUILD, LIB)
    stamp = os.path.join(out_dir, "librsa.stamp")
    if debug:
        extra_flags = ["-DRSA_DEBUG=1", *extra_flags]
    with _lock:
        os.makedirs(out_dir, exist_ok=True)
        dig = _digest(extra_flags)
        if not force and os.path.exists(lib) and os.path.exists(stamp):
            with open(stamp) as f:
                if f.read().strip() == dig:
                    return lib
        cc = nvcc()
        objs = []
        cmds = []
        for src in sources():
            obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
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
        tmp = lib + f".tmp{os.getpid()}"
        link = [cc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart=static"]
        r = subprocess.run(link, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + " ".join(link) + "\n" + r.stdout + r.stderr)
        os.replace(tmp, lib)
        with open(stamp, "w") as f:
            f.write(dig)
        return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True,
                extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else []))
