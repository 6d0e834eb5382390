"""The RSA_DEBUG build (device-side bounds checks on the kernels' computed
global accesses, recorded into the device error word without a trap) runs
the ragged and degenerate parity cases: every one must pass with no bounds
check failing.  This stands in for a memory checker, which this machine does
not offer."""
import os
import subprocess
import sys

import pytest

from conftest import ROOT

pytestmark = pytest.mark.gpu

FILES = ["test_gpu_ring.py", "test_gpu_block.py", "test_gpu_decode.py", "test_gpu_block_kernels.py",
         "test_gpu_failures.py", "test_gpu_two_pass.py", "test_gpu_fuzz.py"]


def test_parity_cases_pass_under_the_bounds_checked_build():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, RSA_DEBUG="1")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           *[os.path.join(ROOT, "tests", f) for f in FILES]]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    assert r.returncode == 0, (r.stdout + r.stderr)[-4000:]
    assert " passed" in r.stdout and "failed" not in r.stdout
    # the subprocess really ran the checked build
    probe = subprocess.run([sys.executable, "-c", "import context_attention_rsa_gb300 as r; "
                            "print(r.load().rsa_debug_checks())"], cwd=ROOT, env=env, capture_output=True,
                           text=True, timeout=600)
    assert probe.stdout.strip().endswith("1"), probe.stderr[-2000:]
