"""The benchmark's multi-rank host logic on two CPU ranks (gloo): every rank
gets the slowest rank's time, the whole-job value counts all ranks' units over
that time, and the reference arm prints one line from rank 0 only.  The GPU
runs of this pool have one GPU each, so the NCCL path is not run here."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 * (rank + 1)           # rank 1 is the slow one
        got = bench.max_over_ranks(dist, ms, "cpu")
        out[rank] = (got, bench.whole_job_tflops(1e12, world, got))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_on_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(2, _free_port(), out), nprocs=2, start_method="spawn", join=True)
        res = dict(out)
    # both ranks see the slowest rank's 20 ms; 2 ranks x 1e12 FLOPs in 20 ms = 100 TFLOP/s
    assert res[0] == res[1] == (20.0, pytest.approx(100.0))


def test_without_a_group_the_local_time_stands():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, 12.5, "cpu") == 12.5
    assert bench.whole_job_tflops(2e12, 1, 20.0) == pytest.approx(100.0)


def test_reference_arm_under_torchrun_two_ranks_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--shape", "1,1,256,64,4,1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
