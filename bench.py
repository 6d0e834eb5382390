#!/usr/bin/env python3
"""Benchmark: blockwise ring self-attention forward on GB300.

One step = one rsa_ring_attn_fwd call over the whole workload (every block-
attention pair of every ring round and every merge), inputs resident in HBM.
Default workload: the page-1 shape (B=8, H=64, T=32768, d=128, N=4 chunks,
causal, bf16).  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle, timed on a sample

Multi-GPU (torchrun): every rank runs its own copy of the workload (independent
batches, no data exchange); value = all ranks' useful FLOPs / max rank time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import time

_ROOT = os.path.dirname(os.path.abspath(__file__))
if _ROOT not in sys.path:
    sys.path.insert(0, _ROOT)

METRIC = "ring-attn fwd TFLOP/s (causal-useful) and % BF16 tensor peak; merge HBM GB/s"
UNIT = "TFLOP/s"


def useful_flops(B, H, T, d, causal):
    pairs = T * (T + 1) // 2 if causal else T * T
    return 4.0 * B * H * d * pairs


def merge_bytes_per_step(w, sched):
    """Algorithmic merge bytes of one ring.  Per row and merge: read the fp32
    accumulator (4d) and the fp32 partial (4d) and both lse values (8), write
    the accumulator (4d) and its lse (4): 12d+12.  A chunk's last merge writes
    the output in the input dtype instead: (8+esz)d+12."""
    BH = w.B * w.H
    Tc = w.T // w.N
    esz = 2 if w.dtype == "bf16" else 4
    total = 0
    for r in range(1, w.N):
        for (i, j) in sched(r):
            last = (i if w.causal else w.N - 1) == r
            per = (8 + esz) * w.d + 12 if last else 12 * w.d + 12
            total += BH * Tc * per
    return total


def read_peaks():
    path = os.path.join(_ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm_gbs=float(p["hbm_gbs"]), bf16_tflops=float(p["bf16_tflops"]),
                    bf16_tflops_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    except Exception:
        return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


def block_traffic():
    """Per-launch DRAM traffic of the block kernel from the committed ncu
    capture, or None if the kernel sources changed since it was taken."""
    import hashlib
    path = os.path.join(_ROOT, "profiles", "block_attn_bf16_page1_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        m = hashlib.sha256()
        for src in rec["sources"]:
            with open(os.path.join(_ROOT, src), "rb") as f:
                m.update(f.read())
        if m.hexdigest()[:16] != rec["source_sha256_16"]:
            return None
        return rec["traffic_bytes_per_launch_mean"]
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock and throttle-reason sampling during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        sm_sorted = sorted(sm)
        return {"sm_mhz": sm_sorted[len(sm_sorted) // 2], "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def two_pass_bytes(B, H, T, d, N, esz=2):
    """HBM bytes one two-pass ring moves at the least.  Per query chunk: every
    score is written (fp32) and read back by the row softmax, which writes P
    (bf16) for the output pass to read: 12 bytes per score over the full
    [Tc, T] rows.  Add Q and K read by the score pass, V by the output pass,
    and out and lse written."""
    BH, Tc = B * H, T // N
    per_chunk = BH * Tc * T * (4 + 4 + 2 + 2) + BH * Tc * d * esz + 2 * BH * T * d * esz + BH * Tc * (d * esz + 4)
    return per_chunk * N


def max_over_ranks(pg, x: float, device) -> float:
    """The largest x of all ranks (x itself when there is no process group):
    a step of the whole job lasts as long as its slowest rank."""
    if pg is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank: float, world: int, ms_per_step: float) -> float:
    """Throughput of the whole job: every rank's units over the slowest rank's time."""
    return flops_per_rank * world / (ms_per_step * 1e-3) / 1e12


def cpu_baseline(w, q_cpu_rows, k_cpu, v_cpu, rows, budget_s=15.0):
    """Time the oracle (as it stands) on a bounded sample of query rows."""
    import numpy as np
    import oracle
    n_thr = oracle.max_threads()
    # size the sample: time a small probe, then scale to ~budget_s
    n_probe = min(16, len(rows))
    t0 = time.perf_counter()
    oracle.attend_rows(q_cpu_rows[:n_probe], k_cpu, v_cpu, rows[:n_probe], w.causal)
    dt = max(time.perf_counter() - t0, 1e-3)
    n = int(min(len(rows), max(n_probe, n_probe * budget_s / dt)))
    n = max(n_thr, (n // n_thr) * n_thr) if n >= n_thr else n
    n = min(n, len(rows))
    t0 = time.perf_counter()
    oracle.attend_rows(q_cpu_rows[:n], k_cpu, v_cpu, rows[:n], w.causal)
    dt = time.perf_counter() - t0
    fl = oracle.rows_flops(rows[:n], w.T, w.d, w.causal)
    # the whole workload at the sample's rate, rows weighted by their key counts
    full_s = useful_flops(w.B, w.H, w.T, w.d, w.causal) / (fl / dt)
    return {"value": fl / dt / 1e12, "unit": UNIT, "cores": n_thr, "kind": "oracle",
            "sample": f"{n} sampled query rows of {w.name} (fp64 C, OpenMP over rows), {dt:.1f} s",
            "rows_per_s": n / dt, "fp64_gflops": fl / dt / 1e9, "full_workload_s_extrapolated": full_s}


def run_reference(args, w):
    """--impl reference: the CPU oracle on a bounded sample per step."""
    import numpy as np
    import torch
    import oracle
    import rsa_inputs
    world, rank, _ = dist_info()
    if rank != 0:
        return 0
    # inputs drawn on the CPU for the sampled heads only: every head is an
    # independent problem, so sample rows from one (b, h) slice
    B1 = rsa_inputs.Workload(w.name, 1, 1, w.T, w.d, w.N, w.causal, w.dtype, w.recipe, w.check)
    q, k, v = rsa_inputs.make_workload(B1, seed=0, device="cpu")
    rows = rsa_inputs.sample_rows(B1, n=4096, seed=1)
    qa = q.view(torch.int16).numpy().view(np.uint16) if q.dtype == torch.bfloat16 else q.numpy()
    q_rows = np.ascontiguousarray(qa[rows[:, 0], rows[:, 1], rows[:, 2]])
    n_thr = oracle.max_threads()
    # rows per step sized so one step takes about 5 s
    t0 = time.perf_counter()
    oracle.attend_rows(q_rows[:n_thr], k, v, rows[:n_thr], w.causal)
    per_row = (time.perf_counter() - t0) / n_thr
    n = int(max(n_thr, min(len(rows), 5.0 / max(per_row, 1e-6) * n_thr / n_thr)))
    n = min(len(rows), max(n_thr, (n // n_thr) * n_thr))
    times, fl = [], oracle.rows_flops(rows[:n], w.T, w.d, w.causal)
    for s in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.attend_rows(q_rows[:n], k, v, rows[:n], w.causal)
        if s >= args.warmup:
            times.append(time.perf_counter() - t0)
    tot = sum(times)
    value = fl * len(times) / tot / 1e12
    line = {"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": tot / len(times) * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "d": w.d, "N": w.N,
                       "causal": w.causal, "input_dtype": w.dtype},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": n_thr, "kind": "oracle",
                             "sample": f"{n} sampled query rows of one head per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="rsa", choices=["rsa", "reference"])
    ap.add_argument("--workload", default="page1_causal_bf16")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-separate-merge", action="store_true",
                    help="skip timing the ring variant with the separate merge kernel")
    ap.add_argument("--no-decode", action="store_true", help="skip timing decode on the million-token cache")
    ap.add_argument("--no-two-pass", action="store_true", help="skip timing the two-pass RSA form")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip timing the ring on the ragged and million-token workloads")
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--e2e-settle-tol", type=float, default=0.1,
                    help="before the e2e timed loop, warm up until two calls in a row agree this closely")
    ap.add_argument("--e2e-settle-s", type=float, default=30.0, help="longest such warm-up")
    ap.add_argument("--shape", default=None,
                    help="B,H,T,d,N,causal: a bf16 normal-recipe workload instead of --workload (profiling)")
    args = ap.parse_args()

    import rsa_inputs
    w = rsa_inputs.WORKLOADS[args.workload]
    if args.shape:
        B_, H_, T_, d_, N_, c_ = (int(x) for x in args.shape.split(","))
        w = rsa_inputs.Workload(f"custom_B{B_}_H{H_}_T{T_}_d{d_}_N{N_}_{'causal' if c_ else 'full'}",
                                B_, H_, T_, d_, N_, bool(c_), "bf16", "normal", "sample")
    if args.impl == "reference":
        return run_reference(args, w)

    import numpy as np
    import torch
    import context_attention_rsa_gb300 as rsa

    world, rank, local = dist_info()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    rsa.load()

    q, k, v = rsa_inputs.make_workload(w, seed=rank, device=dev)
    B, H, T, d, N, causal = w.B, w.H, w.T, w.d, w.N, w.causal
    out = torch.empty_like(q)
    lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)
    ws = torch.empty(max(rsa.workspace_size(q.dtype, B, H, T, d, N, causal), 1), dtype=torch.uint8, device=dev)
    n_launch = rsa.ring_launch_count(N, causal)
    stream = torch.cuda.current_stream()

    def barrier():
        if pg is not None:
            pg.barrier()

    for _ in range(max(args.warmup, 0)):
        rsa.ring_attn(q, k, v, N, causal, out=out, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    rsa.check_device_error()

    # The headline: K plain rsa_ring_attn_fwd calls, nothing else in the timed region.
    t_start = torch.cuda.Event(enable_timing=True)
    t_stop = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    for s in range(args.steps):
        rsa.ring_attn(q, k, v, N, causal, out=out, lse=lse, workspace=ws)
    t_stop.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    rsa.check_device_error()
    ms_total = max_over_ranks(pg, t_start.elapsed_time(t_stop), dev)
    ms_step = ms_total / args.steps

    # Per-kernel breakdown, in a separate loop: the same ring with CUDA events
    # recorded around each launch on the launching stream.
    ev0 = [[torch.cuda.Event(enable_timing=True) for _ in range(n_launch)] for _ in range(args.steps)]
    ev1 = [[torch.cuda.Event(enable_timing=True) for _ in range(n_launch)] for _ in range(args.steps)]
    torch.cuda.synchronize()
    kinds = None
    for s in range(args.steps):
        kinds = rsa.ring_attn_timed(q, k, v, N, causal, out, lse, ws, ev0[s], ev1[s])
    torch.cuda.synchronize()
    rsa.check_device_error()

    # the default ring folds every pair in the block epilogue: all its launches are block launches
    blk_ms = sum(ev0[s][i].elapsed_time(ev1[s][i]) for s in range(args.steps) for i in range(n_launch)
                 if kinds[i] == 0) / args.steps
    n_blk = sum(1 for x in kinds if x == 0)

    flops = useful_flops(B, H, T, d, causal)
    value = whole_job_tflops(flops, world, ms_step)
    peaks = read_peaks()
    blk_tflops = flops / (blk_ms * 1e-3) / 1e12
    mbytes = merge_bytes_per_step(w, lambda r: rsa.ring_schedule(N, causal, r))
    # Per round (one block launch per round when a round has at most 32
    # pairs): time, useful FLOPs and pair-equivalents (a full Tc x Tc block is
    # one; a causal diagonal block (Tc+1)/(2 Tc)).
    rounds = None
    if n_launch == N:
        Tc = T // N
        rounds = []
        for r in range(N):
            pe = sum(((Tc + 1) / (2 * Tc)) if (causal and i == j) else 1.0 for (i, j) in rsa.ring_schedule(N, causal, r))
            r_ms = sum(ev0[s][r].elapsed_time(ev1[s][r]) for s in range(args.steps)) / args.steps
            r_fl = 4.0 * B * H * d * Tc * Tc * pe
            rounds.append({"round": r, "ms": r_ms, "pair_equivalents": pe, "ms_per_pair_equivalent": r_ms / pe,
                           "tflops": r_fl / (r_ms * 1e-3) / 1e12})

    # ---- the ring with the separate merge kernel (RSA_RING_SEPARATE_MERGE) ------
    # Each round's partials go to the workspace and one merge launch folds
    # them in: the merge kernel's HBM roofline is measured here.
    sep = None
    mrg_ms = mrg_gbs = None
    n_mrg = 0
    if not args.no_separate_merge:
        ws_s = torch.empty(max(rsa.workspace_size(q.dtype, B, H, T, d, N, causal, fused=False), 1),
                           dtype=torch.uint8, device=dev)
        n_s = rsa.ring_launch_count(N, causal, fused=False)
        for _ in range(max(args.warmup, 0)):
            rsa.ring_attn(q, k, v, N, causal, out=out, lse=lse, workspace=ws_s, fused=False)
        barrier()
        torch.cuda.synchronize()
        t_start.record(stream)
        for s_ in range(args.steps):
            rsa.ring_attn(q, k, v, N, causal, out=out, lse=lse, workspace=ws_s, fused=False)
        t_stop.record(stream)
        torch.cuda.synchronize()
        barrier()
        rsa.check_device_error()
        s_ms = max_over_ranks(pg, t_start.elapsed_time(t_stop), dev) / args.steps
        se0 = [[torch.cuda.Event(enable_timing=True) for _ in range(n_s)] for _ in range(args.steps)]
        se1 = [[torch.cuda.Event(enable_timing=True) for _ in range(n_s)] for _ in range(args.steps)]
        s_kinds = None
        for s_ in range(args.steps):
            s_kinds = rsa.ring_attn_timed(q, k, v, N, causal, out, lse, ws_s, se0[s_], se1[s_], fused=False)
        torch.cuda.synchronize()
        rsa.check_device_error()
        s_blk = sum(se0[s_][i].elapsed_time(se1[s_][i]) for s_ in range(args.steps) for i in range(n_s)
                    if s_kinds[i] == 0) / args.steps
        mrg_ms = sum(se0[s_][i].elapsed_time(se1[s_][i]) for s_ in range(args.steps) for i in range(n_s)
                     if s_kinds[i] == 1) / args.steps
        n_mrg = sum(1 for x in s_kinds if x == 1)
        mrg_gbs = mbytes / (mrg_ms * 1e-3) / 1e9 if mrg_ms > 0 else None
        sep = {"value": whole_job_tflops(flops, world, s_ms), "unit": UNIT, "ms_per_step": s_ms,
               "block_kernel_tflops": flops / (s_blk * 1e-3) / 1e12, "block_kernel_ms_per_step": s_blk,
               "merge_ms_per_step": mrg_ms, "launches_per_step": n_s, "workspace_bytes": int(ws_s.numel())}
        del ws_s

    # ---- decode against a sharded million-token KV cache (HBM-bound) ---------
    dec = None
    if not args.no_decode and world == 1:
        del ws
        torch.cuda.empty_cache()
        wd = rsa_inputs.WORKLOADS["decode_million_bf16"]
        qd_full, kd, vd = rsa_inputs.make_workload(wd, seed=1, device=dev)
        qd = qd_full[:, :, wd.T - wd.q_len:].contiguous()
        del qd_full
        od = torch.empty_like(qd)
        ld = torch.empty((wd.B, wd.H, wd.q_len), dtype=torch.float32, device=dev)
        wsd = torch.empty(rsa.decode_workspace_size(qd.dtype, wd.B, wd.H, wd.T, wd.d, wd.q_len, wd.N),
                          dtype=torch.uint8, device=dev)
        for _ in range(max(args.warmup, 0)):
            rsa.decode_attn(qd, kd, vd, wd.N, wd.causal, out=od, lse=ld, workspace=wsd)
        torch.cuda.synchronize()
        d0 = torch.cuda.Event(enable_timing=True)
        d1 = torch.cuda.Event(enable_timing=True)
        d0.record(stream)
        for _ in range(args.steps):
            rsa.decode_attn(qd, kd, vd, wd.N, wd.causal, out=od, lse=ld, workspace=wsd)
        d1.record(stream)
        torch.cuda.synchronize()
        rsa.check_device_error()
        d_ms = d0.elapsed_time(d1) / args.steps
        # algorithmic bytes: the whole K and V cache once, the queries and the outputs
        dbytes = 2 * kd.numel() * kd.element_size() + 2 * qd.numel() * qd.element_size() + ld.numel() * 4
        dec = {"workload": wd.name, "B": wd.B, "H": wd.H, "T": wd.T, "d": wd.d, "N": wd.N, "q_len": wd.q_len,
               "ms_per_step": d_ms, "bound": "hbm", "achieved": dbytes / (d_ms * 1e-3) / 1e9, "unit": "GB/s",
               "peak": peaks["hbm_gbs"], "frac": dbytes / (d_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
               "algorithmic_bytes_per_step": dbytes, "useful_tflops": 4.0 * wd.B * wd.H * wd.d * wd.T * wd.q_len
               / (d_ms * 1e-3) / 1e12, "launches_per_step": 2}
        del qd, kd, vd, od, ld, wsd
        torch.cuda.empty_cache()
        ws = None

    # ---- two-pass RSA (full score rows) on the bidirectional workload -------
    tp = None
    if not args.no_two_pass and world == 1:
        wt = rsa_inputs.WORKLOADS["noncausal_bf16"]
        qt, kt, vt = rsa_inputs.make_workload(wt, seed=0, device=dev)
        ot = torch.empty_like(qt)
        lt = torch.empty((wt.B, wt.H, wt.T), dtype=torch.float32, device=dev)
        wst = torch.empty(rsa.two_pass_workspace_size(qt.dtype, wt.B, wt.H, wt.T, wt.d, wt.N), dtype=torch.uint8,
                          device=dev)
        wsr = torch.empty(max(rsa.workspace_size(qt.dtype, wt.B, wt.H, wt.T, wt.d, wt.N, wt.causal), 1),
                          dtype=torch.uint8, device=dev)
        timings, graph_ms = {}, {}
        calls = (("two_pass", lambda: rsa.two_pass_attn(qt, kt, vt, wt.N, wt.causal, out=ot, lse=lt, workspace=wst)),
                 ("online_ring", lambda: rsa.ring_attn(qt, kt, vt, wt.N, wt.causal, out=ot, lse=lt, workspace=wsr)))

        def timed(fn):
            for _ in range(max(args.warmup, 0)):
                fn()
            torch.cuda.synchronize()
            t0_ = torch.cuda.Event(enable_timing=True)
            t1_ = torch.cuda.Event(enable_timing=True)
            t0_.record(stream)
            for _ in range(args.steps):
                fn()
            t1_.record(stream)
            torch.cuda.synchronize()
            return t0_.elapsed_time(t1_) / args.steps

        for name, fn in calls:
            timings[name] = timed(fn)
        # The same calls captured once as CUDA graphs and replayed: the calls
        # only enqueue kernels, so one capture holds the whole ring, and the
        # replay leaves shorter gaps between its kernels.
        for name, fn in calls:
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr):
                fn()
            torch.cuda.synchronize()
            graph_ms[name] = timed(gr.replay)
            del gr
        rsa.check_device_error()
        fl_t = useful_flops(wt.B, wt.H, wt.T, wt.d, wt.causal)
        tp = {"workload": wt.name, "ms_per_step": timings["two_pass"],
              "tflops": fl_t / (timings["two_pass"] * 1e-3) / 1e12,
              "workspace_bytes": int(wst.numel()), "online_ring_ms_per_step": timings["online_ring"],
              "online_ring_tflops": fl_t / (timings["online_ring"] * 1e-3) / 1e12,
              "online_ring_workspace_bytes": int(wsr.numel()), "launches_per_step": 3 * wt.N}
        tb = two_pass_bytes(wt.B, wt.H, wt.T, wt.d, wt.N)
        hbm = read_peaks()["hbm_gbs"]
        tp.update({"bound": "hbm", "algorithmic_bytes_per_step": tb,
                   "achieved_gbs": tb / (timings["two_pass"] * 1e-3) / 1e9,
                   "frac_of_measured_hbm": tb / (timings["two_pass"] * 1e-3) / 1e9 / hbm,
                   "graph_replay": {"ms_per_step": graph_ms["two_pass"],
                                    "achieved_gbs": tb / (graph_ms["two_pass"] * 1e-3) / 1e9,
                                    "frac_of_measured_hbm": tb / (graph_ms["two_pass"] * 1e-3) / 1e9 / hbm,
                                    "online_ring_ms_per_step": graph_ms["online_ring"]}})
        del qt, kt, vt, ot, lt, wst, wsr
        torch.cuda.empty_cache()

    # ---- the ring on the other synthetic workloads (median of 3 timed rings) --
    others = None
    if not args.no_other_workloads and world == 1:
        others = {}
        pk = read_peaks()
        for name in ("tiny_fp32_causal", "ragged_causal_bf16", "million_causal_bf16"):
            wo = rsa_inputs.WORKLOADS[name]
            qo, ko, vo = rsa_inputs.make_workload(wo, seed=0, device=dev)
            oo = torch.empty_like(qo)
            lo = torch.empty((wo.B, wo.H, wo.T), dtype=torch.float32, device=dev)
            wso = torch.empty(max(rsa.workspace_size(qo.dtype, wo.B, wo.H, wo.T, wo.d, wo.N, wo.causal), 1),
                              dtype=torch.uint8, device=dev)
            rsa.ring_attn(qo, ko, vo, wo.N, wo.causal, out=oo, lse=lo, workspace=wso)  # warm-up
            torch.cuda.synchronize()
            times = []
            for _ in range(3):
                a_ = torch.cuda.Event(enable_timing=True)
                b_ = torch.cuda.Event(enable_timing=True)
                a_.record(stream)
                rsa.ring_attn(qo, ko, vo, wo.N, wo.causal, out=oo, lse=lo, workspace=wso)
                b_.record(stream)
                torch.cuda.synchronize()
                times.append(a_.elapsed_time(b_))
            rsa.check_device_error()
            ms_o = sorted(times)[1]
            tf_o = useful_flops(wo.B, wo.H, wo.T, wo.d, wo.causal) / (ms_o * 1e-3) / 1e12
            others[name] = {"B": wo.B, "H": wo.H, "T": wo.T, "d": wo.d, "N": wo.N, "causal": wo.causal,
                            "dtype": wo.dtype, "ms_per_ring_median_of_3": ms_o, "tflops": tf_o}
            if wo.dtype == "bf16":
                others[name]["frac_of_sustained_bf16_peak"] = tf_o / pk["bf16_tflops_sustained"]
            else:  # the SIMT fp32 path: launch-bound at this size, no roofline claim
                others[name]["note"] = "fp32 SIMT path, launch-bound"
            del qo, ko, vo, oo, lo, wso
            torch.cuda.empty_cache()

    # ---- end to end from host memory (public API, rsa_ring_attn_fwd_host) ----
    e2e = None
    if args.e2e_steps > 0:
        qh, kh, vh = (rsa.host_empty(t.shape, t.dtype) for t in (q, k, v))
        for th, td in ((qh, q), (kh, k), (vh, v)):
            th.copy_(td)
        del q, k, v, out, lse, ws
        torch.cuda.empty_cache()
        bufs = {}
        warm_ms = []

        def timed_warmup():
            w0 = torch.cuda.Event(enable_timing=True)
            w1 = torch.cuda.Event(enable_timing=True)
            w0.record(stream)
            rsa.ring_attn_from_host(qh, kh, vh, N, causal, device=dev, buffers=bufs)
            w1.record(stream)
            torch.cuda.synchronize()
            warm_ms.append(round(w0.elapsed_time(w1), 2))

        for _ in range(2):  # warm-up: the library's copy streams, the workspace, the host outputs
            timed_warmup()
        # Host-to-device bandwidth of one copy-engine copy of Q's host buffer,
        # for the record (the call itself routes split parts of a block to the
        # copy kernel, so this probe can be far slower than the call).
        probe = torch.empty_like(qh, device=dev)
        p0 = torch.cuda.Event(enable_timing=True)
        p1 = torch.cuda.Event(enable_timing=True)
        p0.record(stream)
        probe.copy_(qh, non_blocking=True)
        p1.record(stream)
        torch.cuda.synchronize()
        h2d_probe = qh.numel() * qh.element_size() / (p0.elapsed_time(p1) * 1e-3) / 1e9
        del probe
        torch.cuda.empty_cache()
        # Which host pages are huge right before the timed loop, then warm-up
        # calls until two in a row agree within --e2e-settle-tol (at most
        # --e2e-settle-s seconds): on some hosts calls ran 2-15x slower for a
        # while (one host's second call took 1454 ms, later ones 97 ms).
        host_before = {name: dict(rsa.host_info(t), path=rsa.host_copy_path(t)) for name, t in
                       (("q", qh), ("k", kh), ("v", vh), ("out+lse", bufs["out_host"]))}
        t_settle = time.time()
        timed_warmup()
        while True:
            timed_warmup()
            a, b = warm_ms[-2], warm_ms[-1]
            if abs(a - b) <= args.e2e_settle_tol * min(a, b) or time.time() - t_settle >= args.e2e_settle_s:
                break
        settle_s = time.time() - t_settle
        e_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.e2e_steps + 1)]
        barrier()
        torch.cuda.synchronize()
        e_clocks = ClockSampler(local)
        time.sleep(0.3)
        e_ev[0].record(stream)
        for i in range(args.e2e_steps):
            rsa.ring_attn_from_host(qh, kh, vh, N, causal, device=dev, buffers=bufs)
            e_ev[i + 1].record(stream)
        torch.cuda.synchronize()
        e_clk = e_clocks.stop()
        barrier()
        e_steps = [e_ev[i].elapsed_time(e_ev[i + 1]) for i in range(args.e2e_steps)]
        e_ms = max_over_ranks(pg, sum(e_steps) / args.e2e_steps, dev)
        h2d = 3 * qh.numel() * qh.element_size()
        d2h = bufs["out_host"].numel() * bufs["out_host"].element_size() + bufs["lse_host"].numel() * 4
        e2e = {"value": whole_job_tflops(flops, world, e_ms), "unit": UNIT, "ms_per_step": e_ms,
               "call": "rsa_ring_attn_fwd_host", "steps": args.e2e_steps,
               "step_ms": [round(x, 2) for x in e_steps], "warmup_ms": warm_ms, "clocks": e_clk,
               "h2d_gbs_before": round(h2d_probe, 1),
               "settle": {"waited_s": round(settle_s, 1), "tol": args.e2e_settle_tol, "limit_s": args.e2e_settle_s},
               "host_buffers": host_before,
               "host_buffers_after": {name: dict(rsa.host_info(t), path=rsa.host_copy_path(t)) for name, t in
                                      (("q", qh), ("k", kh), ("v", vh), ("out+lse", bufs["out_host"]))},
               "slabs": rsa.slab_plan(B * H),
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
        k_cpu, v_cpu, q_cpu = kh, vh, qh
    else:
        q_cpu, k_cpu, v_cpu = q.cpu(), k.cpu(), v.cpu()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rows = rsa_inputs.sample_rows(w, n=4096, seed=1)
        qa = q_cpu.view(torch.int16).numpy().view(np.uint16) if q_cpu.dtype == torch.bfloat16 else q_cpu.numpy()
        q_rows = np.ascontiguousarray(qa[rows[:, 0], rows[:, 1], rows[:, 2]])
        rng = np.random.default_rng(2)
        perm = rng.permutation(len(rows))
        cpu = cpu_baseline(w, q_rows[perm], k_cpu, v_cpu, rows[perm], budget_s=args.cpu_budget_s)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
            "config": {"workload": w.name, "B": B, "H": H, "T": T, "d": d, "N": N, "causal": causal,
                       "global_batch": B * world, "seq_len": T, "parallelism": f"replicas{world}",
                       "l2": "inputs (3 x %.1f GiB) larger than L2; no flush" % (q_cpu.numel() * 2 / 2**30)},
            "pct_bf16_peak": 100.0 * value / world / peaks["bf16_tflops_sustained"],
            "roofline": {"bound": "tensor", "achieved": blk_tflops, "peak": peaks["bf16_tflops_sustained"],
                         "unit": "TFLOP/s", "frac": blk_tflops / peaks["bf16_tflops_sustained"],
                         "traffic": block_traffic() if w.name == "page1_causal_bf16" else None,
                         "kernel": "block_attn_bf16_kernel<128>",
                         "launches_per_step": n_blk, "ms_per_step": blk_ms, "rounds": rounds,
                         "peak_source": peaks["source"] + " bf16_tflops_sustained"},
            "merge": {"bound": "hbm", "achieved": mrg_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                      "frac": (mrg_gbs / peaks["hbm_gbs"]) if mrg_gbs else None,
                      "algorithmic_bytes_per_step": mbytes, "launches_per_step": n_mrg, "ms_per_step": mrg_ms,
                      "measured_in": "separate_merge_ring",
                      "peak_source": peaks["source"] + " hbm_gbs"},
            "separate_merge_ring": sep,
            "decode": dec,
            "two_pass_rsa": tp,
            "e2e": e2e,
            "other_workloads": others,
            "gpu_launches": n_launch * args.steps,
            "cpu_baseline": cpu,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
