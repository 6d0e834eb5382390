"""The benchmark's GPU arm on a small workload: one JSON line carrying every key
its output contract names (roofline of the dominant kernel, the CPU oracle
baseline, the end-to-end number through the public API with its copy volumes,
the count of this library's kernel launches and the clocks sampled while the
timed region ran)."""
import json
import os
import subprocess
import sys

import pytest

from conftest import ROOT

pytestmark = pytest.mark.gpu


def test_gpu_arm_prints_one_full_contract_line():
    B, H, T, d, N = 1, 4, 2048, 128, 4
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--shape", f"{B},{H},{T},{d},{N},1",
                        "--steps", "3", "--warmup", "3", "--e2e-steps", "2", "--cpu-budget-s", "2",
                        "--no-separate-merge", "--no-decode", "--no-two-pass", "--no-other-workloads",
                        "--e2e-settle-s", "0"],
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.strip().splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e",
                "gpu_launches", "clocks"):
        assert key in line, key
    assert line["n_gpus"] == 1 and line["steps"] == 3 and line["warmup"] == 3
    assert line["value"] > 0 and line["ms_per_step"] > 0 and line["higher_is_better"] is True
    assert line["dtype"] == "bf16" and line["scaling"] == "weak"
    assert line["config"]["workload"].startswith(f"custom_B{B}_H{H}_T{T}_d{d}_N{N}")

    roof = line["roofline"]
    assert roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s"
    assert roof["achieved"] > 0 and roof["peak"] > 0
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-9
    assert roof["traffic"] is None  # DRAM counters are recorded for the page-1 workload only

    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["sample"]

    e = line["e2e"]
    assert e["value"] > 0 and e["unit"] == line["unit"]
    # inputs in: q, k and v; results out: out (bf16) and lse (fp32)
    assert e["h2d_bytes_per_step"] == 3 * B * H * T * d * 2
    assert e["d2h_bytes_per_step"] == B * H * T * d * 2 + B * H * T * 4
    assert len(e["step_ms"]) == 2 and e["h2d_gbs_before"] > 0 and "settle" in e
    assert len(e["warmup_ms"]) >= 4  # two set-up calls, then at least two settling calls
    assert e["call"] == "rsa_ring_attn_fwd_host" and e["steps"] == 2
    assert set(e["host_buffers"]) == {"q", "k", "v", "out+lse"}
    for info in e["host_buffers"].values():
        assert info["kind"] in ("registered-huge", "pinned") and info["bytes"] > 0
    assert sum(e["slabs"]) == B * H

    assert line["gpu_launches"] > 0
    assert "sm_mhz" in line["clocks"] and "reasons" in line["clocks"]
