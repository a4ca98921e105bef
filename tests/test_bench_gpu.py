"""bench.py on the GPU: one short run must print exactly one JSON line with
every key the benchmark contract asks for, and numbers that hang together."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


def test_bench_prints_the_contract_line(arlib):
    steps, warmup = 50, 3
    r = subprocess.run([sys.executable, "bench.py", "--quick", "--steps", str(steps), "--warmup",
                        str(warmup)], cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] == warmup
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert "workload" in d["config"] and d["data"] == "synthetic"
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["sample"]
    assert cb["single_thread"]["value"] > 0 and cb["single_thread"]["cores"] == 1
    assert cb["cpu_model"]
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert e["residual_out_equals_device_path"] is True
    assert e["copy_engines"]["value"] > 0
    assert d["gpu_launches"] == steps * d["config"]["plan"]["launches"]
    assert set(d["clocks"]) >= {"sm_mhz", "sm_max_mhz", "reasons"}
    # value is bytes per step x steps over the timed region, in GB/s
    n, m, H = d["config"]["n"], d["config"]["m"], d["config"]["H"]
    algo = (n + 3) * m * H * 2 + H * 2
    assert abs(algo / (d["ms_per_step"] * 1e-3) / 1e9 - d["value"]) / d["value"] < 0.02
    assert d["latency_vs_m"] and all("auto" in row for row in d["latency_vs_m"])
