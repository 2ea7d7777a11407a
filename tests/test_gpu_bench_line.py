"""The benchmark's contract line, on a short run: one JSON line with every
key the contract names, a roofline object for the dominant kernel, the CPU
baseline, the end-to-end figure with its host traffic, and a launch count."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--configs", "main", "--steps", "40",
                        "--warmup", "3", "--cpu-budget", "0.5"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "clocks", "roofline", "cpu_baseline", "e2e", "gpu_launches"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 40 and d["warmup"] == 3
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert "workload" in d["config"] and "model" not in d["config"]
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == "GB/s"
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] == 2 * 40
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
    # integer results of the CUDA path and of the oracle, checksummed alike
    ck = d["checks"]
    assert ck["match"] is True and ck["gpu"] == ck["oracle"], ck
    assert d["gpu"]["sms"] > 0 and d["build"]["source_sha256"]
