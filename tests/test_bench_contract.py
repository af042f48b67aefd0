"""The bench's one-line JSON contract: the reference arm (the oracle on the
host, no GPU needed) and the GPU arm carry every key the driver reads, with
the same metric, unit and direction."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args, timeout=600):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                       text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def _common(d, steps, warmup):
    import bench
    assert d["metric"] == bench.METRIC
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] == warmup
    assert d["scaling"] == "weak" and d["dtype"] == "bf16" and d["vs_baseline"] is None
    assert isinstance(d["value"], float) and d["value"] > 0 and d["ms_per_step"] > 0
    assert "synthetic" in d["data"] and "workload" in d["config"]
    assert set(d["e2e"]) >= {"value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"}
    assert d["e2e"]["unit"] == d["unit"]


def test_reference_arm_line():
    d = _run("--impl", "reference", "--steps", "1", "--warmup", "3", "--ref-budget", "1")
    _common(d, 1, 3)
    assert d["impl"] == "reference"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_warmup_below_three_is_refused():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"], cwd=ROOT,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode != 0 and "warmup" in r.stderr


@pytest.mark.gpu
def test_gpu_arm_line():
    d = _run("--tokens", "1024", "--steps", "3", "--warmup", "3", "--no-cpu-baseline")
    _common(d, 3, 3)
    assert "impl" not in d
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    assert rf["traffic"] is None          # the committed capture is of T=8192, not 1024
    assert d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["d2h_bytes_per_step"] > 0
    assert isinstance(d["gpu_launches"], int) and d["gpu_launches"] >= 3 * 3
    assert set(d["clocks"]) >= {"sm_mhz", "sm_max_mhz", "reasons"}
    assert d["config"]["T"] == 1024
