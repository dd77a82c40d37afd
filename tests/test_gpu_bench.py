"""bench.py end to end on the GPU, on the tiny workload: one JSON line with
every key of the contract (roofline, CPU baseline, end-to-end, launches,
clocks), exactly the steps and warm-up asked, a clean mailbox and sane
values."""
import json
import subprocess
import sys
from pathlib import Path

import pytest

pytestmark = pytest.mark.gpu
ROOT = Path(__file__).resolve().parents[1]


def test_bench_line_has_every_contract_key(cuda):
    res = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--workload", "tiny",
                          "--steps", "60", "--warmup", "3", "--cpu-seconds", "0.1"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    line = json.loads(res.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert key in line, key
    assert line["n_gpus"] == 1 and line["steps"] == 60 and line["warmup"] == 3
    assert line["value"] > 0
    assert line["higher_is_better"] is True and line["scaling"] == "weak"
    roof = line["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in roof, key
    assert roof["bound"] == "hbm" and roof["traffic"] is None  # recorded for the headline only
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] == 1 and cpu["value"] > 0
    assert cpu["all_cores"]["cores"] >= 1 and cpu["all_cores"]["value"] > 0
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] == 256 + 8  # x [1][256] + scales [1][8]
    assert e2e["d2h_bytes_per_step"] == 256 * 2  # out [1][256] BF16
    assert line["gpu_launches"] == 2 * 60
    assert "sm_mhz" in line["clocks"] and "reasons" in line["clocks"]
    assert "window" in line["clocks"]
    assert line["workloads"] == {}  # the other workloads ride on the headline's line only
    assert "L2" in line["config"]["l2"]
