"""The GPU arm's JSON line on one GB300, for one short run of the decode sweep: the metric and timing
fields, the roofline of the dominant kernel (achieved over the measured peak, frac their ratio,
and the achieved figure at most what the whole step's bytes over its time allow), the clocks sampled
during the timed region, the launch count and the end-to-end block with its copied bytes."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_decode_sweep_line():
    r = subprocess.run([sys.executable, "bench.py", "--workload", "decode", "--steps", "20", "--warmup", "3",
                        "--no-cpu-baseline"], cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = lines[0]
    assert d["unit"] == "tokens/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 20 and d["warmup"] == 3 and d["ms_per_step"] > 0
    assert d["scaling"] == "weak" and d["data"] == "synthetic" and isinstance(d["config"]["workload"], str)
    assert d["gpu_launches"] > 0
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    # one launch per layer: the kernel's figure is the step's bytes over the step's time
    lr = d["layer_roofline"]
    assert rf["achieved"] <= lr["achieved"] * 1.000001
    ck = d["clocks"]
    assert ck["sm_mhz"] > 0 and ck["sm_max_mhz"] > 0 and isinstance(ck["reasons"], list)
    e2e = d["e2e"]
    assert e2e["unit"] == d["unit"] and 0 < e2e["value"]
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
