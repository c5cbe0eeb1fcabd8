"""bench.py's JSON line on the GPU: one short run, every key of the
contract present and consistent (the driver reads these)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_keys():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "3", "--warmup", "3",
                        "--no-cpu-baseline", "--no-rows"], capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks", "cpu_baseline"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["value"] > 0 and d["unit"] == "TOPS" and d["higher_is_better"] is True
    assert d["gpu_launches"] >= d["steps"]  # row quantization and the product each step
    rf = d["roofline"]
    assert rf["bound"] == "tensor" and rf["unit"] == "TFLOP/s" and 0 < rf["frac"] < 1.5
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["clocks"]["sm_mhz"] > 0
    assert d["cpu_baseline"] is None  # skipped by the flag
    for k in ("quantize_linear", "dequantize_linear", "quantize_linear_s8_per_tensor",
              "dequantize_linear_s8_per_tensor"):
        assert d[k]["value"] > 0 and 0 < d[k]["frac_hbm"] < 1.5
