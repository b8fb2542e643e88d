"""The benchmark's one JSON line on the GPU: printed alone, short enough to be
read whole at the end of the output, and carrying every key of the line's
contract (roofline with the traffic record, CPU baseline, end-to-end leg,
clocks, kernel launches) and the five workload configurations."""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_prints_one_complete_line():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "5", "--warmup", "3",
                          "--e2e-steps", "2"], cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, lines
    assert len(lines[0]) < 3000
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e",
                "gpu_launches", "clocks", "configs"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3 and d["gpu_launches"] == 5
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and 0 < r["frac"] < 1.5
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    assert r["traffic"] is None or 0 < r["traffic"] <= 306184192          # read once: never above the algorithmic bytes
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] == 268435456 and e["d2h_bytes_per_step"] == 37748736
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
    assert sorted(d["configs"]) == ["1", "2", "3", "4", "5"]
