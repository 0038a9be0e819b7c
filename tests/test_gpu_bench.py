"""The benchmark's JSON line on a GB300 (needs a GPU): the contract fields, the
timed steps replayed as one graph of exactly --steps launches, and the
secondary record through the same timing path."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


def test_bench_line_has_the_contract_fields():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "7",
                        "--warmup", "3", "--no-cpu-baseline", "--workload",
                        "qwen2.5-0.5b-mlp-m128", "--secondary", "qwen2.5-7b-decode-m16"],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in line, key
    assert line["steps"] == 7 and line["warmup"] == 3 and line["gpu_launches"] == 7
    assert line["value"] > 0 and line["n_gpus"] == 1
    assert "exactly 7 steps" in line["config"]["launch"]
    roof = line["roofline"]
    assert roof["bound"] == "hbm" and 0 < roof["frac"] < 1.5
    assert abs(roof["avg_launch_us"] * 1e-3 - line["ms_per_step"]) < 1e-3
    e2e = line["e2e"]
    assert e2e["h2d_bytes_per_step"] == 2 * 128 * 896 and e2e["d2h_bytes_per_step"] == 2 * 128 * 4864
    assert e2e["copy_rates"]["h2d_gbs"] > 0 and e2e["copy_rates"]["d2h_gbs"] > 0
    assert all(e2e["phases"][k] > 0 for k in ("h2d_ms", "kernel_ms", "d2h_ms"))
    (sec,) = line["secondary"]
    assert sec["workload"] == "qwen2.5-7b-decode-m16" and sec["gpu_launches"] == 7
    assert sec["roofline"]["kernel"] == "fused_small_m_kernel" and sec["value"] > 0
