"""The benchmark's JSON line on the GPU: one line from a short run of the
default workload, with the keys its contract asks for and values that hold
together (device-timed throughput from the step time, the roofline fraction
from its parts, end-to-end bytes counted from the copied tensors)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_default_bench_line_has_the_contract_keys():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--extra=", "--steps", "3",
                        "--warmup", "3", "--no-cpu-baseline"],
                       capture_output=True, text=True, cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "clocks", "gpu_launches", "graph_ms_per_step"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["config"]["workload"] == "block_bf16_d768"
    tokens = 8 * 1024
    assert abs(d["value"] - tokens / (d["ms_per_step"] / 1e3)) <= 1e-6 * d["value"]
    rf = d["roofline"]
    assert rf["bound"] in ("tensor", "hbm") and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) <= 1e-9
    e = d["e2e"]
    assert e["unit"] == "tokens/s" and 0 < e["value"]
    assert e["h2d_bytes_per_step"] == e["d2h_bytes_per_step"] == tokens * 768 * 2  # bf16 x, out
    assert e["link"]["h2d_gbs"] > 0 and e["host_enqueue_ms_per_step"] > 0
    assert d["gpu_launches"] > 0 and d["clocks"]["sm_max_mhz"] > 0
    assert d["cached_weights"]["ms_per_step"] > 0
