"""bench.py's GPU arm on a shrunk headline step: the one JSON line carries the
fields the benchmark contract names, with values consistent with each other."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_contract():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--tokens-per-rank", "256",
                        "--steps", "4", "--warmup", "3", "--no-sweep", "--no-cpu-baseline",
                        "--no-next-rows"],
                       capture_output=True, text=True, cwd=ROOT, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "roofline",
                "e2e", "gpu_launches", "clocks", "breakdown"):
        assert key in line, key
    assert line["n_gpus"] == 1 and line["steps"] == 4 and line["warmup"] == 3
    assert line["higher_is_better"] is True and line["unit"] == "GB/s" and line["value"] > 0
    assert line["config"]["workload"].startswith("moe-layer R8 E256 K8 S256 H7168 B32")
    roof = line["roofline"]
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s" and roof["kernel"] in ("k_dispatch", "k_combine")
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"], rel=1e-3)
    # the traffic record belongs to the full-size workload only
    assert roof["traffic"] is None
    e2e = line["e2e"]
    assert e2e["unit"] == "GB/s" and e2e["value"] > 0
    # inputs: topk_idx int32 + topk_w fp32 + hidden bf16; outputs: out bf16 + the status word
    N, K, H = 8 * 256, 8, 7168
    assert e2e["h2d_bytes_per_step"] == N * K * 4 + N * K * 4 + N * H * 2
    assert e2e["d2h_bytes_per_step"] == N * H * 2 + 4
    # k_hist, k_plan, k_offsets (no k_gsum at 8 tiles), dispatch, combine per timed step
    assert line["gpu_launches"] == 4 * 5
    assert "medium_step" in line["breakdown"] and line["breakdown"]["medium_step"]["reduce_grad_gbs"] > 0
    assert line["clocks"]["sm_max_mhz"] is None or line["clocks"]["sm_max_mhz"] > 0
