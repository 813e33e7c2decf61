"""Host-side logic of bench.py: max-over-ranks timing on two gloo ranks (CPU),
whole-job aggregation, byte accounting and the reference arm's CPU sample."""

import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from load_balancing_topk_gb300 import synth  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = [10.0 + rank, 5.0 - rank]
    got = bench.max_over_ranks(mine, dist)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, got))


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [11.0, 5.0]


def test_max_over_ranks_single_process():
    assert bench.max_over_ranks([1.5, 2.0], None) == [1.5, 2.0]


def test_whole_job_gbs_counts_every_rank():
    assert bench.whole_job_gbs(1, 2e9, 1000.0) == pytest.approx(2.0)
    assert bench.whole_job_gbs(4, 2e9, 1000.0) == pytest.approx(8.0)


def test_step_bytes():
    s = synth.MEDIUM
    se = np.array([[-1] * 8] * 7 + [[3, 3, 5, -1, -1, -1, -1, -1]], dtype=np.int32)
    nb = bench.step_bytes(s, 2048 * 1408, se)
    assert nb["dispatch"] == s.N * s.H * 2 + s.A * s.H * 2 + 4 * s.A
    assert nb["combine"] == s.A * s.H * 2 + s.N * s.H * 2 + 8 * s.A
    assert nb["used"] == 3 and nb["distinct"] == 2
    assert nb["reduce_grad"] == 2 * (3 + 2) * 2048 * 1408 * 4 + 4 * 64


def test_step_bytes_without_gradients():
    s = synth.LARGE
    nb = bench.step_bytes(s)
    assert nb["reduce_grad"] == 0
    assert nb["total"] == nb["plan"] + nb["dispatch"] + nb["combine"]
    # dispatch + combine = 2 (1 + K) N H 2 bytes plus the index / weight words
    assert nb["dispatch"] + nb["combine"] == 2 * (1 + s.K) * s.N * s.H * 2 + 12 * s.A


def test_oracle_step_sample_runs_small():
    s, alpha = bench.medium_workload()
    r = bench.oracle_step_sample(s, alpha, 0.005, grads=True)
    assert r["bytes"] > 0 and r["seconds"] > 0 and r["n_tok"] == int(32768 * 0.005)
    s, alpha = bench.headline_workload()
    r = bench.oracle_step_sample(s, alpha, 0.0005, grads=False)
    assert r["reduce_s"] < 1e-3 and r["n_tok"] == int(65536 * 0.0005)
    assert abs(r["maxvio"] - 0.5) < 0.01


def test_reference_arm_prints_the_contract_line():
    import json
    import subprocess

    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True, cwd=ROOT,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "GB/s" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["steps"] == 1 and line["warmup"] == 3
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == line["value"] and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"].startswith("moe-layer R8 E256 K8 S8192 H7168 B32")


def test_bench_rejects_short_warmup():
    import subprocess

    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"],
                       capture_output=True, text=True, cwd=ROOT, timeout=120)
    assert r.returncode != 0 and "warmup" in r.stderr
