"""mep_plan_static_scratch: the planner for callers that cannot allocate.

Such callers (a host program that reaches the GPU only through the C ABI,
or a runtime whose device memory belongs to one pool allocator) cannot hand
mep_plan a workspace, so this entry point uses a fixed scratch array
compiled into the library. The tests call it through the C ABI several times
in a row on the shared array, on routings of different sizes in both orders
(the larger stress routing before and after the medium one, then a small
routing after the largest; then sixteen random shapes, capacity refusals among
them), and check every output bit for bit against the CPU oracle's plan (the
fixed routings also against mep_plan's; integer outputs: bit-exact, the
tolerance of the plan tests). A later, smaller call therefore cannot pass
on scratch bytes left over from a larger one. They also check that sizes
needing more scratch than the array holds are refused before anything runs.
"""

import ctypes

import numpy as np
import pytest
import torch

import load_balancing_topk_gb300 as mep
import oracle
from load_balancing_topk_gb300 import _build, synth

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return mep.load_library()


def _plan_static(lib, idx_d, s):
    out = dict(
        expert_counts=torch.full((s.E,), -7, dtype=torch.int32, device=DEV),
        cu_seqlens=torch.full((s.R, s.E + s.B), -7, dtype=torch.int32, device=DEV),
        slot_expert=torch.full((s.R, s.B), -7, dtype=torch.int32, device=DEV),
        dst_pos=torch.full((s.N, s.K), -7, dtype=torch.int32, device=DEV),
        status=torch.full((1,), -7, dtype=torch.int32, device=DEV),
    )
    rc = lib.mep_plan_static_scratch(
        idx_d.data_ptr(), s.R, s.S, s.K, s.E, s.B, out["expert_counts"].data_ptr(),
        out["cu_seqlens"].data_ptr(), out["slot_expert"].data_ptr(), out["dst_pos"].data_ptr(),
        out["status"].data_ptr(), torch.cuda.current_stream(DEV).cuda_stream)
    assert rc == 0, mep.STATUS.get(rc, rc)
    return out


CASES = {
    "medium": (synth.MEDIUM, dict(alpha=0.075684), 0),
    "stress": (synth.STRESS, dict(alpha=1.2, kind="hot"), 1),
    "small": (synth.Shape(R=4, E=12, K=3, S=1000, H=8, B=9), dict(alpha=1.0), 2),
}


def _inputs(names):
    out = []
    for name in names:
        s, kw, seed = CASES[name]
        idx, _ = synth.routing(s, seed=seed, **kw)
        out.append((name, s, idx, torch.from_numpy(idx).to(DEV)))
    return out


@pytest.mark.parametrize("order", [("medium", "stress", "small"), ("stress", "medium", "small")],
                         ids=lambda o: "-".join(o))
def test_static_scratch_plan_matches_oracle_and_mep_plan_on_calls_in_a_row(lib, order):
    inputs = _inputs(order)
    # calls in a row on the shared scratch, then the workspace entry point
    static = [_plan_static(lib, idx_d, s) for _, s, _, idx_d in inputs]
    torch.cuda.synchronize()
    static = [{k: v.cpu().numpy() for k, v in o.items()} for o in static]
    for (name, s, idx, idx_d), got in zip(inputs, static):
        want = oracle.plan(idx, s.R, s.S, s.K, s.E, s.B)
        assert want["status"] == "ok"
        assert int(got["status"][0]) == 0, name
        np.testing.assert_array_equal(got["expert_counts"], want["counts"], err_msg=name)
        for key in ("cu_seqlens", "slot_expert", "dst_pos"):
            np.testing.assert_array_equal(got[key], want[key], err_msg=f"{name} {key}")
        ref = mep.mep_plan(idx_d, s.R, s.S, s.K, s.E, s.B)
        torch.cuda.synchronize()
        assert int(ref.status.item()) == 0
        for key in ("expert_counts", "cu_seqlens", "slot_expert", "dst_pos"):
            np.testing.assert_array_equal(got[key], getattr(ref, key).cpu().numpy(),
                                          err_msg=f"{name} {key}")


def test_static_scratch_random_shapes_in_a_row(lib):
    """Random shapes (K up to 12, capacity refusals among them) planned back
    to back on the shared scratch, each against the oracle: status, counts,
    cu_seqlens and slot table always, destination rows when the plan is ok."""
    codes = {"ok": 0, "capacity": mep.STATUS_CODE["MEP_ERR_CAPACITY"]}
    g = np.random.default_rng(31337)
    draws = []
    for i in range(16):
        R = int(g.choice([1, 2, 4, 8, 16, 33]))
        E = R * int(g.integers(1, 9))
        K = int(min(E, g.choice([1, 2, 4, 6, 8, 12])))
        S = int(g.integers(0, 1500))
        B = int(g.integers(0, 8))
        s = synth.Shape(R=R, E=E, K=K, S=S, H=8, B=B)
        idx, _ = synth.routing(s, seed=i, alpha=float(g.uniform(0, 2)))
        draws.append((s, idx, torch.from_numpy(idx).to(DEV)))
    outs = [_plan_static(lib, idx_d, s) for s, _, idx_d in draws]
    torch.cuda.synchronize()
    n_ok = 0
    for (s, idx, _), got in zip(draws, outs):
        got = {k: v.cpu().numpy() for k, v in got.items()}
        want = oracle.plan(idx, s.R, s.S, s.K, s.E, s.B)
        assert int(got["status"][0]) == codes[want["status"]]
        np.testing.assert_array_equal(got["expert_counts"], want["counts"])
        np.testing.assert_array_equal(got["cu_seqlens"], want["cu_seqlens"])
        np.testing.assert_array_equal(got["slot_expert"], want["slot_expert"])
        if want["status"] == "ok":
            n_ok += 1
            np.testing.assert_array_equal(got["dst_pos"], want["dst_pos"])
    assert n_ok >= 6


def test_static_scratch_refuses_sizes_beyond_its_array(lib):
    # E = 4096 experts with 2^20 tokens needs 256 tile histograms of 16 KB: > 4 MiB
    R, S, K, E, B = 16, 65536, 1, 4096, 8
    assert mep.plan_workspace_bytes(R, S, K, E, B) > 4 << 20
    rc = lib.mep_plan_static_scratch(None, R, S, K, E, B, None, None, None, None, None, None)
    assert rc == mep.STATUS_CODE["MEP_ERR_INVALID_ARG"]
