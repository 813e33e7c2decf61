"""mep_plan_static_scratch: the planner for callers that cannot allocate.

Such callers (a host program that reaches the GPU only through the C ABI,
or a runtime whose device memory belongs to one pool allocator) cannot hand
mep_plan a workspace, so this entry point uses a fixed scratch array
compiled into the library. The test calls it through the C ABI twice in a
row, on different routings, and checks every output against mep_plan's
(integer outputs: bit-exact, the tolerance of the plan tests). It also
checks that sizes needing more scratch than the array holds are refused
before anything runs.
"""

import ctypes

import numpy as np
import pytest
import torch

import load_balancing_topk_gb300 as mep
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


def test_static_scratch_plan_matches_mep_plan_on_two_calls_in_a_row(lib):
    cases = [(synth.MEDIUM, dict(alpha=0.075684), 0),
             (synth.STRESS, dict(alpha=1.2, kind="hot"), 1)]
    inputs = []
    for s, kw, seed in cases:
        idx, _ = synth.routing(s, seed=seed, **kw)
        inputs.append((s, torch.from_numpy(idx).to(DEV)))
    # two calls in a row on the shared scratch, then the workspace entry point
    static = [_plan_static(lib, idx_d, s) for s, idx_d in inputs]
    torch.cuda.synchronize()
    static = [{k: v.cpu().numpy() for k, v in o.items()} for o in static]
    for (s, idx_d), got in zip(inputs, static):
        ref = mep.mep_plan(idx_d, s.R, s.S, s.K, s.E, s.B)
        torch.cuda.synchronize()
        assert int(got["status"][0]) == int(ref.status.item()) == 0
        for name in ("expert_counts", "cu_seqlens", "slot_expert", "dst_pos"):
            np.testing.assert_array_equal(got[name], getattr(ref, name).cpu().numpy(), err_msg=name)


def test_static_scratch_refuses_sizes_beyond_its_array(lib):
    # E = 4096 experts with 2^20 tokens needs 256 tile histograms of 16 KB: > 4 MiB
    R, S, K, E, B = 16, 65536, 1, 4096, 8
    assert mep.plan_workspace_bytes(R, S, K, E, B) > 4 << 20
    rc = lib.mep_plan_static_scratch(None, R, S, K, E, B, None, None, None, None, None, None)
    assert rc == mep.STATUS_CODE["MEP_ERR_INVALID_ARG"]
