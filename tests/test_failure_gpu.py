"""The bounded waits that keep a GPU usable when a pipeline stalls.

Every mbarrier wait of the grouped GEMM gives up after a time limit, raises
MEP_ERR_TIMEOUT on the device status word and lets the kernel drain and exit.
mep_wait_selftest runs that wait on a barrier that nothing completes (no copy
or tensor-core operation in flight), so the failure path is exercised without
breaking a kernel or faulting the GPU.
"""

import numpy as np
import pytest
import torch

import load_balancing_topk_gb300 as mep
import oracle
from load_balancing_topk_gb300 import synth

from gpu_util import DEV, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_ns", [2_000_000, 20_000_000])
def test_wait_gives_up_after_its_limit_and_reports_timeout(limit_ns):
    status, elapsed = mep.mep_wait_selftest(limit_ns, device=DEV)
    torch.cuda.synchronize()
    assert int(status.item()) == mep.STATUS_CODE["MEP_ERR_TIMEOUT"]
    waited = int(elapsed.item())
    assert limit_ns <= waited < limit_ns + 50_000_000, waited


def test_context_usable_after_a_timeout():
    status, _ = mep.mep_wait_selftest(1_000_000, device=DEV)
    torch.cuda.synchronize()
    assert int(status.item()) == mep.STATUS_CODE["MEP_ERR_TIMEOUT"]
    s = synth.TINY
    idx, _ = synth.routing(s, seed=0, alpha=1.0)
    p = mep.mep_plan(to_dev(idx), s.R, s.S, s.K, s.E, s.B)
    torch.cuda.synchronize()
    ref = oracle.plan(idx, s.R, s.S, s.K, s.E, s.B)
    assert int(p.status.item()) == 0
    np.testing.assert_array_equal(p.dst_pos.cpu().numpy(), ref["dst_pos"])
