"""GPU parity of mep_prefetch against the CPU oracle: a byte copy of each used
slot's home expert weights, unused slots untouched; bit-exact."""

import numpy as np
import pytest
import torch

import load_balancing_topk_gb300 as mep
import oracle
from load_balancing_topk_gb300 import synth

from gpu_util import DEV, to_dev, to_np

pytestmark = pytest.mark.gpu


def check(se, home, slot, E, status=None):
    st_ref, s_ref = oracle.prefetch(se, home, slot, E)
    hd, sd = to_dev(home), to_dev(slot)
    mep.mep_prefetch(to_dev(se) if isinstance(se, np.ndarray) else se, hd, sd, status, E)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_np(sd), s_ref)
    np.testing.assert_array_equal(to_np(hd), home)
    return st_ref


def _bf16_weights(rows, n, seed):
    return synth.bf16_normal(rows, n, seed=seed, tag=31)


def test_prefetch_plan_map_bf16_weights():
    """Weights of E=64 experts of H=2048 x H'=1408 bf16, slot map from the
    E=64 / R=8 / K=6 / S=4096 plan (maxvio 0.5)."""
    s = synth.MEDIUM
    idx, _ = synth.routing(s, seed=0, alpha=0.075684)
    p = mep.mep_plan(to_dev(idx), s.R, s.S, s.K, s.E, s.B)
    torch.cuda.synchronize()
    se = to_np(p.slot_expert)
    n = synth.GRAD_H * synth.GRAD_HP
    home = _bf16_weights(s.E, n, 0)
    slot = _bf16_weights(s.R * s.B, n, 1)
    assert check(se, home, slot, s.E, p.status) == "ok"
    assert (se >= 0).sum() > 0


def test_prefetch_all_slots_fp32():
    E, R, B = 64, 8, 8
    se = synth.full_slot_map(E, R, B, seed=2)
    rng = np.random.default_rng(0)
    home = rng.standard_normal((E, 4096 + 8)).astype(np.float32)
    slot = rng.standard_normal((R * B, 4096 + 8)).astype(np.float32)
    check(se, home, slot, E)


@pytest.mark.parametrize("n", [8, 24, 1000, 4104])
def test_prefetch_ragged_sizes(n):
    E, R, B = 6, 3, 2
    se = np.array([[1, 4], [-1, -1], [4, 2]], dtype=np.int32)
    home = _bf16_weights(E, n, 3)
    slot = _bf16_weights(R * B, n, 4)
    check(se, home, slot, E)


def test_prefetch_bad_map_and_status():
    E, R, B, n = 4, 2, 2, 64
    home = _bf16_weights(E, n, 5)
    slot = np.zeros((R * B, n), np.uint16)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    sd = to_dev(slot)
    mep.mep_prefetch(to_dev(np.array([[0, 4], [1, -1]], np.int32)), to_dev(home), sd, status, E)
    torch.cuda.synchronize()
    assert int(status.item()) == mep.STATUS_CODE["MEP_ERR_BAD_SLOT_MAP"]
    assert (to_np(sd) == 0).all()
    status.fill_(mep.STATUS_CODE["MEP_ERR_CAPACITY"])
    mep.mep_prefetch(to_dev(np.array([[0, 3], [1, -1]], np.int32)), to_dev(home), sd, status, E)
    torch.cuda.synchronize()
    assert (to_np(sd) == 0).all()


@pytest.mark.parametrize("R,B,E,n,frac", [
    (1024, 32, 4096, 8, 0.6),     # R*B = 32768, the slot limit; expert ids up to 4095; 16-byte experts
    (64, 64, 4096, 24, 0.3),      # 4096 slots, experts of 48 bytes: every item spans many slots
    (16, 24, 384, 520, 0.9),      # experts of 1040 bytes (65 vectors): items cross slot boundaries
])
def test_prefetch_large_slot_maps(R, B, E, n, frac):
    """Slot maps far larger than a plan's: the used slots are listed by every
    CTA (one part of the map per warp), their vectors cut into equal items that
    cross from slot to slot; the largest expert id and the largest slot id
    both occur. Unused slots must stay untouched."""
    rng = np.random.default_rng([R, B, E, n])
    se = rng.integers(0, E, size=(R, B), dtype=np.int32)
    se[rng.random((R, B)) > frac] = -1
    se[0, 0] = E - 1
    se[R - 1, B - 1] = E - 1
    home = _bf16_weights(E, n, 6)
    slot = _bf16_weights(R * B, n, 7)
    assert check(se, home, slot, E) == "ok"
