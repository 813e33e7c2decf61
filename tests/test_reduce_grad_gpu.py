"""GPU parity of mep_reduce_grad against the CPU oracle.

Both add the slot gradients of an expert to its home gradient in ascending
(rank, slot) order in fp32, so the result is expected bit-exact; the stated
bar is |gpu - oracle| <= 1e-6 * (|home| + sum |slots|) per element.
Consumed slots must be exactly zero and unused slots untouched.
"""

import numpy as np
import pytest
import torch

import load_balancing_topk_gb300 as mep
import oracle
from load_balancing_topk_gb300 import synth

from gpu_util import DEV, to_dev, to_np

pytestmark = pytest.mark.gpu

REL = 1e-6


def check(se, home, slots, E, status=None):
    st_ref, h_ref, s_ref = oracle.reduce_grad(se, home, slots, E)
    hd, sd = to_dev(home), to_dev(slots)
    mep.mep_reduce_grad(to_dev(se) if isinstance(se, np.ndarray) else se, hd, sd, status, E)
    torch.cuda.synchronize()
    h_got, s_got = to_np(hd), to_np(sd)
    # per-element bound from the magnitudes of the summed terms
    mag = np.abs(home).astype(np.float64)
    se_flat = np.asarray(se).reshape(-1)
    for s_idx, e in enumerate(se_flat):
        if e >= 0:
            mag[e] += np.abs(slots[s_idx])
    assert (np.abs(h_got.astype(np.float64) - h_ref) <= REL * mag).all()
    np.testing.assert_array_equal(s_got, s_ref)
    return h_got, h_ref


def test_reduce_grad_config_plan_map():
    """E=64, R=8, B=8, H=2048, H'=1408, slot map from a plan of the E=64,
    K=6, S=4096 workload (maxvio 0.5)."""
    s = synth.MEDIUM
    idx, _ = synth.routing(s, seed=0, alpha=0.075684)
    p = mep.mep_plan(to_dev(idx), s.R, s.S, s.K, s.E, s.B)
    ref_plan = oracle.plan(idx, s.R, s.S, s.K, s.E, s.B)
    torch.cuda.synchronize()
    se = to_np(p.slot_expert)
    np.testing.assert_array_equal(se, ref_plan["slot_expert"])
    HHp = synth.GRAD_H * synth.GRAD_HP
    home, slots = synth.grads(synth.GRAD_E, synth.GRAD_R, synth.GRAD_B, HHp, seed=0)
    h_got, h_ref = check(se, home, slots, synth.GRAD_E, p.status)
    print(f"slots used {(se >= 0).sum()}, exact {np.mean(h_got == h_ref):.6f}")
    assert (h_got == h_ref).all()


def test_reduce_grad_all_slots_used():
    E, R, B = synth.GRAD_E, synth.GRAD_R, synth.GRAD_B
    HHp = synth.GRAD_H * synth.GRAD_HP
    se = synth.full_slot_map(E, R, B, seed=0)
    home, slots = synth.grads(E, R, B, HHp, seed=1)
    h_got, h_ref = check(se, home, slots, E)
    assert (h_got == h_ref).all()


def test_reduce_grad_many_slots_per_expert():
    # one expert replicated on every slot of every rank: a 32-term ordered sum
    E, R, B, HHp = 8, 8, 4, 4096 + 4
    se = np.full((R, B), 3, dtype=np.int32)
    se[2, 1] = 5
    se[7, 3] = -1
    rng = np.random.default_rng(0)
    home = rng.standard_normal((E, HHp)).astype(np.float32)
    slots = (rng.standard_normal((R * B, HHp)) * 10.0 ** rng.integers(-4, 4, (R * B, 1))).astype(np.float32)
    h_got, h_ref = check(se, home, slots, E)
    assert (h_got == h_ref).all()


# 1, 3, 1001, 4097: single floats; 12, 4100: 16-byte vectors; 4104: 32-byte
@pytest.mark.parametrize("HHp", [1, 3, 12, 1001, 4097, 4100, 4104])
def test_reduce_grad_ragged_sizes(HHp):
    E, R, B = 6, 3, 2
    se = np.array([[1, 4], [0, -1], [4, 2]], dtype=np.int32)
    rng = np.random.default_rng(HHp)
    home = rng.standard_normal((E, HHp)).astype(np.float32)
    slots = rng.standard_normal((R * B, HHp)).astype(np.float32)
    h_got, h_ref = check(se, home, slots, E)
    assert (h_got == h_ref).all()


@pytest.mark.parametrize("shift", [4, 8], ids=["16B_aligned", "32B_aligned"])
def test_reduce_grad_buffer_alignment(shift):
    """Buffers that start 16 but not 32 bytes into an allocation take the
    16-byte path; the result is the same either way."""
    E, R, B, HHp = 5, 2, 3, 4104
    se = np.array([[3, 0, -1], [3, 4, 1]], dtype=np.int32)
    rng = np.random.default_rng(shift)
    home = rng.standard_normal((E, HHp)).astype(np.float32)
    slots = rng.standard_normal((R * B, HHp)).astype(np.float32)
    st_ref, h_ref, s_ref = oracle.reduce_grad(se, home, slots, E)
    hbuf = torch.zeros(E * HHp + 8, dtype=torch.float32, device=DEV)
    sbuf = torch.zeros(R * B * HHp + 8, dtype=torch.float32, device=DEV)
    hd = hbuf[shift:shift + E * HHp].view(E, HHp)
    sd = sbuf[shift:shift + R * B * HHp].view(R * B, HHp)
    hd.copy_(to_dev(home))
    sd.copy_(to_dev(slots))
    mep.mep_reduce_grad(to_dev(se), hd, sd, None, E)
    torch.cuda.synchronize()
    assert st_ref == "ok"
    np.testing.assert_array_equal(to_np(hd), h_ref)
    np.testing.assert_array_equal(to_np(sd), s_ref)
    assert (hbuf[:shift] == 0).all() and (sbuf[shift + R * B * HHp:] == 0).all()


def test_reduce_grad_order_fixture_values():
    # (1 + -1) + 2^-30 = 2^-30, the reverse order gives 0
    se = np.array([[1], [1]], dtype=np.int32)
    home = np.array([[5.0], [1.0]], dtype=np.float32)
    slots = np.array([[-1.0], [2.0 ** -30]], dtype=np.float32)
    h_got, _ = check(se, home, slots, 2)
    assert h_got[1, 0] == np.float32(2.0 ** -30)


def test_reduce_grad_bad_map_changes_nothing():
    E, R, B, HHp = 4, 2, 2, 64
    se = np.array([[0, 4], [1, -1]], dtype=np.int32)
    home = np.ones((E, HHp), np.float32)
    slots = np.ones((R * B, HHp), np.float32)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    hd, sd = to_dev(home), to_dev(slots)
    mep.mep_reduce_grad(to_dev(se), hd, sd, status, E)
    torch.cuda.synchronize()
    assert int(status.item()) == mep.STATUS_CODE["MEP_ERR_BAD_SLOT_MAP"]
    assert (to_np(hd) == 1).all() and (to_np(sd) == 1).all()


def test_reduce_grad_skips_on_status():
    E, R, B, HHp = 4, 2, 2, 64
    se = np.array([[0, 3], [1, -1]], dtype=np.int32)
    status = torch.full((1,), mep.STATUS_CODE["MEP_ERR_CAPACITY"], dtype=torch.int32, device=DEV)
    hd = torch.ones((E, HHp), dtype=torch.float32, device=DEV)
    sd = torch.ones((R * B, HHp), dtype=torch.float32, device=DEV)
    mep.mep_reduce_grad(to_dev(se), hd, sd, status, E)
    torch.cuda.synchronize()
    assert (hd == 1).all() and (sd == 1).all()
