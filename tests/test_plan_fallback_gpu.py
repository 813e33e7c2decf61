"""GPU parity of mep_plan_remote_fallback (the inference reading of the slot
budget) against the oracle's fallback plan: bit-exact counts, cu_seqlens,
slot table and destination rows, including ranks whose pieces overflow
their B slots into the experts' own rows."""

import numpy as np
import pytest
import torch

import load_balancing_topk_gb300 as mep
import oracle
from load_balancing_topk_gb300 import synth

from gpu_util import DEV, to_dev, to_np
from plan_checks import check_invariants_fallback

pytestmark = pytest.mark.gpu


def assert_fallback_plan_equal(idx, R, S, K, E, B):
    ref = oracle.plan(idx, R, S, K, E, B, fallback=True)
    p = mep.mep_plan_remote_fallback(to_dev(idx), R, S, K, E, B)
    torch.cuda.synchronize()
    assert ref["status"] == "ok" and int(p.status.item()) == 0
    got = dict(status="ok", counts=to_np(p.expert_counts), cu_seqlens=to_np(p.cu_seqlens),
               slot_expert=to_np(p.slot_expert), dst_pos=to_np(p.dst_pos))
    for k in ("counts", "cu_seqlens", "slot_expert", "dst_pos"):
        np.testing.assert_array_equal(got[k], ref[k], err_msg=k)
    check_invariants_fallback(got, idx, R, S, K, E, B)
    training = oracle.plan(idx, R, S, K, E, B)
    return p, training["status"] == "capacity"


@pytest.mark.parametrize("name,B,kw", [
    ("large", 4, dict(alpha=0.195312)),
    ("large", 3, dict(alpha=0.12207)),
    ("stress", 4, dict(alpha=1.2, kind="hot")),
    ("stress", 3, dict(alpha=1.2, kind="hot", placement="identity")),
    ("medium", 2, dict(alpha=0.3)),
])
def test_fallback_plan_on_inference_budgets(name, B, kw):
    s = synth.SHAPES[name]
    idx, _ = synth.routing(s, seed=0, **kw)
    _, needed = assert_fallback_plan_equal(idx, s.R, s.S, s.K, s.E, B)
    assert needed  # these budgets are too small for the training reading


def test_fallback_fixture_on_gpu():
    idx = np.array([[0, 1], [0, 2], [0, 1], [1, 0], [0, 5], [1, 3]], dtype=np.int32)
    p, needed = assert_fallback_plan_equal(idx, 3, 2, 2, 6, 1)
    assert needed
    np.testing.assert_array_equal(to_np(p.dst_pos).reshape(-1),
                                  [0, 4, 1, 5, 2, 9, 10, 3, 7, 8, 11, 6])


def test_fallback_random_sweep():
    rng = np.random.default_rng(7)
    n_needed = 0
    for i in range(50):
        R = int(rng.integers(2, 9))
        per = int(rng.integers(1, 6))
        E, K = R * per, int(rng.integers(1, min(R * per, 6) + 1))
        S = int(rng.integers(1, 800))
        B = int(rng.integers(0, 3))
        s = synth.Shape(R=R, E=E, K=K, S=S, H=8, B=B)
        idx, _ = synth.routing(s, seed=i, alpha=float(rng.uniform(0.5, 3)), placement="identity")
        _, needed = assert_fallback_plan_equal(idx, R, S, K, E, B)
        n_needed += needed
    assert n_needed > 20


def test_fallback_round_trip():
    s = synth.Shape(R=8, E=64, K=6, S=1000, H=256, B=2)
    idx, w = synth.routing(s, seed=3, alpha=0.4)
    ref = oracle.plan(idx, s.R, s.S, s.K, s.E, s.B, fallback=True)
    p = mep.mep_plan_remote_fallback(to_dev(idx), s.R, s.S, s.K, s.E, s.B)
    x = synth.hidden(s, seed=3)
    buf = mep.mep_dispatch(to_dev(x), p.dst_pos, p.status, s.R, s.S, s.K)
    out = mep.mep_combine(buf, to_dev(w), p.dst_pos, p.status, s.R, s.S, s.K)
    torch.cuda.synchronize()
    buf_ref = oracle.dispatch(x, ref["dst_pos"], s.A)
    np.testing.assert_array_equal(to_np(buf), buf_ref)
    np.testing.assert_array_equal(to_np(out), oracle.combine(buf_ref, w, ref["dst_pos"]))
