"""Randomised shapes through the whole library against the oracle.

Each seed draws a small layer (ranks, experts, K, tokens, H, H', slots,
routing skew, training or inference planner) and runs plan -> dispatch ->
combine -> prefetch -> grouped GEMM -> reduce_grad on the GPU and in the
oracle. Integer work is compared bit for bit; the grouped GEMM runs on
integer-valued inputs so that its fp32 sums are exact in any order; combine
and reduce_grad use the same operations in the same order on both sides.
A plan that needs more than B slots must report MEP_ERR_CAPACITY, as the
oracle does, and leave the later steps as no-ops.
"""

import numpy as np
import pytest
import torch

import load_balancing_topk_gb300 as mep
import oracle
from load_balancing_topk_gb300 import synth

from gpu_util import DEV, to_dev, to_np

pytestmark = pytest.mark.gpu


def _draw(seed):
    g = np.random.default_rng([seed, 2024])
    R = int(g.choice([1, 2, 3, 4, 8]))
    E = R * int(g.integers(1, 17))
    K = int(g.integers(1, min(8, E) + 1))
    S = int(g.integers(1, 301))
    H = int(g.choice([64, 128, 192]))
    Hp = int(g.choice([8, 24, 64, 136, 264]))
    B = int(g.integers(0, 7))
    alpha = float(g.uniform(0.0, 2.0))
    fallback = bool(g.integers(0, 2))
    return R, E, K, S, H, Hp, B, alpha, fallback


@pytest.mark.parametrize("seed", range(16))
def test_random_layer_chain(seed):
    R, E, K, S, H, Hp, B, alpha, fallback = _draw(seed)
    s = synth.Shape(R=R, E=E, K=K, S=S, H=H, B=B)
    idx, w = synth.routing(s, seed=seed, alpha=alpha)
    ref = oracle.plan(idx, R, S, K, E, B, fallback=fallback)
    plan_fn = mep.mep_plan_remote_fallback if fallback else mep.mep_plan
    p = plan_fn(to_dev(idx), R, S, K, E, B)
    torch.cuda.synchronize()
    if ref["status"] != "ok":
        assert ref["status"] == "capacity"
        assert int(p.status.item()) == mep.STATUS_CODE["MEP_ERR_CAPACITY"]
        return
    assert int(p.status.item()) == 0
    for name in ("cu_seqlens", "slot_expert", "dst_pos"):
        np.testing.assert_array_equal(to_np(getattr(p, name)), ref[name], err_msg=name)

    # dispatch / combine
    hidden = synth.bf16_normal(s.N, H, seed=seed, tag=90)
    buf = mep.mep_dispatch(to_dev(hidden), p.dst_pos, p.status, R, S, K)
    torch.cuda.synchronize()
    buf_r = oracle.dispatch(hidden, ref["dst_pos"], s.A)
    np.testing.assert_array_equal(to_np(buf), buf_r)
    # combine of independent expert outputs (a token's K dispatched rows are
    # equal copies, which would hide a row or weight paired with the wrong k)
    y_e = synth.bf16_normal(s.A, H, seed=seed, tag=93)
    buf.copy_(to_dev(y_e))
    out = mep.mep_combine(buf, to_dev(w), p.dst_pos, p.status, R, S, K)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_np(out), oracle.combine(y_e, w, ref["dst_pos"]))

    # prefetch + grouped GEMM on integer-valued rows and weights
    xi = oracle.f32_to_bf16(synth.integer_valued((s.A, H), seed, -2, 2, tag=91))
    wh = oracle.f32_to_bf16(synth.integer_valued((E, H, Hp), seed, -2, 2, tag=92))
    wh_d = to_dev(wh)
    ws_d = torch.zeros((R, B, H, Hp), dtype=torch.bfloat16, device=DEV) if B > 0 else None
    if B > 0:
        mep.mep_prefetch(p.slot_expert, wh_d, ws_d, p.status, E)
    y = mep.mep_grouped_gemm(to_dev(xi), p.cu_seqlens, wh_d, ws_d, p.status, R, S, K)
    torch.cuda.synchronize()
    ws_r = np.zeros((R, B, H, Hp), np.uint16)
    used = ref["slot_expert"] >= 0
    ws_r[used] = wh[ref["slot_expert"][used]]
    y_r = oracle.f32_to_bf16(oracle.grouped_gemm(xi, ref["cu_seqlens"], wh, ws_r).astype(np.float32))
    np.testing.assert_array_equal(to_np(y), y_r)

    # reduce_grad over this plan's slot map
    if B > 0:
        HHp = 40
        home, slots = synth.grads(E, R, B, HHp, seed=seed)
        home_d, slots_d = to_dev(home), to_dev(slots)
        mep.mep_reduce_grad(p.slot_expert, home_d, slots_d, p.status, E)
        torch.cuda.synchronize()
        st, h_r, s_r = oracle.reduce_grad(ref["slot_expert"], home, slots, E)
        assert st == "ok"
        np.testing.assert_array_equal(to_np(home_d), h_r)
        np.testing.assert_array_equal(to_np(slots_d), s_r)
