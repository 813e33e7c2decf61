"""Randomised parity sweeps of the row kernels against the oracle.

- permute chain: random ranks, experts, K up to 12, tokens and row widths
  (8 to 7168 elements), through plan -> dispatch -> combine of independent
  expert outputs -> dispatch backward -> combine backward. Every other draw
  places hidden, y and dout 16 bytes into their buffers, so the kernels take
  their 16-byte vector forms; the others are 32-byte aligned.
- slot maps: random maps with holes and experts repeated across slots
  through reduce_grad (fp32 sums in rank, slot order) and prefetch (byte
  copy), also with and without a 16-byte offset.

Integer and copy work and the in-order fp32 sums are compared bit for bit;
dw (the kernel's own fp32 summation order) within the bound derived in
test_backward_gpu.
"""

import numpy as np
import pytest
import torch

import load_balancing_topk_gb300 as mep
import oracle
from load_balancing_topk_gb300 import synth

from gpu_util import DEV, to_dev, to_np
from test_backward_gpu import dw_bound

pytestmark = pytest.mark.gpu


def _placed(a_np, off_elems):
    """A device copy of a_np that starts off_elems elements into its buffer."""
    t = to_dev(a_np)
    if off_elems == 0:
        return t
    big = torch.empty(t.numel() + off_elems, dtype=t.dtype, device=DEV)
    v = big[off_elems:].view(t.shape)
    v.copy_(t)
    return v


@pytest.mark.parametrize("draw", range(40))
def test_permute_chain_fuzz(draw):
    g = np.random.default_rng([draw, 777])
    R = int(g.choice([1, 2, 4, 8, 16]))
    E = R * int(g.integers(1, 13))
    K = int(g.integers(1, min(12, E) + 1))
    S = int(g.integers(1, 400))
    H = int(g.choice([8, 24, 64, 136, 1000, 2056, 4104, 7168]))
    B = int(g.integers(2, 17))
    s = synth.Shape(R=R, E=E, K=K, S=S, H=H, B=B)
    idx, w = synth.routing(s, seed=draw, alpha=float(g.uniform(0, 1.2)))
    ref = oracle.plan(idx, R, S, K, E, B)
    if ref["status"] != "ok":
        pytest.skip("the draw needs more than B slots")
    p = mep.mep_plan(to_dev(idx), R, S, K, E, B)
    off = 8 if draw % 2 else 0          # 16 bytes of bf16
    dst = ref["dst_pos"]
    hidden = synth.bf16_normal(s.N, H, seed=draw, tag=90)
    buf = mep.mep_dispatch(_placed(hidden, off), p.dst_pos, p.status, R, S, K)
    y = synth.bf16_normal(s.A, H, seed=draw, tag=93)
    y_d, w_d = _placed(y, off), to_dev(w)
    out = mep.mep_combine(y_d, w_d, p.dst_pos, p.status, R, S, K)
    dh = mep.mep_dispatch_backward(y_d, p.dst_pos, p.status, R, S, K)
    dout = synth.bf16_normal(s.N, H, seed=draw, tag=94)
    dout_d = _placed(dout, off)
    dy, dw = mep.mep_combine_backward(dout_d, y_d, w_d, p.dst_pos, p.status, R, S, K)
    torch.cuda.synchronize()
    assert int(p.status.item()) == 0
    np.testing.assert_array_equal(to_np(p.dst_pos), dst)
    np.testing.assert_array_equal(to_np(buf), oracle.dispatch(hidden, dst, s.A))
    np.testing.assert_array_equal(to_np(out), oracle.combine(y, w, dst))
    np.testing.assert_array_equal(to_np(dh), oracle.dispatch_backward(y, dst))
    dy_ref, dw_ref = oracle.combine_backward(dout, y, w, dst)
    np.testing.assert_array_equal(to_np(dy), dy_ref)
    err = np.abs(to_np(dw).astype(np.float64) - dw_ref)
    assert (err <= dw_bound(dout_d, y_d, p.dst_pos, H)).all()


@pytest.mark.parametrize("draw", range(40))
def test_slot_map_fuzz(draw):
    g = np.random.default_rng([draw, 4242])
    R = int(g.choice([1, 2, 3, 8, 16]))
    B = int(g.integers(1, 9))
    E = int(g.integers(1, 70))
    HHp = int(g.choice([4, 12, 100, 1000, 4100, 4104, 65544]))
    se = g.integers(-1, E, size=(R, B)).astype(np.int32)   # holes and repeated experts
    home = g.standard_normal((E, HHp)).astype(np.float32) * np.float32(1e-3)
    slot = g.standard_normal((R * B, HHp)).astype(np.float32) * np.float32(1e-3)
    off = 4 if draw % 2 else 0          # 16 bytes of fp32
    home_d, slot_d = _placed(home, off), _placed(slot, off)
    mep.mep_reduce_grad(to_dev(se), home_d, slot_d, None, E)
    n_el = int(g.choice([8, 24, 520, 4104]))
    wh = g.integers(0, 65535, size=(E, n_el), dtype=np.uint16)
    ws = g.integers(0, 65535, size=(R * B, n_el), dtype=np.uint16)
    wh_d, ws_d = _placed(wh, 2 * off), _placed(ws, 2 * off)
    mep.mep_prefetch(to_dev(se), wh_d, ws_d, None, E)
    torch.cuda.synchronize()
    _, home_ref, slot_ref = oracle.reduce_grad(se, home, slot, E)
    np.testing.assert_array_equal(to_np(home_d), home_ref)
    np.testing.assert_array_equal(to_np(slot_d), slot_ref)
    _, ws_ref = oracle.prefetch(se, wh, ws, E)
    np.testing.assert_array_equal(to_np(ws_d), ws_ref)
    np.testing.assert_array_equal(to_np(wh_d), wh)
