"""GPU parity of mep_dispatch_backward and mep_combine_backward against the
CPU oracle.

dhidden and dy are expected bit-exact: same fp32 operations in the same
order as the oracle. dw's fp32 summation order is the kernel's own (per lane,
then a warp butterfly), so it is checked against the oracle's fp64 dot
product within the bound that order guarantees. A lane's fma chain holds at
most n = ceil(H / (32 c)) * c products (c = 16 bf16 per 32-byte vector when
H % 16 == 0, else 8), and a 5-level butterfly follows: a summation tree of
height n + 4, so
|dw - exact| <= gamma_(n+4) * S <= (n + 5) * 2^-24 * S,
S = sum_h |dout[t,h] * y[dst_pos[t,k],h]|.
"""

import numpy as np
import pytest
import torch

import load_balancing_topk_gb300 as mep
import oracle
from load_balancing_topk_gb300 import synth

from gpu_util import DEV, to_dev, to_np

pytestmark = pytest.mark.gpu


def lane_chain(H):
    """Longest per-lane fma chain of the dw dot product."""
    c = 16 if H % 16 == 0 else 8
    return -(-H // (32 * c)) * c


def dw_bound(dout_d, y_d, dst_d, H):
    """Per-(t,k) bound (n + 5) * 2^-24 * sum_h |dout * y| computed on the GPU."""
    N, K = dst_d.shape
    out = torch.empty((N, K), dtype=torch.float64, device=DEV)
    for lo in range(0, N, 2048):
        hi = min(N, lo + 2048)
        d = dout_d[lo:hi].abs().double()
        yy = y_d[dst_d[lo:hi].reshape(-1).long()].abs().double().view(hi - lo, K, -1)
        out[lo:hi] = torch.einsum("th,tkh->tk", d, yy)
    return (out * ((lane_chain(H) + 5) * 2.0 ** -24)).cpu().numpy()


SHAPES = [
    synth.TINY,
    synth.Shape(R=4, E=12, K=3, S=1000, H=264, B=9),
    synth.Shape(R=2, E=16, K=8, S=700, H=1032, B=8),
    synth.Shape(R=2, E=4, K=1, S=100, H=8, B=2),
    synth.Shape(R=2, E=16, K=10, S=150, H=64, B=8),
    synth.Shape(R=2, E=80, K=40, S=50, H=32, B=40),
    synth.Shape(R=2, E=8, K=4, S=96, H=4096, B=4),   # 32-byte vectors in combine_backward
    synth.Shape(R=4, E=128, K=64, S=24, H=40, B=16),  # K = 64, the limit
    synth.Shape(R=2, E=16, K=8, S=128, H=7168, B=8),  # K = 8 at H = 7168 (32-byte vectors)
]


def _plan(s, seed=0, alpha=1.0):
    idx, w = synth.routing(s, seed=seed, alpha=alpha)
    ref = oracle.plan(idx, s.R, s.S, s.K, s.E, s.B)
    assert ref["status"] == "ok"
    p = mep.mep_plan(to_dev(idx), s.R, s.S, s.K, s.E, s.B)
    return w, ref, p


@pytest.mark.parametrize("s", SHAPES, ids=lambda s: f"R{s.R}E{s.E}K{s.K}S{s.S}H{s.H}")
def test_backward_matches_oracle(s):
    w, ref, p = _plan(s)
    dbuf = synth.bf16_normal(s.A, s.H, seed=1, tag=61)
    dout = synth.bf16_normal(s.N, s.H, seed=1, tag=62)
    y = synth.bf16_normal(s.A, s.H, seed=1, tag=63)
    dh = mep.mep_dispatch_backward(to_dev(dbuf), p.dst_pos, p.status, s.R, s.S, s.K)
    dout_d, y_d = to_dev(dout), to_dev(y)
    dy, dw = mep.mep_combine_backward(dout_d, y_d, to_dev(w), p.dst_pos, p.status, s.R, s.S, s.K)
    torch.cuda.synchronize()
    assert int(p.status.item()) == 0
    np.testing.assert_array_equal(to_np(dh), oracle.dispatch_backward(dbuf, ref["dst_pos"]))
    dy_ref, dw_ref = oracle.combine_backward(dout, y, w, ref["dst_pos"])
    np.testing.assert_array_equal(to_np(dy), dy_ref)
    err = np.abs(to_np(dw).astype(np.float64) - dw_ref)
    bound = dw_bound(dout_d, y_d, p.dst_pos, s.H)
    assert (err <= bound).all(), float((err / np.maximum(bound, 1e-300)).max())


def test_backward_medium_full():
    s = synth.MEDIUM
    w, ref, p = _plan(s, alpha=0.075684)
    dbuf = synth.bf16_normal(s.A, s.H, seed=2, tag=61)
    dh = mep.mep_dispatch_backward(to_dev(dbuf), p.dst_pos, p.status, s.R, s.S, s.K)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_np(dh), oracle.dispatch_backward(dbuf, ref["dst_pos"]))
    dout = synth.bf16_normal(s.N, s.H, seed=2, tag=62)
    dout_d, y_d = to_dev(dout), to_dev(dbuf)
    dy, dw = mep.mep_combine_backward(dout_d, y_d, to_dev(w), p.dst_pos, p.status, s.R, s.S, s.K)
    torch.cuda.synchronize()
    dy_ref, dw_ref = oracle.combine_backward(dout, dbuf, w, ref["dst_pos"])
    np.testing.assert_array_equal(to_np(dy), dy_ref)
    err = np.abs(to_np(dw).astype(np.float64) - dw_ref)
    bound = dw_bound(dout_d, y_d, p.dst_pos, s.H)
    ratio = float((err / np.maximum(bound, 1e-300)).max())
    print(f"dw max error / bound = {ratio:.3e}")
    assert ratio <= 1.0


def test_dispatch_backward_order_fixture_on_gpu():
    # rows 2^24, 1 + 2^-7, -2^24 summed in k order give 2.0 (bits 4000)
    dbuf = np.zeros((3, 8), np.uint16)
    dbuf[0, :], dbuf[1, :], dbuf[2, :] = 0x4B80, 0x3F81, 0xCB80
    dst = np.array([[0, 1, 2]], dtype=np.int32)
    dh = mep.mep_dispatch_backward(to_dev(dbuf), to_dev(dst), None, 1, 1, 3)
    torch.cuda.synchronize()
    assert (to_np(dh) == 0x4000).all()


def test_combine_backward_rounding_fixture_on_gpu():
    # w = 0x3f382ee7, dout = 0x3f83: the fp32 product sits on a bf16 tie -> 0x3f3c
    w = np.array([[0x3F382EE7]], dtype=np.uint32).view(np.float32)
    dout = np.full((1, 8), 0x3F83, np.uint16)
    y = np.zeros((1, 8), np.uint16)
    dy, dw = mep.mep_combine_backward(to_dev(dout), to_dev(y), to_dev(w),
                                      to_dev(np.zeros((1, 1), np.int32)), None, 1, 1, 1)
    torch.cuda.synchronize()
    assert (to_np(dy) == 0x3F3C).all() and float(dw.item()) == 0.0


def test_backward_no_op_on_status():
    s = synth.TINY
    w, ref, p = _plan(s)
    status = torch.full((1,), mep.STATUS_CODE["MEP_ERR_CAPACITY"], dtype=torch.int32, device=DEV)
    dh = torch.zeros((s.N, s.H), dtype=torch.bfloat16, device=DEV)
    mep.mep_dispatch_backward(torch.ones((s.A, s.H), dtype=torch.bfloat16, device=DEV), p.dst_pos,
                              status, s.R, s.S, s.K, dhidden=dh)
    dy = torch.zeros((s.A, s.H), dtype=torch.bfloat16, device=DEV)
    dw = torch.zeros((s.N, s.K), dtype=torch.float32, device=DEV)
    one = torch.ones((s.N, s.H), dtype=torch.bfloat16, device=DEV)
    mep.mep_combine_backward(one, dy.clone() + 1, to_dev(w), p.dst_pos, status, s.R, s.S, s.K,
                             dy=dy, dw=dw)
    torch.cuda.synchronize()
    assert (dh.view(torch.int16) == 0).all() and (dy.view(torch.int16) == 0).all()
    assert (dw == 0).all()
