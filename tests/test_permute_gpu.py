"""GPU parity of mep_dispatch / mep_combine against the CPU oracle.

dispatch is a bit copy: compared bit-exactly. combine accumulates in fp32
with one fused multiply-add per k in k order and rounds to nearest-even
bf16, exactly as the oracle does, so it is expected bit-exact; the test bar
is at most 1 bf16 ulp per element (the stated tolerance) and the exact
match rate is reported.
"""

import numpy as np
import pytest
import torch

import load_balancing_topk_gb300 as mep
import oracle
from load_balancing_topk_gb300 import synth

from gpu_util import DEV, bf16_ulp_diff, to_dev, to_np

pytestmark = pytest.mark.gpu

COMBINE_MAX_ULP = 1


def plan_both(s, **kw):
    idx, w = synth.routing(s, seed=kw.pop("seed", 0), **kw)
    ref = oracle.plan(idx, s.R, s.S, s.K, s.E, s.B)
    assert ref["status"] == "ok"
    p = mep.mep_plan(to_dev(idx), s.R, s.S, s.K, s.E, s.B)
    return idx, w, ref, p


SHAPES = [
    synth.TINY,
    synth.Shape(R=4, E=12, K=3, S=1000, H=264, B=9),      # several tiles, ragged
    synth.Shape(R=3, E=9, K=2, S=333, H=9000, B=6),       # 18000-byte rows: 2 chunks, ragged
    synth.Shape(R=2, E=4, K=1, S=100, H=8, B=2),          # 16-byte rows
    synth.Shape(R=2, E=16, K=10, S=150, H=64, B=8),       # K = 10: generic combine path
    synth.Shape(R=2, E=80, K=40, S=50, H=32, B=40),       # K > 32: two rows per lane
    synth.Shape(R=4, E=128, K=64, S=24, H=40, B=16),      # K = 64, the limit
    synth.Shape(R=2, E=8, K=4, S=96, H=4160, B=4),        # 260 32-byte vectors a row: 16 per lane, ragged
    synth.Shape(R=2, E=16, K=8, S=128, H=7168, B=8),      # K = 8 at H = 7168: the large workload's kernels
    synth.Shape(R=8, E=256, K=8, S=256, H=7168, B=32),    # the large workload's shape with S = 256
]


@pytest.mark.parametrize("s", SHAPES, ids=lambda s: f"R{s.R}E{s.E}K{s.K}S{s.S}H{s.H}")
def test_dispatch_and_combine_match_oracle(s):
    idx, w, ref, p = plan_both(s, alpha=1.0)
    x = synth.hidden(s, seed=1)
    buf = mep.mep_dispatch(to_dev(x), p.dst_pos, p.status, s.R, s.S, s.K)
    y = synth.expert_out(s, seed=2)
    out = mep.mep_combine(to_dev(y), to_dev(w), p.dst_pos, p.status, s.R, s.S, s.K)
    torch.cuda.synchronize()
    assert int(p.status.item()) == 0
    np.testing.assert_array_equal(to_np(buf), oracle.dispatch(x, ref["dst_pos"], s.A))
    want = oracle.combine(y, w, ref["dst_pos"])
    got = to_np(out)
    assert bf16_ulp_diff(got, want).max() <= COMBINE_MAX_ULP
    exact = float(np.mean(got == want))
    print(f"combine exact match rate {exact:.6f}")
    assert exact == 1.0  # same arithmetic, same order


def test_medium_full_parity():
    s = synth.MEDIUM
    idx, w, ref, p = plan_both(s, alpha=0.075684)
    x = synth.hidden(s, seed=0)
    xd = to_dev(x)
    buf = mep.mep_dispatch(xd, p.dst_pos, p.status, s.R, s.S, s.K)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_np(buf), oracle.dispatch(x, ref["dst_pos"], s.A))
    del buf
    y = synth.expert_out(s, seed=0)
    out = mep.mep_combine(to_dev(y), to_dev(w), p.dst_pos, p.status, s.R, s.S, s.K)
    torch.cuda.synchronize()
    want = oracle.combine(y, w, ref["dst_pos"])
    got = to_np(out)
    assert bf16_ulp_diff(got, want).max() <= COMBINE_MAX_ULP
    assert (got == want).all()


@pytest.mark.parametrize("name,kw", [
    ("large", dict(alpha=0.195312)),
    ("large", dict(kind="round_robin")),
    ("stress", dict(alpha=1.2, kind="hot")),
])
def test_full_size_dispatch_and_combine(name, kw):
    """Full-size launches (the configuration the benchmark times): every
    buffer row is checked against the oracle's plan, then combine runs on
    independent expert outputs y (not the dispatched copies, whose K rows per
    token are equal) and every output element is compared with the oracle's
    combine: a wrong row or a weight paired with the wrong k shows up."""
    s = synth.SHAPES[name]
    idx, w, ref, p = plan_both(s, **kw)
    x = synth.hidden(s, seed=0)
    xd = to_dev(x)
    buf = mep.mep_dispatch(xd, p.dst_pos, p.status, s.R, s.S, s.K)
    torch.cuda.synchronize()
    assert int(p.status.item()) == 0
    np.testing.assert_array_equal(to_np(p.dst_pos), ref["dst_pos"])
    # every row of the [R*S*K, H] buffer holds the token the oracle puts there
    src_tok = np.empty(s.A, dtype=np.int64)
    src_tok[ref["dst_pos"].reshape(-1)] = np.repeat(np.arange(s.N), s.K)
    st = torch.from_numpy(src_tok).to(DEV)
    for lo in range(0, s.A, 1 << 16):
        hi = min(s.A, lo + (1 << 16))
        assert torch.equal(buf[lo:hi].view(torch.int16), xd[st[lo:hi]].view(torch.int16)), lo
    del xd, st
    # combine of independent expert outputs, written into the same buffer
    y = synth.expert_out(s, seed=5)
    for lo in range(0, s.A, 1 << 16):
        hi = min(s.A, lo + (1 << 16))
        buf[lo:hi].copy_(to_dev(y[lo:hi]))
    out = mep.mep_combine(buf, to_dev(w), p.dst_pos, p.status, s.R, s.S, s.K)
    torch.cuda.synchronize()
    del buf
    want = oracle.combine(y, w, ref["dst_pos"])
    got = to_np(out)
    assert bf16_ulp_diff(got, want).max() <= COMBINE_MAX_ULP
    exact = float(np.mean(got == want))
    print(f"{name}: combine exact match rate {exact:.6f} over {got.size} elements")
    assert exact == 1.0


def test_k1_unit_weight_round_trip_is_identity():
    s = synth.Shape(R=4, E=8, K=1, S=2000, H=512, B=6)
    idx, _, ref, p = plan_both(s, alpha=2.0)
    x = to_dev(synth.hidden(s, seed=3))
    buf = mep.mep_dispatch(x, p.dst_pos, p.status, s.R, s.S, s.K)
    out = mep.mep_combine(buf, torch.ones((s.N, 1), dtype=torch.float32, device=DEV), p.dst_pos,
                          p.status, s.R, s.S, s.K)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), x.view(torch.int16))


def test_nonzero_status_makes_steps_no_ops():
    s = synth.TINY
    idx, w, ref, p = plan_both(s, alpha=1.0)
    x = to_dev(synth.hidden(s, seed=0))
    status = torch.full((1,), mep.STATUS_CODE["MEP_ERR_CAPACITY"], dtype=torch.int32, device=DEV)
    buf = torch.zeros((s.A, s.H), dtype=torch.bfloat16, device=DEV)
    mep.mep_dispatch(x, p.dst_pos, status, s.R, s.S, s.K, buf=buf)
    out = torch.zeros((s.N, s.H), dtype=torch.bfloat16, device=DEV)
    mep.mep_combine(buf, to_dev(w), p.dst_pos, status, s.R, s.S, s.K, out=out)
    torch.cuda.synchronize()
    assert (buf.view(torch.int16) == 0).all() and (out.view(torch.int16) == 0).all()


def test_bad_positions_are_reported_and_skipped():
    s = synth.Shape(R=2, E=4, K=2, S=64, H=64, B=2)
    idx, w, ref, p = plan_both(s, alpha=0.5)
    dst = p.dst_pos.clone()
    dst[7, 1] = s.A          # one past the end
    dst[9, 0] = -1
    x = to_dev(synth.hidden(s, seed=0))
    for fn in ("dispatch", "combine"):
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        buf = torch.zeros((s.A + 8, s.H), dtype=torch.bfloat16, device=DEV)  # guard rows
        if fn == "dispatch":
            mep.mep_dispatch(x, dst, status, s.R, s.S, s.K, buf=buf[: s.A])
            torch.cuda.synchronize()
            assert (buf[s.A:].view(torch.int16) == 0).all()
        else:
            out = torch.zeros((s.N, s.H), dtype=torch.bfloat16, device=DEV)
            mep.mep_combine(buf[: s.A], to_dev(w), dst, status, s.R, s.S, s.K, out=out)
            torch.cuda.synchronize()
        assert int(status.item()) == mep.STATUS_CODE["MEP_ERR_BAD_POSITION"]


def test_null_status_is_allowed():
    s = synth.TINY
    idx, w, ref, p = plan_both(s, alpha=1.0)
    x = synth.hidden(s, seed=0)
    buf = mep.mep_dispatch(to_dev(x), p.dst_pos, None, s.R, s.S, s.K)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_np(buf), oracle.dispatch(x, ref["dst_pos"], s.A))
