"""GPU parity of mep_grouped_gemm (tcgen05 + TMA) against the CPU oracle.

The grouped expert product: group j of rank r (its rows given by
cu_seqlens) times weight row j of the [E+B, H, H'] tensor -- w_home[j] below
E, the rank's prefetch slot w_slot[r, j - E] above ("月之暗面开源MoonEP：面向MoE
训练的专家并行通信库", section 内存契约与权重布局).

Two bars:
* integer-valued inputs (|x|, |w| <= 2, so every partial sum is an integer
  below 2^24 and exact in fp32 whatever the tensor cores' order): the bf16
  output must equal the oracle's exact sum rounded to nearest-even, bit for bit;
* normal inputs: the tensor cores' fp32 accumulation order and internal
  precision are unspecified, so the bound assumes only that each of the H
  additions has relative error <= 2^-23, then one bf16 rounding:
  |y - exact| <= 2^-8 |exact| + (1 + 2^-8) H 2^-23 sum_h |x w|.
"""

import numpy as np
import pytest
import torch

import load_balancing_topk_gb300 as mep
import oracle
from load_balancing_topk_gb300 import synth

from gpu_util import DEV, to_dev, to_np

pytestmark = pytest.mark.gpu


def _int_bf16(shape, seed, tag):
    return oracle.f32_to_bf16(synth.integer_valued(shape, seed, -2, 2, tag=tag))


def _normal_bf16(shape, seed, tag):
    rows = int(np.prod(shape[:-1]))
    return synth.bf16_normal(rows, shape[-1], seed=seed, tag=tag).reshape(shape)


def _inputs(R, SK, E, B, H, Hp, seed, integer):
    make = _int_bf16 if integer else _normal_bf16
    x = make((R * SK, H), seed, 70)
    wh = make((E, H, Hp), seed, 71)
    ws = make((R, B, H, Hp), seed, 72) if B > 0 else np.zeros((R, 0, H, Hp), np.uint16)
    return x, wh, ws


def _run(x, cu, wh, ws, R, S, K, status=None):
    E, H, Hp = wh.shape
    B = cu.shape[1] - E
    st = status if status is not None else torch.zeros(1, dtype=torch.int32, device=DEV)
    y = mep.mep_grouped_gemm(to_dev(x), to_dev(cu), to_dev(wh), to_dev(ws) if B > 0 else None,
                             st, R, S, K)
    torch.cuda.synchronize()
    return y, st


def _check(y_bits, x, cu, wh, ws, integer, rows=None):
    ref = oracle.grouped_gemm(x, cu, wh, ws, rows=rows)
    if integer:
        np.testing.assert_array_equal(y_bits, oracle.f32_to_bf16(ref.astype(np.float32)))
        return
    mag = oracle.grouped_gemm(x & 0x7FFF, cu, wh & 0x7FFF, ws & 0x7FFF, rows=rows)
    H = x.shape[1]
    got = oracle.bf16_to_f32(y_bits).astype(np.float64)
    tol = 2.0 ** -8 * np.abs(ref) + (1 + 2.0 ** -8) * H * 2.0 ** -23 * mag
    err = np.abs(got - ref)
    assert np.isfinite(got).all()
    assert (err <= tol).all(), float((err / np.maximum(tol, 1e-30)).max())


# hand-made group tables: (R, S, K, E, B, H, Hp, cu rows)
MANUAL = {
    "one_tile": (1, 64, 2, 1, 0, 64, 256, [[128]]),
    "k_steps": (1, 64, 2, 1, 0, 512, 256, [[128]]),
    "ragged_n": (1, 64, 2, 1, 0, 128, 200, [[128]]),
    "two_n_blocks": (1, 64, 2, 1, 0, 128, 448, [[128]]),
    "ragged_m": (1, 100, 2, 2, 0, 128, 128, [[72, 200]]),
    "slots_and_empty": (2, 96, 2, 3, 2, 192, 64, [[0, 70, 70, 150, 192], [30, 30, 31, 31, 192]]),
    "small_buffer": (1, 16, 2, 2, 0, 64, 64, [[5, 32]]),
    "narrow_ragged_n": (1, 64, 2, 1, 0, 128, 72, [[128]]),   # last block: N = 128 MMAs, 72 columns
    "deep_k": (1, 96, 2, 2, 0, 7168, 136, [[100, 192]]),      # H = 7168: 112 K steps, ragged rows
}


@pytest.mark.parametrize("integer", [True, False], ids=["int", "normal"])
@pytest.mark.parametrize("name", list(MANUAL))
def test_manual_tables(name, integer):
    R, S, K, E, B, H, Hp, cu = MANUAL[name]
    cu = np.array(cu, np.int32)
    x, wh, ws = _inputs(R, S * K, E, B, H, Hp, seed=1, integer=integer)
    y, st = _run(x, cu, wh, ws, R, S, K)
    assert int(st.item()) == 0
    _check(to_np(y), x, cu, wh, ws, integer)


PLANNED = [
    # (shape, H', alpha, fallback)
    (synth.Shape(R=2, E=8, K=2, S=64, H=128, B=4), 128, 1.0, False),
    (synth.Shape(R=4, E=16, K=4, S=512, H=512, B=4), 320, 1.0, False),
    (synth.Shape(R=4, E=16, K=4, S=256, H=256, B=1), 136, 1.5, True),
    (synth.Shape(R=8, E=64, K=6, S=300, H=256, B=8), 1408, 0.5, False),
]


@pytest.mark.parametrize("integer", [True, False], ids=["int", "normal"])
@pytest.mark.parametrize("case", PLANNED, ids=lambda c: f"R{c[0].R}E{c[0].E}K{c[0].K}S{c[0].S}H{c[0].H}Hp{c[1]}"
                         + ("fb" if c[3] else ""))
def test_planned_groups(case, integer):
    s, Hp, alpha, fallback = case
    idx, _ = synth.routing(s, seed=0, alpha=alpha)
    p = oracle.plan(idx, s.R, s.S, s.K, s.E, s.B, fallback=fallback)
    assert p["status"] == "ok"
    cu = p["cu_seqlens"]
    x, wh, ws = _inputs(s.R, s.S * s.K, s.E, s.B, s.H, Hp, seed=2, integer=integer)
    y, st = _run(x, cu, wh, ws, s.R, s.S, s.K)
    assert int(st.item()) == 0
    _check(to_np(y), x, cu, wh, ws, integer)


@pytest.mark.parametrize("draw", range(24))
def test_random_group_tables(draw):
    """Any valid table: per rank, E+B groups cut at random points of the
    rank's S*K rows (empty groups included), H and H' across their ranges,
    slot rows on some draws; integer inputs, so the result is exact."""
    g = np.random.default_rng([draw, 1408])
    R = int(g.choice([1, 2, 3, 4]))
    E = int(g.integers(1, 9))
    B = int(g.integers(0, 4))
    S, K = int(g.integers(1, 200)), int(g.integers(1, 5))
    H = int(g.choice([64, 128, 192, 320, 1024]))
    Hp = int(g.choice([8, 24, 64, 136, 264, 520, 1408]))
    SK, G = S * K, E + B
    cuts = np.sort(g.integers(0, SK + 1, size=(R, G - 1)), axis=1)
    cu = np.concatenate([cuts, np.full((R, 1), SK)], axis=1).astype(np.int32)
    x, wh, ws = _inputs(R, SK, E, B, H, Hp, seed=draw, integer=True)
    y, st = _run(x, cu, wh, ws, R, S, K)
    assert int(st.item()) == 0
    _check(to_np(y), x, cu, wh, ws, True)


def test_gemm_on_device_plan_and_dispatch():
    """mep_plan -> mep_dispatch -> mep_prefetch -> mep_grouped_gemm: every
    assignment (t, k) meets its routed expert's weights, bit-exact on integers."""
    s = synth.Shape(R=4, E=16, K=4, S=256, H=256, B=4)
    Hp = 192
    idx, _ = synth.routing(s, seed=3, alpha=1.0)
    p = mep.mep_plan(to_dev(idx), s.R, s.S, s.K, s.E, s.B)
    hidden = _int_bf16((s.N, s.H), 3, 73)
    wh = _int_bf16((s.E, s.H, Hp), 3, 74)
    buf = mep.mep_dispatch(to_dev(hidden), p.dst_pos, p.status, s.R, s.S, s.K)
    wh_d = to_dev(wh)
    ws_d = torch.zeros((s.R, s.B, s.H, Hp), dtype=torch.bfloat16, device=DEV)
    mep.mep_prefetch(p.slot_expert, wh_d, ws_d, p.status, s.E)
    y = mep.mep_grouped_gemm(buf, p.cu_seqlens, wh_d, ws_d, p.status, s.R, s.S, s.K)
    torch.cuda.synchronize()
    assert int(p.status.item()) == 0
    yb, dst = to_np(y), to_np(p.dst_pos)
    for t in range(0, s.N, 7):
        for k in range(s.K):
            exact = oracle.bf16_to_f32(hidden[t]).astype(np.float64) @ \
                oracle.bf16_to_f32(wh[idx[t, k]]).astype(np.float64)
            np.testing.assert_array_equal(yb[dst[t, k]], oracle.f32_to_bf16(exact.astype(np.float32)))


def test_medium_full_size_sampled_rows():
    """The full layer: R8 E64 K6 S4096, H 2048 -> H' 1408, B 8; the first and
    last row of every non-empty group plus random rows against the oracle."""
    s = synth.MEDIUM
    Hp = synth.GRAD_HP
    idx, _ = synth.routing(s, seed=0, alpha=0.075684)
    p = oracle.plan(idx, s.R, s.S, s.K, s.E, s.B)
    cu = p["cu_seqlens"]
    SK = s.S * s.K
    x, wh, ws = _inputs(s.R, SK, s.E, s.B, s.H, Hp, seed=4, integer=False)
    y, st = _run(x, cu, wh, ws, s.R, s.S, s.K)
    assert int(st.item()) == 0
    rows = set()
    for r in range(s.R):
        lo = 0
        for j in range(s.E + s.B):
            hi = int(cu[r, j])
            if hi > lo:
                rows.update((r * SK + lo, r * SK + hi - 1))
            lo = hi
    g = np.random.default_rng(5)
    rows.update(g.choice(s.R * SK, size=256, replace=False).tolist())
    rows = np.array(sorted(rows), np.int64)
    yb = to_np(y)
    _check(yb[rows], x, cu, wh, ws, integer=False, rows=rows)


def test_status_and_bad_tables():
    R, S, K, E, B, H, Hp = 2, 64, 2, 4, 2, 64, 64
    x, wh, ws = _inputs(R, S * K, E, B, H, Hp, seed=6, integer=True)
    good = np.array([[30, 60, 90, 128, 128, 128]] * R, np.int32)
    # a nonzero status on entry: nothing is written
    st = torch.full((1,), mep.STATUS_CODE["MEP_ERR_CAPACITY"], dtype=torch.int32, device=DEV)
    y0 = torch.full((R * S * K, Hp), 7.0, dtype=torch.bfloat16, device=DEV)
    mep.mep_grouped_gemm(to_dev(x), to_dev(good), to_dev(wh), to_dev(ws), st, R, S, K, y=y0)
    torch.cuda.synchronize()
    assert (y0 == 7.0).all() and int(st.item()) == mep.STATUS_CODE["MEP_ERR_CAPACITY"]
    # malformed tables: MEP_ERR_BAD_SEQLENS, nothing written
    for bad in ([30, 20, 90, 128, 128, 128], [30, 60, 90, 128, 128, 127], [-1, 60, 90, 128, 128, 128]):
        cu = good.copy()
        cu[1] = bad
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        y1 = torch.full((R * S * K, Hp), 7.0, dtype=torch.bfloat16, device=DEV)
        mep.mep_grouped_gemm(to_dev(x), to_dev(cu), to_dev(wh), to_dev(ws), st, R, S, K, y=y1)
        torch.cuda.synchronize()
        assert int(st.item()) == mep.STATUS_CODE["MEP_ERR_BAD_SEQLENS"]
        assert (y1 == 7.0).all()


def test_host_rejects_bad_sizes():
    x = torch.zeros((128, 96), dtype=torch.bfloat16, device=DEV)   # H % 64 != 0
    cu = torch.tensor([[128]], dtype=torch.int32, device=DEV)
    wh = torch.zeros((1, 96, 64), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(mep.MepError):
        mep.mep_grouped_gemm(x, cu, wh, None, None, 1, 64, 2)
    x = torch.zeros((128, 64), dtype=torch.bfloat16, device=DEV)
    wh = torch.zeros((1, 64, 68), dtype=torch.bfloat16, device=DEV)  # H' % 8 != 0
    with pytest.raises(mep.MepError):
        mep.mep_grouped_gemm(x, cu, wh, None, None, 1, 64, 2)
