"""Pins for the oracle's grouped expert product (CPU only).

The grouped GEMM consumes one [E+B, H, H'] weight tensor per projection:
rows [0, E) are the experts' own weights, rows [E, E+B) the rank's prefetch
slots, and cu_seqlens says which buffer rows each weight row serves
("月之暗面开源MoonEP：面向MoE训练的专家并行通信库", section 内存契约与权重布局).
The oracle computes y[row] = x[row] @ W_j in double; these tests pin it to:

* a closed form: scaled identities give y[row] = c_j * x[row], with the group
  of every row found by numpy's searchsorted instead of the oracle's scan;
* numpy's float64 matmul, group by group, on random ragged group tables
  (empty groups, a rank whose rows all sit in one group);
* the routing semantics end to end: on a real plan, with slot weights the
  prefetched copies of their experts' home weights, the row of every
  assignment (t, k) equals hidden[t] @ W[idx[t, k]];
* rejection of malformed group tables.
"""

import numpy as np
import pytest

import oracle
from load_balancing_topk_gb300 import synth


def _bf16(a):
    return oracle.f32_to_bf16(np.asarray(a, dtype=np.float32))


def _f(h):
    return oracle.bf16_to_f32(h).astype(np.float64)


def _random_cu(rng, R, G, SK, empty_frac=0.3):
    cu = np.empty((R, G), np.int32)
    for r in range(R):
        if r == R - 1:
            sizes = np.zeros(G, np.int64)  # the whole rank in one group
            sizes[rng.integers(G)] = SK
        else:
            wts = rng.random(G) * (rng.random(G) > empty_frac)
            wts[rng.integers(G)] += 1e-3
            sizes = np.floor(wts / wts.sum() * SK).astype(np.int64)
            sizes[np.argmax(wts)] += SK - sizes.sum()
        cu[r] = np.cumsum(sizes)
    return cu


def test_scaled_identity_closed_form():
    s = synth.TINY
    idx, _ = synth.routing(s, seed=3, alpha=1.0)
    p = oracle.plan(idx, s.R, s.S, s.K, s.E, s.B)
    assert p["status"] == "ok"
    SK, G, H = s.S * s.K, s.E + s.B, 16
    rng = np.random.default_rng(7)
    x = _bf16(rng.integers(-8, 9, size=(s.R * SK, H)) / 4.0)
    eye = np.eye(H, dtype=np.float32)
    w_home = np.stack([_bf16((j + 1) * eye) for j in range(s.E)])
    w_slot = np.stack([np.stack([_bf16((100 + 10 * r + b) * eye) for b in range(s.B)])
                       for r in range(s.R)])
    y = oracle.grouped_gemm(x, p["cu_seqlens"], w_home, w_slot)
    for r in range(s.R):
        i = np.arange(SK)
        j = np.searchsorted(p["cu_seqlens"][r], i, side="right")
        c = np.where(j < s.E, j + 1, 100 + 10 * r + (j - s.E)).astype(np.float64)
        np.testing.assert_array_equal(y[r * SK:(r + 1) * SK], c[:, None] * _f(x[r * SK:(r + 1) * SK]))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_matches_numpy_matmul_per_group(seed):
    rng = np.random.default_rng(seed)
    R, E, B, SK, H, Hp = 3, 6, 3, 50, 24, 40
    G = E + B
    cu = _random_cu(rng, R, G, SK)
    x = _bf16(rng.standard_normal((R * SK, H)))
    w_home = _bf16(rng.standard_normal((E, H, Hp)))
    w_slot = _bf16(rng.standard_normal((R, B, H, Hp)))
    y = oracle.grouped_gemm(x, cu, w_home, w_slot)
    for r in range(R):
        lo = 0
        for j in range(G):
            hi = int(cu[r, j])
            W = _f(w_home[j]) if j < E else _f(w_slot[r, j - E])
            xs = _f(x[r * SK + lo:r * SK + hi])
            ref = xs @ W
            bound = 1e-13 * (np.abs(xs) @ np.abs(W))
            assert (np.abs(y[r * SK + lo:r * SK + hi] - ref) <= bound).all()
            lo = hi
    # a row subset returns the same rows
    rows = rng.choice(R * SK, size=17, replace=False)
    np.testing.assert_array_equal(oracle.grouped_gemm(x, cu, w_home, w_slot, rows=rows), y[rows])


@pytest.mark.parametrize("alpha", [1.0, 2.0])
def test_every_assignment_meets_its_routed_expert(alpha):
    s = synth.TINY
    idx, _ = synth.routing(s, seed=1, alpha=alpha)
    p = oracle.plan(idx, s.R, s.S, s.K, s.E, s.B)
    assert p["status"] == "ok" and (p["slot_expert"] >= 0).any()
    H, Hp = 32, 24
    rng = np.random.default_rng(11)
    hidden = _bf16(rng.standard_normal((s.N, H)))
    w_home = _bf16(rng.standard_normal((s.E, H, Hp)))
    w_slot = np.zeros((s.R, s.B, H, Hp), np.uint16)
    used = p["slot_expert"] >= 0
    w_slot[used] = w_home[p["slot_expert"][used]]
    buf = oracle.dispatch(hidden, p["dst_pos"], s.A)
    y = oracle.grouped_gemm(buf, p["cu_seqlens"], w_home, w_slot)
    for t in range(s.N):
        for k in range(s.K):
            ref = _f(hidden[t]) @ _f(w_home[idx[t, k]])
            bound = 1e-13 * (np.abs(_f(hidden[t])) @ np.abs(_f(w_home[idx[t, k]])))
            assert (np.abs(y[p["dst_pos"][t, k]] - ref) <= bound).all(), (t, k)


def test_rejects_bad_tables():
    R, E, B, SK, H, Hp = 2, 4, 2, 8, 8, 8
    x = np.zeros((R * SK, H), np.uint16)
    wh = np.zeros((E, H, Hp), np.uint16)
    ws = np.zeros((R, B, H, Hp), np.uint16)
    good = np.tile(np.array([2, 4, 6, 8, 8, 8], np.int32), (R, 1))
    oracle.grouped_gemm(x, good, wh, ws)
    for bad in ([2, 4, 3, 8, 8, 8], [2, 4, 6, 8, 8, 7], [-1, 4, 6, 8, 8, 8]):
        cu = good.copy()
        cu[1] = bad
        with pytest.raises(ValueError):
            oracle.grouped_gemm(x, cu, wh, ws)
    with pytest.raises(ValueError):
        oracle.grouped_gemm(x, good, wh, ws, rows=[R * SK])
