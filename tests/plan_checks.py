"""Checks on a plan that do not reuse the oracle's arithmetic.

They test what the pages fix for any correct plan
("月之暗面开源MoonEP：面向MoE训练的专家并行通信库", sections 核心技术 and
内存契约与权重布局; "Moonshot AI Open-Sources MoonEP for Expert Parallelism",
paragraphs 2-3):

* every rank receives exactly S*K rows (cu_seqlens[r][-1] == S*K);
* every assignment is placed exactly once (dst_pos is a permutation);
* an expert's tokens are split between its home row and redundant slots,
  whose lengths add up to T_e (conservation);
* rows [0, E) of rank r other than its E/R home rows are empty;
* at most B slots per rank, filled from slot 0 upwards;
* inside one group, tokens appear in ascending token order.

``derive_dst_pos`` is a second route to the destination rows: it computes
each assignment's (rank, row) from the plan's group table and the expert's
token list, then ranks all assignments by (rank, row, token) with a stable
``numpy.lexsort``, sharing nothing with the oracle's position step.
"""

from __future__ import annotations

import numpy as np


def group_sizes(cu: np.ndarray) -> np.ndarray:
    cu = np.asarray(cu, dtype=np.int64)
    c = cu.copy()
    c[:, 1:] -= cu[:, :-1]
    return c


def check_invariants(p: dict, idx: np.ndarray, R: int, S: int, K: int, E: int, B: int) -> None:
    assert p["status"] == "ok", p["status"]
    N = R * S
    A = N * K
    per = E // R
    SK = S * K
    cu = np.asarray(p["cu_seqlens"], dtype=np.int64).reshape(R, E + B)
    se = np.asarray(p["slot_expert"]).reshape(R, B)
    c = group_sizes(cu)
    counts = np.bincount(np.asarray(idx).reshape(-1), minlength=E)
    assert (np.asarray(p["counts"]) == counts).all()
    # exactly S*K per rank
    assert (cu[:, -1] == SK).all() if E + B > 0 else True
    assert (c >= 0).all()
    # non-home rows are empty
    for r in range(R):
        home = np.zeros(E, dtype=bool)
        home[r * per:(r + 1) * per] = True
        assert (c[r, :E][~home] == 0).all()
    # slots: filled from 0, valid experts, lengths > 0, unused -> width 0
    for r in range(R):
        used = se[r] >= 0
        nu = int(used.sum())
        assert used[:nu].all() and not used[nu:].any()
        assert (se[r][used] < E).all()
        assert (c[r, E:][used] > 0).all()
        assert (c[r, E:][~used] == 0).all()
        # a slot never holds one of the rank's own experts
        assert ((se[r][used] // per) != r).all()
    # conservation per expert
    tot = np.zeros(E, dtype=np.int64)
    for e in range(E):
        tot[e] += c[e // per, e]
    for r in range(R):
        for b in range(B):
            if se[r, b] >= 0:
                tot[se[r, b]] += c[r, E + b]
    assert (tot == counts).all()
    # dst_pos is a permutation of [0, A)
    d = np.asarray(p["dst_pos"], dtype=np.int64).reshape(-1)
    assert d.size == A
    if A:
        assert d.min() == 0 and d.max() == A - 1
        assert np.bincount(d, minlength=A).max() == 1


def derive_dst_pos(idx: np.ndarray, cu: np.ndarray, slot_expert: np.ndarray,
                   slot_lo: np.ndarray, R: int, S: int, K: int, E: int, B: int) -> np.ndarray:
    """Destination rows from the group table by a stable lexsort."""
    idx = np.asarray(idx, dtype=np.int64)
    N = R * S
    A = N * K
    per = E // R
    SK = S * K
    cu = np.asarray(cu, dtype=np.int64).reshape(R, E + B)
    c = group_sizes(cu)
    se = np.asarray(slot_expert).reshape(R, B)
    lo = np.asarray(slot_lo, dtype=np.int64).reshape(R, B)
    flat_e = idx.reshape(-1)
    tok = np.repeat(np.arange(N, dtype=np.int64), K)
    # index of each assignment in its expert's ascending token list
    order = np.argsort(flat_e, kind="stable")
    li = np.empty(A, dtype=np.int64)
    starts = np.concatenate([[0], np.cumsum(np.bincount(flat_e, minlength=E))])
    li[order] = np.arange(A) - starts[flat_e[order]]
    keep = np.array([c[e // per, e] for e in range(E)], dtype=np.int64)
    dst_rank = np.empty(A, dtype=np.int64)
    row = np.empty(A, dtype=np.int64)
    home = li < keep[flat_e]
    dst_rank[home] = flat_e[home] // per
    row[home] = flat_e[home]
    spill = np.nonzero(~home)[0]
    for a in spill:
        e, i = flat_e[a], li[a]
        hit = [(r, b) for r in range(R) for b in range(B)
               if se[r, b] == e and lo[r, b] <= i < lo[r, b] + c[r, E + b]]
        assert len(hit) == 1, (a, e, i, hit)
        dst_rank[a], row[a] = hit[0][0], E + hit[0][1]
    keyorder = np.lexsort((tok, row, dst_rank))
    out = np.empty(A, dtype=np.int64)
    out[keyorder] = np.arange(A)
    # the lexsort rank must fall inside the group's span of the static buffer
    start = np.array([r * SK + (cu[r, j] - c[r, j]) for r, j in zip(dst_rank, row)])
    assert (out >= start).all()
    return out.reshape(N, K)


def check_invariants_fallback(p: dict, idx: np.ndarray, R: int, S: int, K: int, E: int, B: int) -> None:
    """The invariants under the inference reading: as check_invariants, except
    that a rank's non-home rows [0, E) may hold a piece once all of its B slots
    are in use."""
    assert p["status"] == "ok", p["status"]
    N, A, per, SK = R * S, R * S * K, E // R, S * K
    cu = np.asarray(p["cu_seqlens"], dtype=np.int64).reshape(R, E + B)
    se = np.asarray(p["slot_expert"]).reshape(R, B)
    c = group_sizes(cu)
    counts = np.bincount(np.asarray(idx).reshape(-1), minlength=E)
    assert (np.asarray(p["counts"]) == counts).all()
    assert (cu[:, -1] == SK).all() and (c >= 0).all()
    tot = np.zeros(E, dtype=np.int64)
    for r in range(R):
        used = se[r] >= 0
        nu = int(used.sum())
        assert used[:nu].all() and not used[nu:].any()
        assert ((se[r][used] // per) != r).all()
        nonhome = np.ones(E, dtype=bool)
        nonhome[r * per:(r + 1) * per] = False
        if (c[r, :E][nonhome] > 0).any():
            assert nu == B  # remote rows only once the slots are full
        tot += c[r, :E]
        for b in range(B):
            if se[r, b] >= 0:
                tot[se[r, b]] += c[r, E + b]
                # a rank holds at most one piece of an expert
                assert c[r, se[r, b]] == 0
    assert (tot == counts).all()
    d = np.asarray(p["dst_pos"], dtype=np.int64).reshape(-1)
    if A:
        assert np.bincount(d, minlength=A).max() == 1 and d.min() == 0 and d.max() == A - 1


def derive_dst_pos_from_groups(idx, cu, slot_expert, R, S, K, E, B) -> np.ndarray:
    """Destination rows from the group table alone. Expert e's tokens fill its
    home row, then its pieces on the other ranks in ascending rank order: a
    slot row E+b where slot_expert[r,b] == e, else the rank's row e. Each
    assignment's (rank, row) comes from its index in e's list; a stable
    lexsort on (rank, row, token) gives the rows."""
    idx = np.asarray(idx, dtype=np.int64)
    N, A, per = R * S, R * S * K, E // R
    cu = np.asarray(cu, dtype=np.int64).reshape(R, E + B)
    c = group_sizes(cu)
    se = np.asarray(slot_expert).reshape(R, B)
    flat_e = idx.reshape(-1)
    tok = np.repeat(np.arange(N, dtype=np.int64), K)
    order = np.argsort(flat_e, kind="stable")
    li = np.empty(A, dtype=np.int64)
    starts = np.concatenate([[0], np.cumsum(np.bincount(flat_e, minlength=E))])
    li[order] = np.arange(A) - starts[flat_e[order]]
    segs = {}  # e -> list of (lo, hi, rank, row)
    for e in range(E):
        h = e // per
        lo = c[h, e]
        segs[e] = [(0, lo, h, e)]
        for r in range(R):
            if r == h:
                continue
            row = None
            for b in range(B):
                if se[r, b] == e:
                    row = E + b
            width = c[r, row] if row is not None else c[r, e]
            if row is None:
                row = e
            if width:
                segs[e].append((lo, lo + width, r, row))
                lo += width
    rank = np.empty(A, dtype=np.int64)
    rowj = np.empty(A, dtype=np.int64)
    for a in range(A):
        e, i = flat_e[a], li[a]
        hit = [(r, j) for lo, hi, r, j in segs[e] if lo <= i < hi]
        assert len(hit) == 1
        rank[a], rowj[a] = hit[0]
    keyorder = np.lexsort((tok, rowj, rank))
    out = np.empty(A, dtype=np.int64)
    out[keyorder] = np.arange(A)
    return out.reshape(N, K)
