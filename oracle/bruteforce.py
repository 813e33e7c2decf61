"""Exhaustive minimum-replica search on tiny instances (test infrastructure).

The pages call the planner "online integer linear programming" with a
"near-optimal" GPU kernel ("Valhalla 静态工程审阅 #004｜MoonshotAI MoonEP
源码证据驱动评测", 摘要; "月之暗面开源MoonEP：面向MoE训练的专家并行通信库",
section 核心技术) but give no formulation. This module states the plainest
integer program the rest of the pages support and solves it by enumeration,
so the home-first planner can be reported against the true optimum:

    choose integers x[e, r] >= 0 with
        sum_r x[e, r] = T_e                 (every assignment placed)
        sum_e x[e, r] = S*K                 (the S*K invariant, 核心技术)
        #{e : x[e, r] > 0, home(e) != r} <= B   (B prefetch slots per rank,
                                                  内存契约与权重布局)
    minimising the number of redundant pairs #{(e, r) : x[e, r] > 0, home(e) != r}.

For a fixed set P of allowed redundant pairs, feasibility is a transportation
problem, decided exactly by a max-flow (scipy's integer max-flow):
source -> expert e (capacity T_e) -> its home rank and the ranks r with
(e, r) in P -> sink (capacity S*K per rank). Sets are enumerated by size, so
the first feasible size is the minimum.
"""

from __future__ import annotations

import itertools

import numpy as np
from scipy.sparse import csr_matrix
from scipy.sparse.csgraph import maximum_flow


def _feasible(T, R, SK, B, pairs) -> bool:
    E = len(T)
    per = E // R
    per_rank = np.zeros(R, dtype=np.int64)
    for _, r in pairs:
        per_rank[r] += 1
    if (per_rank > B).any():
        return False
    # nodes: 0 = source, 1..E experts, E+1..E+R ranks, E+R+1 sink
    src, snk = 0, E + R + 1
    big = int(sum(T)) + 1
    rows, cols, caps = [], [], []
    for e in range(E):
        rows.append(src); cols.append(1 + e); caps.append(int(T[e]))
        rows.append(1 + e); cols.append(1 + E + e // per); caps.append(big)
    for e, r in pairs:
        rows.append(1 + e); cols.append(1 + E + r); caps.append(big)
    for r in range(R):
        rows.append(1 + E + r); cols.append(snk); caps.append(int(SK))
    g = csr_matrix((np.array(caps, dtype=np.int32), (rows, cols)), shape=(snk + 1, snk + 1))
    flow = maximum_flow(g, src, snk).flow_value
    return flow == int(sum(T))


def min_replicas(T, R: int, S: int, K: int, B: int, max_size: int | None = None):
    """Smallest number of redundant (expert, rank) pairs that balances T.

    Returns None if no set of at most ``max_size`` pairs (default: R*B) works.
    """
    T = np.asarray(T, dtype=np.int64)
    E = T.size
    per = E // R
    SK = S * K
    cand = [(e, r) for e in range(E) if T[e] > 0 for r in range(R) if r != e // per]
    limit = R * B if max_size is None else max_size
    for size in range(0, min(limit, len(cand)) + 1):
        for pairs in itertools.combinations(cand, size):
            if _feasible(T, R, SK, B, pairs):
                return size
    return None


def min_replicas_two_ranks(T, S: int, K: int) -> int:
    """Closed form for R = 2: the fewest experts of the over-loaded rank whose
    counts cover its overflow (each replica can take all of its expert)."""
    T = np.asarray(T, dtype=np.int64)
    per = T.size // 2
    SK = S * K
    loads = [int(T[:per].sum()), int(T[per:].sum())]
    over = max(loads[0] - SK, loads[1] - SK, 0)
    if over == 0:
        return 0
    hot = 0 if loads[0] > SK else 1
    vals = np.sort(T[hot * per:(hot + 1) * per])[::-1]
    return int(np.searchsorted(np.cumsum(vals), over) + 1)
