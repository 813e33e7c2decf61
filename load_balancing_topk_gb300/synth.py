"""Seeded synthetic inputs for the dynamic-redundant-expert hot path.

This module only draws inputs: router choices, routing weights, token rows and
gradient tensors. It holds none of the method's arithmetic (no counting, no
planning, no permutation, no rounding of results) and imports neither the
CUDA library nor the CPU oracle, so both sides can be fed from it.

The pages describe the workload only as "top-K routing with skew" measured by
maxvio (Moonshot AI Open-Sources MoonEP for Expert Parallelism, second
paragraph; 月之暗面开源MoonEP：面向MoE训练的专家并行通信库, section
解决的核心问题). No routing trace is published, so a synthetic router stands
in for a trained one:

* logits[t, e] = N(0, 1) - alpha * ln(pop_rank[e] + 1), a Zipf(alpha)
  log-popularity bias, where pop_rank is a seeded permutation of the experts
  (or the identity, the adversarial placement that puts the hottest experts
  on rank 0);
* topk_idx[t] = the K largest logits in descending order, ties going to the
  lower expert id;
* topk_w[t] = softmax of the chosen logits, computed in float32;
* "round_robin" routing, idx[t, k] = (t*K + k) mod E, gives every expert the
  same count (the maxvio = 0 point);
* "hot" routing forces one expert (the most popular) into the top-K of a
  Bernoulli(p) subset of tokens and out of the rest; its weight keeps the
  expert's natural logit.

Every array comes from its own counter-free numpy PCG64 stream keyed by
(seed, tag), so drawing one tensor never shifts another.
"""

from __future__ import annotations

import dataclasses

import numpy as np

# Stream tags: one independent PCG64 stream per tensor kind.
_TAG_PLACEMENT = 1
_TAG_LOGITS = 2
_TAG_HOT = 3
_TAG_RR_WEIGHTS = 4
_TAG_HIDDEN = 5
_TAG_Y = 6
_TAG_HOME_GRAD = 7
_TAG_SLOT_GRAD = 8
_TAG_SLOT_MAP = 9


def _rng(seed: int, tag: int, sub: int = 0) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(seed), tag, int(sub)]))


@dataclasses.dataclass(frozen=True)
class Shape:
    """Sizes of one MoE layer's routing problem.

    R virtual ranks, E routed experts (E/R per rank), K experts per token,
    S tokens per rank, H hidden size, B redundant slots per rank.
    """

    R: int
    E: int
    K: int
    S: int
    H: int
    B: int

    @property
    def N(self) -> int:
        return self.R * self.S

    @property
    def A(self) -> int:
        return self.R * self.S * self.K


# The workloads the library is measured and checked on.
TINY = Shape(R=2, E=8, K=2, S=64, H=128, B=4)
MEDIUM = Shape(R=8, E=64, K=6, S=4096, H=2048, B=8)
LARGE = Shape(R=8, E=256, K=8, S=8192, H=7168, B=32)
STRESS = Shape(R=16, E=384, K=8, S=4096, H=7168, B=24)
# reduce_grad: E=64 experts on R=8 ranks with B=8 slots, H=2048, H'=1408.
GRAD_E, GRAD_R, GRAD_B, GRAD_H, GRAD_HP = 64, 8, 8, 2048, 1408

SHAPES = {"tiny": TINY, "medium": MEDIUM, "large": LARGE, "stress": STRESS}


def _order_key(logits: np.ndarray) -> np.ndarray:
    """A unique uint64 key per (row, expert) whose order is (logit desc, id asc)."""
    E = logits.shape[1]
    u = logits.astype(np.float32, copy=False).view(np.uint32)
    neg = (u & np.uint32(0x80000000)) != 0
    mono = np.where(neg, ~u, u | np.uint32(0x80000000)).astype(np.uint64)
    ids = np.arange(E, dtype=np.uint64)
    return (mono << np.uint64(32)) | (np.uint64(0xFFFFFFFF) - ids)[None, :]


def _topk_desc(keys: np.ndarray, K: int) -> np.ndarray:
    """Column indices of the K largest keys per row, largest first."""
    E = keys.shape[1]
    if K == E:
        part = np.broadcast_to(np.arange(E), keys.shape).copy()
    else:
        part = np.argpartition(keys, E - K, axis=1)[:, E - K:]
    sel = np.take_along_axis(keys, part, axis=1)
    order = np.argsort(sel, axis=1)[:, ::-1]
    return np.take_along_axis(part, order, axis=1)


def _softmax_f32(x: np.ndarray) -> np.ndarray:
    x = x.astype(np.float32)
    m = np.max(x, axis=1, keepdims=True)
    ex = np.exp(x - m, dtype=np.float32)
    return (ex / np.sum(ex, axis=1, keepdims=True, dtype=np.float32)).astype(np.float32)


def routing(shape: Shape, seed: int = 0, alpha: float = 1.0, kind: str = "zipf",
            placement: str = "permuted", hot_frac: float = 0.3,
            chunk: int = 8192) -> tuple[np.ndarray, np.ndarray]:
    """Return (topk_idx int32 [N, K], topk_w float32 [N, K]) for one layer.

    kind: "zipf" (logit bias), "hot" (zipf plus one forced hot expert) or
    "round_robin" (idx[t, k] = (t*K + k) mod E).
    """
    N, E, K = shape.N, shape.E, shape.K
    if K > E:
        raise ValueError("K > E")
    if kind == "round_robin":
        t = np.arange(N, dtype=np.int64)[:, None]
        k = np.arange(K, dtype=np.int64)[None, :]
        idx = ((t * K + k) % E).astype(np.int32)
        g = _rng(seed, _TAG_RR_WEIGHTS)
        z = g.standard_normal((N, K), dtype=np.float32)
        z = -np.sort(-z, axis=1)
        return idx, _softmax_f32(z)
    if kind not in ("zipf", "hot"):
        raise ValueError(kind)
    if placement == "permuted":
        pop_rank = _rng(seed, _TAG_PLACEMENT).permutation(E)
    elif placement == "identity":
        pop_rank = np.arange(E)
    else:
        raise ValueError(placement)
    bias = (-alpha * np.log(pop_rank.astype(np.float64) + 1.0)).astype(np.float32)
    hot = int(np.argmin(pop_rank))
    g = _rng(seed, _TAG_LOGITS)
    forced = None
    if kind == "hot":
        forced = _rng(seed, _TAG_HOT).random(N) < hot_frac
    idx = np.empty((N, K), dtype=np.int32)
    w = np.empty((N, K), dtype=np.float32)
    for lo in range(0, N, chunk):
        hi = min(N, lo + chunk)
        lg = g.standard_normal((hi - lo, E), dtype=np.float32) + bias[None, :]
        sel_logits = lg
        if forced is not None:
            sel_logits = lg.copy()
            f = forced[lo:hi]
            sel_logits[f, hot] = np.float32(np.inf)
            sel_logits[~f, hot] = np.float32(-np.inf)
        cols = _topk_desc(_order_key(sel_logits), K)
        idx[lo:hi] = cols
        w[lo:hi] = _softmax_f32(np.take_along_axis(lg, cols, axis=1))
    return idx, w


def _parallel(fn, n_items: int) -> None:
    """Run fn(i) for i in range(n_items) on a thread pool (numpy and torch
    release the GIL while filling large arrays)."""
    import os
    from concurrent.futures import ThreadPoolExecutor

    workers = max(1, min(n_items, os.cpu_count() or 1))
    if workers == 1:
        for i in range(n_items):
            fn(i)
        return
    with ThreadPoolExecutor(workers) as ex:
        list(ex.map(fn, range(n_items)))


def bf16_normal(n_rows: int, n_cols: int, seed: int, tag: int = _TAG_HIDDEN,
                chunk_rows: int = 4096):
    """Rows of N(0, 1) values stored as bfloat16 bit patterns (uint16 [n_rows, n_cols]).

    The float32 draws are narrowed by torch's CPU bf16 conversion. Each block
    of ``chunk_rows`` rows has its own stream, so the result does not depend
    on the number of threads.
    """
    import torch

    out = np.empty((n_rows, n_cols), dtype=np.uint16)
    starts = list(range(0, n_rows, chunk_rows))

    def one(i):
        lo = starts[i]
        hi = min(n_rows, lo + chunk_rows)
        x = _rng(seed, tag, lo).standard_normal((hi - lo, n_cols), dtype=np.float32)
        out[lo:hi] = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)

    _parallel(one, len(starts))
    return out


def hidden(shape: Shape, seed: int = 0) -> np.ndarray:
    """Token rows hidden[N, H], bf16 bits, ~N(0, 1)."""
    return bf16_normal(shape.N, shape.H, seed, _TAG_HIDDEN)


def expert_out(shape: Shape, seed: int = 0) -> np.ndarray:
    """Expert outputs y[R*S*K, H], bf16 bits, ~N(0, 1)."""
    return bf16_normal(shape.A, shape.H, seed, _TAG_Y)


def grads(E: int, R: int, B: int, HHp: int, seed: int = 0, sigma: float = 1e-3,
          chunk: int = 1 << 22) -> tuple[np.ndarray, np.ndarray]:
    """(home_grad float32 [E, HHp], slot_grad float32 [R*B, HHp]), ~N(0, sigma^2)."""

    def draw(rows, tag):
        a = np.empty((rows, HHp), dtype=np.float32)
        flat = a.reshape(-1)
        starts = list(range(0, flat.size, chunk))

        def one(i):
            lo = starts[i]
            hi = min(flat.size, lo + chunk)
            flat[lo:hi] = _rng(seed, tag, i).standard_normal(hi - lo, dtype=np.float32) * np.float32(sigma)

        _parallel(one, len(starts))
        return a

    return draw(E, _TAG_HOME_GRAD), draw(R * B, _TAG_SLOT_GRAD)


def full_slot_map(E: int, R: int, B: int, seed: int = 0) -> np.ndarray:
    """A seeded slot -> expert map that fills every slot (int32 [R, B]).

    Used for the reduce_grad throughput variant in which all R*B slots are
    consumed. Expert e's home rank is e // (E // R); each slot gets an expert
    homed elsewhere, and when R*B == E the map is a bijection.
    """
    per = E // R
    g = _rng(seed, _TAG_SLOT_MAP)
    for _ in range(1000):
        perm = g.permutation(np.resize(np.arange(E), R * B))
        m = perm.reshape(R, B)
        if all((m[r] // per != r).all() for r in range(R)):
            return m.astype(np.int32)
    raise RuntimeError("could not draw a slot map with no home slots")


def integer_valued(shape, seed: int, lo: int = -8, hi: int = 8, tag: int = 99) -> np.ndarray:
    """Small integers stored as float32: sums of these are exact in any order."""
    g = _rng(seed, tag)
    return g.integers(lo, hi + 1, size=shape).astype(np.float32)


def alpha_for(name: str, target_maxvio: float, table: dict | None = None) -> float:
    """Look up a calibrated Zipf alpha for a workload and target maxvio.

    The table (``zipf_alpha.json`` beside this module) holds, per workload
    and target, the alpha whose seed-0 routing realises that maxvio within
    0.5%; it is fitted by bisection on the realised maxvio."""
    if table is None:
        import json
        import os

        path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "zipf_alpha.json")
        with open(path) as f:
            table = json.load(f)
    key = f"{target_maxvio:g}"
    try:
        return float(table[name][key])
    except KeyError as exc:
        raise KeyError(f"no calibrated alpha for {name} at maxvio {key}") from exc



__all__ = [
    "Shape", "TINY", "MEDIUM", "LARGE", "STRESS", "SHAPES",
    "GRAD_E", "GRAD_R", "GRAD_B", "GRAD_H", "GRAD_HP",
    "routing", "hidden", "expert_out", "grads", "full_slot_map", "bf16_normal",
    "integer_valued", "alpha_for",
]
