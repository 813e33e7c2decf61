"""CPU oracle for the dynamic-redundant-expert hot path (test infrastructure).

Only the tests, the package's smoke check and the benchmark's CPU-baseline
leg may import this module. It wraps ``oracle.c`` (plain C, built with gcc)
through ctypes and shares no code with the CUDA library.

Functions follow the pages' definitions (see the header of ``oracle.c`` for
the step list and citations):

* :func:`maxvio` -- max_e T_e / T_bar - 1 ("月之暗面开源MoonEP：面向MoE训练的
  专家并行通信库", section 解决的核心问题);
* :func:`plan` -- histogram, home-first planner, cu_seqlens and destination
  rows (same page, sections 核心技术 and 内存契约与权重布局);
* :func:`dispatch` / :func:`combine` -- the fused permute / weighted unpermute
  (section 核心技术, 零拷贝与静态形状);
* :func:`reduce_grad` -- slot gradients into home gradients, consumed slots
  zeroed (section 内存契约与权重布局, gradient paragraph);
* :func:`prefetch` -- redundant slots receive a copy of their expert's home
  weights (sections 核心技术 and 内存契约与权重布局);
* :func:`dispatch_backward` / :func:`combine_backward` -- the gradients of the
  fused permute and of the weighted unpermute (section 核心技术 names the
  pair; their arithmetic is this library's reading, stated in oracle.c);
* :func:`grouped_gemm` -- the grouped expert product over the static buffer,
  group j of rank r times weight row j of the [E+B, H, H'] tensor (section
  内存契约与权重布局), in double.

Parity status: every function here is pinned by the ``-m "not gpu"`` tests
(closed forms, brute force, an independent lexsort derivation, hand-worked
fixtures under ``tests/golden/`` and library routines). The planner's rule
itself is this library's reading of "online planning"; its agreement with
MoonEP's own planner is unpinned (no planner output is published).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

STATUS = {0: "ok", -1: "bad_arg", 1: "bad_routing", 2: "capacity"}


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so beside it (plain gcc, no OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            i32p = ctypes.POINTER(ctypes.c_int32)
            c_i64 = ctypes.c_int64
            lib.orc_maxvio.restype = ctypes.c_double
            lib.orc_maxvio.argtypes = [i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
            lib.orc_validate.restype = ctypes.c_int
            lib.orc_validate.argtypes = [i32p, c_i64, ctypes.c_int, ctypes.c_int]
            lib.orc_counts.restype = None
            lib.orc_counts.argtypes = [i32p, c_i64, ctypes.c_int, ctypes.c_int, i32p]
            lib.orc_plan.restype = ctypes.c_int
            lib.orc_plan.argtypes = [i32p] + [ctypes.c_int] * 5 + [i32p] * 7
            lib.orc_plan_fallback.restype = ctypes.c_int
            lib.orc_plan_fallback.argtypes = [i32p] + [ctypes.c_int] * 5 + [i32p] * 7
            lib.orc_dispatch.restype = None
            lib.orc_dispatch.argtypes = [ctypes.c_void_p, i32p, c_i64, ctypes.c_int, c_i64, ctypes.c_void_p]
            lib.orc_combine.restype = None
            lib.orc_combine.argtypes = [ctypes.c_void_p, ctypes.c_void_p, i32p, ctypes.c_void_p,
                                        c_i64, ctypes.c_int, c_i64, ctypes.c_void_p]
            lib.orc_reduce_grad.restype = ctypes.c_int
            lib.orc_reduce_grad.argtypes = [i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, c_i64,
                                            ctypes.c_void_p, ctypes.c_void_p]
            lib.orc_prefetch.restype = ctypes.c_int
            lib.orc_prefetch.argtypes = [i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, c_i64,
                                         ctypes.c_void_p, ctypes.c_void_p]
            lib.orc_dispatch_backward.restype = None
            lib.orc_dispatch_backward.argtypes = [ctypes.c_void_p, i32p, c_i64, ctypes.c_int, c_i64,
                                                  ctypes.c_void_p]
            lib.orc_combine_backward.restype = None
            lib.orc_combine_backward.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, i32p,
                                                 c_i64, ctypes.c_int, c_i64, ctypes.c_void_p,
                                                 ctypes.c_void_p]
            lib.orc_f32_to_bf16_array.restype = None
            lib.orc_f32_to_bf16_array.argtypes = [ctypes.c_void_p, c_i64, ctypes.c_void_p]
            lib.orc_grouped_gemm.restype = ctypes.c_int
            lib.orc_grouped_gemm.argtypes = [ctypes.c_void_p, i32p, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_int, c_i64, ctypes.c_int, ctypes.c_int, c_i64,
                                             c_i64, ctypes.c_void_p, c_i64, ctypes.c_void_p]
            _lib = lib
    return _lib


def _i32(a: np.ndarray):
    assert a.dtype == np.int32 and a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def maxvio(counts, R: int, S: int, K: int) -> float:
    """max_e T_e / T_bar - 1 with T_bar = R*S*K/E (float64)."""
    c = np.ascontiguousarray(counts, dtype=np.int32)
    return float(_load().orc_maxvio(_i32(c), int(c.size), R, S, K))


def validate(idx: np.ndarray, E: int) -> str:
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    N, K = idx.shape
    return STATUS[_load().orc_validate(_i32(idx), N, K, E)]


def counts(idx: np.ndarray, E: int) -> np.ndarray:
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    N, K = idx.shape
    out = np.zeros(E, dtype=np.int32)
    _load().orc_counts(_i32(idx), N, K, E, _i32(out))
    return out


def plan(idx: np.ndarray, R: int, S: int, K: int, E: int, B: int, fallback: bool = False) -> dict:
    """Home-first plan of one layer's routing.

    Returns a dict with status ("ok" / "bad_routing" / "capacity" /
    "bad_arg"), counts [E], cu_seqlens [R, E+B] (inclusive ends),
    slot_expert [R, B] (-1 = unused), slot_lo / slot_len [R, B] (range of the
    expert's token list that the slot holds), dst_pos [R*S, K] and n_pieces.

    fallback=True is the inference reading: a rank's pieces beyond B take the
    expert's own row e of that rank instead of failing with "capacity".
    """
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    N = R * S
    if idx.shape != (N, K):
        raise ValueError(f"idx shape {idx.shape} != {(N, K)}")
    G = E + B
    out = dict(
        counts=np.zeros(E, dtype=np.int32),
        cu_seqlens=np.zeros((R, G), dtype=np.int32),
        slot_expert=np.full((R, B), -1, dtype=np.int32),
        slot_lo=np.zeros((R, B), dtype=np.int32),
        slot_len=np.zeros((R, B), dtype=np.int32),
        dst_pos=np.full((N, K), -1, dtype=np.int32),
    )
    npieces = np.zeros(1, dtype=np.int32)
    fn = _load().orc_plan_fallback if fallback else _load().orc_plan
    st = fn(_i32(idx), R, S, K, E, B, _i32(out["counts"]), _i32(out["cu_seqlens"]),
                          _i32(out["slot_expert"]), _i32(out["slot_lo"]), _i32(out["slot_len"]),
                          _i32(out["dst_pos"]), _i32(npieces))
    out["status"] = STATUS[st]
    out["n_pieces"] = int(npieces[0])
    return out


def dispatch(hidden: np.ndarray, dst_pos: np.ndarray, n_rows: int) -> np.ndarray:
    """buf[n_rows, H] (bf16 bits) with buf[dst_pos[t, k]] = hidden[t]; rows never written stay 0."""
    hidden = np.ascontiguousarray(hidden, dtype=np.uint16)
    dst_pos = np.ascontiguousarray(dst_pos, dtype=np.int32)
    N, H = hidden.shape
    K = dst_pos.shape[1]
    buf = np.zeros((n_rows, H), dtype=np.uint16)
    _load().orc_dispatch(hidden.ctypes.data, _i32(dst_pos), N, K, H, buf.ctypes.data)
    return buf


def combine(y: np.ndarray, w: np.ndarray, dst_pos: np.ndarray, tokens=None) -> np.ndarray:
    """out[t] = bf16(sum_k fp32 w[t,k] * y[dst_pos[t,k]]) for all tokens, or for ``tokens``."""
    y = np.ascontiguousarray(y, dtype=np.uint16)
    w = np.ascontiguousarray(w, dtype=np.float32)
    dst_pos = np.ascontiguousarray(dst_pos, dtype=np.int32)
    N, K = dst_pos.shape
    H = y.shape[1]
    if tokens is None:
        n_tok, tok_ptr = N, None
    else:
        tokens = np.ascontiguousarray(tokens, dtype=np.int64)
        n_tok, tok_ptr = tokens.size, tokens.ctypes.data
    out = np.empty((n_tok, H), dtype=np.uint16)
    _load().orc_combine(y.ctypes.data, w.ctypes.data, _i32(dst_pos), tok_ptr, n_tok, K, H,
                        out.ctypes.data)
    return out


def reduce_grad(slot_expert: np.ndarray, home: np.ndarray, slot: np.ndarray, E: int):
    """Returns (status, home', slot') without touching the inputs.

    home is [E, HHp] fp32, slot is [R*B, HHp] fp32 (any shape that flattens to it).
    """
    se = np.ascontiguousarray(slot_expert, dtype=np.int32)
    R, B = se.shape
    h = np.array(home, dtype=np.float32, copy=True, order="C")
    s = np.array(slot, dtype=np.float32, copy=True, order="C")
    HHp = h.size // E
    assert h.size == E * HHp and s.size == R * B * HHp
    st = _load().orc_reduce_grad(_i32(se), E, R, B, HHp, h.ctypes.data, s.ctypes.data)
    return STATUS[st], h, s


def prefetch(slot_expert: np.ndarray, home: np.ndarray, slot: np.ndarray, E: int):
    """Returns (status, slot') without touching the inputs: slot'[s] = home[slot_expert[s]]
    (a byte copy) for every used slot, unused slots unchanged. home is [E, ...], slot is
    [R*B, ...] of the same dtype and trailing size."""
    se = np.ascontiguousarray(slot_expert, dtype=np.int32)
    R, B = se.shape
    h = np.ascontiguousarray(home)
    s = np.array(slot, copy=True, order="C")
    nbytes = h.nbytes // E
    assert h.nbytes == E * nbytes and s.nbytes == R * B * nbytes and h.dtype == s.dtype
    st = _load().orc_prefetch(_i32(se), E, R, B, nbytes, h.ctypes.data, s.ctypes.data)
    return STATUS[st], s


def dispatch_backward(dbuf: np.ndarray, dst_pos: np.ndarray) -> np.ndarray:
    """dhidden[t] = bf16(sum_k fp32 dbuf[dst_pos[t, k]]), adds in k order."""
    dbuf = np.ascontiguousarray(dbuf, dtype=np.uint16)
    dst_pos = np.ascontiguousarray(dst_pos, dtype=np.int32)
    N, K = dst_pos.shape
    H = dbuf.shape[1]
    out = np.empty((N, H), dtype=np.uint16)
    _load().orc_dispatch_backward(dbuf.ctypes.data, _i32(dst_pos), N, K, H, out.ctypes.data)
    return out


def combine_backward(dout: np.ndarray, y: np.ndarray, w: np.ndarray, dst_pos: np.ndarray):
    """(dy bf16 [A, H], dw float64 [N, K]) of out[t] = sum_k w[t,k] y[dst_pos[t,k]].

    Rows of dy that no assignment maps to are left 0."""
    dout = np.ascontiguousarray(dout, dtype=np.uint16)
    y = np.ascontiguousarray(y, dtype=np.uint16)
    w = np.ascontiguousarray(w, dtype=np.float32)
    dst_pos = np.ascontiguousarray(dst_pos, dtype=np.int32)
    N, K = dst_pos.shape
    H = dout.shape[1]
    dy = np.zeros_like(y)
    dw = np.empty((N, K), dtype=np.float64)
    _load().orc_combine_backward(dout.ctypes.data, y.ctypes.data, w.ctypes.data, _i32(dst_pos), N, K,
                                 H, dy.ctypes.data, dw.ctypes.data)
    return dy, dw


def grouped_gemm(x: np.ndarray, cu: np.ndarray, w_home: np.ndarray, w_slot: np.ndarray,
                 rows=None) -> np.ndarray:
    """y[row] = x[row] @ W_j in double for the buffer rows (all, or ``rows``).

    x is [R*SK, H] bf16 bits, cu [R, E+B] inclusive group ends, w_home
    [E, H, H'] and w_slot [R, B, H, H'] bf16 bits. Group j of rank r uses
    w_home[j] (j < E) or w_slot[r, j - E]. Raises ValueError on a bad table."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    cu = np.ascontiguousarray(cu, dtype=np.int32)
    w_home = np.ascontiguousarray(w_home, dtype=np.uint16)
    w_slot = np.ascontiguousarray(w_slot, dtype=np.uint16)
    R, G = cu.shape
    E, H, Hp = w_home.shape
    B = G - E
    assert w_slot.shape == (R, B, H, Hp) and x.shape[1] == H and x.shape[0] % R == 0
    SK = x.shape[0] // R
    if rows is None:
        n, rp = x.shape[0], None
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        n, rp = rows.size, rows.ctypes.data
    y = np.empty((n, Hp), dtype=np.float64)
    st = _load().orc_grouped_gemm(x.ctypes.data, _i32(cu), w_home.ctypes.data, w_slot.ctypes.data,
                                  R, SK, E, B, H, Hp, rp, n, y.ctypes.data)
    if st != 0:
        raise ValueError(f"grouped_gemm: {STATUS[st]}")
    return y


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().orc_f32_to_bf16_array(x.ctypes.data, x.size, out.ctypes.data)
    return out


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    """Widen bf16 bits to float32 (exact: the bits become the top half)."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)
