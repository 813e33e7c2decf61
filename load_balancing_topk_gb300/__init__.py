"""GB300 (sm_103a) dynamic-redundant-expert hot path: thin Python binding.

The computation lives in ``libmep.so`` (hand-written CUDA behind the C ABI of
``include/mep.h``). This module only marshals torch CUDA tensors into that
ABI: it checks dtypes, shapes and devices, allocates outputs when the caller
does not pass them, and passes raw device pointers plus torch's current
stream. It never computes a step itself and has no CPU fallback: if the
library is missing, every call raises.

Entry points (same names as the C ABI):

* :func:`mep_plan` -- routing histogram, home-first planner, cu_seqlens and
  destination rows for one layer ("月之暗面开源MoonEP：面向MoE训练的专家并行
  通信库", sections 核心技术 and 内存契约与权重布局);
* :func:`mep_dispatch` -- fused permute into the static [R, S*K, H] buffer;
* :func:`mep_combine` -- fused weighted unpermute back to [R*S, H];
* :func:`mep_reduce_grad` -- slot gradients into home gradients, consumed
  slots zeroed;
* :func:`mep_prefetch` -- redundant experts' weights copied into their slots;
* :func:`mep_dispatch_backward` / :func:`mep_combine_backward` -- gradients of
  the two permutes.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import NamedTuple, Optional

__all__ = [
    "MepError", "Plan", "library_path", "load_library", "status_string", "version",
    "plan_workspace_bytes", "plan_kernel_count", "mep_plan", "mep_plan_remote_fallback", "mep_dispatch", "mep_combine", "mep_reduce_grad",
    "mep_prefetch", "mep_dispatch_backward", "mep_combine_backward", "STATUS",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libmep.so"
_lock = threading.Lock()
_lib = None

# Codes from include/mep.h.
STATUS = {
    0: "MEP_OK",
    1: "MEP_ERR_INVALID_ARG",
    2: "MEP_ERR_CUDA",
    3: "MEP_ERR_BAD_ROUTING",
    4: "MEP_ERR_CAPACITY",
    5: "MEP_ERR_BAD_POSITION",
    6: "MEP_ERR_BAD_SLOT_MAP",
    7: "MEP_ERR_TIMEOUT",
    8: "MEP_ERR_BAD_SEQLENS",
}
STATUS_CODE = {v: k for k, v in STATUS.items()}

# (name, restype, argtypes) of every function include/mep.h declares.
_VP = ctypes.c_void_p
_I = ctypes.c_int
SIGNATURES = [
    ("mep_version", _I, []),
    ("mep_status_string", ctypes.c_char_p, [_I]),
    ("mep_plan_workspace_bytes", _I, [_I, _I, _I, _I, _I, ctypes.POINTER(ctypes.c_size_t)]),
    ("mep_plan_kernel_count", _I, [_I, _I, _I, _I, _I, ctypes.POINTER(_I)]),
    ("mep_plan", _I, [_VP, _I, _I, _I, _I, _I, _VP, ctypes.c_size_t, _VP, _VP, _VP, _VP, _VP, _VP]),
    ("mep_plan_remote_fallback", _I, [_VP, _I, _I, _I, _I, _I, _VP, ctypes.c_size_t, _VP, _VP, _VP, _VP, _VP, _VP]),
    ("mep_plan_static_scratch", _I, [_VP, _I, _I, _I, _I, _I, _VP, _VP, _VP, _VP, _VP, _VP]),
    ("mep_dispatch", _I, [_VP, _VP, _VP, _I, _I, _I, _I, _VP, _VP]),
    ("mep_combine", _I, [_VP, _VP, _VP, _VP, _I, _I, _I, _I, _VP, _VP]),
    ("mep_reduce_grad", _I, [_VP, _I, _I, _I, ctypes.c_int64, _VP, _VP, _VP, _VP]),
    ("mep_prefetch", _I, [_VP, _I, _I, _I, ctypes.c_int64, _VP, _VP, _VP, _VP]),
    ("mep_dispatch_backward", _I, [_VP, _VP, _VP, _I, _I, _I, _I, _VP, _VP]),
    ("mep_combine_backward", _I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _VP, _VP, _VP]),
    ("mep_grouped_gemm_workspace_bytes", _I, [_I, _I, _I, _I, _I, ctypes.POINTER(ctypes.c_size_t)]),
    ("mep_grouped_gemm", _I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _I, _VP, ctypes.c_size_t,
                              _VP, _VP]),
    ("mep_wait_selftest", _I, [_VP, ctypes.c_int64, _VP, _VP]),
]


class MepError(RuntimeError):
    """A host-side error code returned by the library."""

    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} returned {STATUS.get(code, code)}: {status_string(code)}")


def library_path() -> str:
    return os.path.join(_PKG, _LIB_NAME)


def load_library():
    """Load libmep.so (built in-tree by ``_build.build()``); raises if absent."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it with load_balancing_topk_gb300._build.build() "
                    "(there is no fallback implementation)")
            lib = ctypes.CDLL(path)
            for name, res, args in SIGNATURES:
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def version() -> tuple[int, int]:
    v = load_library().mep_version()
    return v >> 16, v & 0xFFFF


def status_string(code: int) -> str:
    return load_library().mep_status_string(int(code)).decode()


def _check(fn: str, rc: int) -> None:
    if rc != 0:
        raise MepError(fn, rc)


def plan_workspace_bytes(R: int, S: int, K: int, E: int, B: int) -> int:
    out = ctypes.c_size_t(0)
    _check("mep_plan_workspace_bytes",
           load_library().mep_plan_workspace_bytes(R, S, K, E, B, ctypes.byref(out)))
    return int(out.value)


def plan_kernel_count(R: int, S: int, K: int, E: int, B: int) -> int:
    """Kernels one mep_plan call enqueues for these sizes (launch accounting)."""
    n = _I(0)
    _check("mep_plan_kernel_count", load_library().mep_plan_kernel_count(R, S, K, E, B, ctypes.byref(n)))
    return int(n.value)


def grouped_gemm_workspace_bytes(R: int, S: int, K: int, E: int, B: int) -> int:
    out = ctypes.c_size_t(0)
    _check("mep_grouped_gemm_workspace_bytes",
           load_library().mep_grouped_gemm_workspace_bytes(R, S, K, E, B, ctypes.byref(out)))
    return int(out.value)


# ---------------------------------------------------------------------------
def _torch():
    import torch

    return torch


def _need(t, name, dtype, shape=None, device=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(device) -> int:
    torch = _torch()
    return torch.cuda.current_stream(device).cuda_stream


class Plan(NamedTuple):
    """Outputs of :func:`mep_plan` (all on the device)."""

    expert_counts: "torch.Tensor"   # int32 [E]
    cu_seqlens: "torch.Tensor"      # int32 [R, E+B]
    slot_expert: "torch.Tensor"     # int32 [R, B]
    dst_pos: "torch.Tensor"         # int32 [R*S, K]
    status: "torch.Tensor"          # int32 [1]
    workspace: "torch.Tensor"       # uint8 scratch, reusable for the same sizes


def mep_plan(topk_idx, R: int, S: int, K: int, E: int, B: int, out: Optional[Plan] = None) -> Plan:
    """Plan one layer's routing. ``topk_idx`` is int32 [R*S, K] on the device.

    Nothing is synchronised: read ``status`` (0 = ok) when convenient.
    """
    return _plan("mep_plan", topk_idx, R, S, K, E, B, out)


def mep_plan_remote_fallback(topk_idx, R: int, S: int, K: int, E: int, B: int,
                             out: Optional[Plan] = None) -> Plan:
    """mep_plan under the inference reading: pieces beyond a rank's B slots
    take the expert's own row (served by its home weights) instead of failing."""
    return _plan("mep_plan_remote_fallback", topk_idx, R, S, K, E, B, out)


def _plan(fn: str, topk_idx, R, S, K, E, B, out):
    torch = _torch()
    _need(topk_idx, "topk_idx", torch.int32, (R * S, K))
    dev = topk_idx.device
    ws_bytes = plan_workspace_bytes(R, S, K, E, B)
    if out is None:
        out = Plan(
            expert_counts=torch.empty(E, dtype=torch.int32, device=dev),
            cu_seqlens=torch.empty((R, E + B), dtype=torch.int32, device=dev),
            slot_expert=torch.empty((R, B), dtype=torch.int32, device=dev),
            dst_pos=torch.empty((R * S, K), dtype=torch.int32, device=dev),
            status=torch.empty(1, dtype=torch.int32, device=dev),
            workspace=torch.empty(ws_bytes, dtype=torch.uint8, device=dev),
        )
    else:
        _need(out.expert_counts, "expert_counts", torch.int32, (E,), dev)
        _need(out.cu_seqlens, "cu_seqlens", torch.int32, (R, E + B), dev)
        _need(out.slot_expert, "slot_expert", torch.int32, (R, B), dev)
        _need(out.dst_pos, "dst_pos", torch.int32, (R * S, K), dev)
        _need(out.status, "status", torch.int32, (1,), dev)
        _need(out.workspace, "workspace", torch.uint8, None, dev)
        if out.workspace.numel() < ws_bytes:
            raise ValueError(f"workspace has {out.workspace.numel()} bytes, needs {ws_bytes}")
    with torch.cuda.device(dev):
        rc = getattr(load_library(), fn)(
            _ptr(topk_idx), R, S, K, E, B, _ptr(out.workspace), out.workspace.numel(),
            _ptr(out.expert_counts), _ptr(out.cu_seqlens), _ptr(out.slot_expert),
            _ptr(out.dst_pos), _ptr(out.status), _stream(dev))
    _check(fn, rc)
    return out


def mep_dispatch(hidden, dst_pos, status, R: int, S: int, K: int, buf=None):
    """buf[dst_pos[t, k]] = hidden[t]; returns buf (bf16 [R*S*K, H])."""
    torch = _torch()
    _need(hidden, "hidden", torch.bfloat16)
    N, H = hidden.shape
    if N != R * S:
        raise ValueError("hidden must be [R*S, H]")
    dev = hidden.device
    _need(dst_pos, "dst_pos", torch.int32, (N, K), dev)
    if status is not None:
        _need(status, "status", torch.int32, (1,), dev)
    if buf is None:
        buf = torch.empty((N * K, H), dtype=torch.bfloat16, device=dev)
    else:
        _need(buf, "buf", torch.bfloat16, None, dev)
        if buf.numel() != N * K * H:
            raise ValueError("buf must hold R*S*K rows of H")
    with torch.cuda.device(dev):
        rc = load_library().mep_dispatch(_ptr(hidden), _ptr(dst_pos), _ptr(status), R, S, K, H,
                                         _ptr(buf), _stream(dev))
    _check("mep_dispatch", rc)
    return buf


def mep_combine(y, topk_w, dst_pos, status, R: int, S: int, K: int, out=None):
    """out[t] = bf16(sum_k topk_w[t, k] * y[dst_pos[t, k]]) (fp32 fma in k order)."""
    torch = _torch()
    _need(y, "y", torch.bfloat16)
    H = y.shape[-1]
    N = R * S
    if y.numel() != N * K * H:
        raise ValueError("y must hold R*S*K rows of H")
    dev = y.device
    _need(topk_w, "topk_w", torch.float32, (N, K), dev)
    _need(dst_pos, "dst_pos", torch.int32, (N, K), dev)
    if status is not None:
        _need(status, "status", torch.int32, (1,), dev)
    if out is None:
        out = torch.empty((N, H), dtype=torch.bfloat16, device=dev)
    else:
        _need(out, "out", torch.bfloat16, (N, H), dev)
    with torch.cuda.device(dev):
        rc = load_library().mep_combine(_ptr(y), _ptr(topk_w), _ptr(dst_pos), _ptr(status),
                                        R, S, K, H, _ptr(out), _stream(dev))
    _check("mep_combine", rc)
    return out


def mep_reduce_grad(slot_expert, home_grad, slot_grad, status, E: int):
    """home_grad[e] += slots of e in (r, b) order; consumed slots zeroed. In place.

    home_grad: fp32 [E, ...]; slot_grad: fp32 [R, B, ...] with the same
    trailing element count (H*H'); slot_expert: int32 [R, B].
    """
    torch = _torch()
    _need(slot_expert, "slot_expert", torch.int32)
    R, B = slot_expert.shape
    dev = slot_expert.device
    _need(home_grad, "home_grad", torch.float32, None, dev)
    _need(slot_grad, "slot_grad", torch.float32, None, dev)
    if home_grad.numel() % E:
        raise ValueError("home_grad must be [E, H*H']")
    HHp = home_grad.numel() // E
    if slot_grad.numel() != R * B * HHp:
        raise ValueError("slot_grad must be [R, B, H*H']")
    if status is not None:
        _need(status, "status", torch.int32, (1,), dev)
    with torch.cuda.device(dev):
        rc = load_library().mep_reduce_grad(_ptr(slot_expert), E, R, B, HHp, _ptr(home_grad),
                                            _ptr(slot_grad), _ptr(status), _stream(dev))
    _check("mep_reduce_grad", rc)
    return home_grad, slot_grad


def mep_prefetch(slot_expert, home_w, slot_w, status, E: int):
    """slot_w[r, b] = home_w[slot_expert[r, b]] for every used slot (in place).

    home_w: [E, ...]; slot_w: [R, B, ...] with the same dtype and trailing
    size; slot_expert: int32 [R, B]. Any dtype (the copy is bytewise).
    """
    torch = _torch()
    _need(slot_expert, "slot_expert", torch.int32)
    R, B = slot_expert.shape
    dev = slot_expert.device
    _need(home_w, "home_w", home_w.dtype, None, dev)
    _need(slot_w, "slot_w", home_w.dtype, None, dev)
    nbytes = home_w.numel() * home_w.element_size()
    if nbytes % E:
        raise ValueError("home_w must be [E, ...]")
    per = nbytes // E
    if slot_w.numel() * slot_w.element_size() != R * B * per:
        raise ValueError("slot_w must be [R, B, ...] with home_w's trailing size")
    if status is not None:
        _need(status, "status", torch.int32, (1,), dev)
    with torch.cuda.device(dev):
        rc = load_library().mep_prefetch(_ptr(slot_expert), E, R, B, per, _ptr(home_w),
                                         _ptr(slot_w), _ptr(status), _stream(dev))
    _check("mep_prefetch", rc)
    return slot_w


def mep_dispatch_backward(dbuf, dst_pos, status, R: int, S: int, K: int, dhidden=None):
    """dhidden[t] = bf16(sum_k dbuf[dst_pos[t, k]]) (fp32 adds in k order)."""
    torch = _torch()
    _need(dbuf, "dbuf", torch.bfloat16)
    H = dbuf.shape[-1]
    N = R * S
    if dbuf.numel() != N * K * H:
        raise ValueError("dbuf must hold R*S*K rows of H")
    dev = dbuf.device
    _need(dst_pos, "dst_pos", torch.int32, (N, K), dev)
    if status is not None:
        _need(status, "status", torch.int32, (1,), dev)
    if dhidden is None:
        dhidden = torch.empty((N, H), dtype=torch.bfloat16, device=dev)
    else:
        _need(dhidden, "dhidden", torch.bfloat16, (N, H), dev)
    with torch.cuda.device(dev):
        rc = load_library().mep_dispatch_backward(_ptr(dbuf), _ptr(dst_pos), _ptr(status), R, S, K,
                                                  H, _ptr(dhidden), _stream(dev))
    _check("mep_dispatch_backward", rc)
    return dhidden


def mep_combine_backward(dout, y, topk_w, dst_pos, status, R: int, S: int, K: int, dy=None,
                         dw=None):
    """(dy, dw) with dy[dst_pos[t,k]] = bf16(w[t,k] * dout[t]) and
    dw[t,k] = <dout[t], y[dst_pos[t,k]]> (fp32)."""
    torch = _torch()
    _need(dout, "dout", torch.bfloat16)
    N, H = dout.shape
    if N != R * S:
        raise ValueError("dout must be [R*S, H]")
    dev = dout.device
    _need(y, "y", torch.bfloat16, None, dev)
    if y.numel() != N * K * H:
        raise ValueError("y must hold R*S*K rows of H")
    _need(topk_w, "topk_w", torch.float32, (N, K), dev)
    _need(dst_pos, "dst_pos", torch.int32, (N, K), dev)
    if status is not None:
        _need(status, "status", torch.int32, (1,), dev)
    if dy is None:
        dy = torch.empty((N * K, H), dtype=torch.bfloat16, device=dev)
    else:
        _need(dy, "dy", torch.bfloat16, None, dev)
        if dy.numel() != N * K * H:
            raise ValueError("dy must hold R*S*K rows of H")
    if dw is None:
        dw = torch.empty((N, K), dtype=torch.float32, device=dev)
    else:
        _need(dw, "dw", torch.float32, (N, K), dev)
    with torch.cuda.device(dev):
        rc = load_library().mep_combine_backward(_ptr(dout), _ptr(y), _ptr(topk_w), _ptr(dst_pos),
                                                 _ptr(status), R, S, K, H, _ptr(dy), _ptr(dw),
                                                 _stream(dev))
    _check("mep_combine_backward", rc)
    return dy, dw


def mep_grouped_gemm(x, cu_seqlens, w_home, w_slot, status, R: int, S: int, K: int,
                     y=None, workspace=None):
    """y[row] = bf16(x[row] @ W_j) for the group j of every buffer row.

    x: bf16 [R*S*K, H] (the dispatch buffer); cu_seqlens: int32 [R, E+B];
    w_home: bf16 [E, H, H']; w_slot: bf16 [R, B, H, H'] (None when B == 0).
    Group j of rank r uses w_home[j] below E and w_slot[r, j - E] above.
    Returns y, bf16 [R*S*K, H'].
    """
    torch = _torch()
    _need(x, "x", torch.bfloat16)
    dev = x.device
    _need(w_home, "w_home", torch.bfloat16, None, dev)
    E, H, Hp = w_home.shape
    _need(cu_seqlens, "cu_seqlens", torch.int32, None, dev)
    if cu_seqlens.dim() != 2 or cu_seqlens.shape[0] != R:
        raise ValueError("cu_seqlens must be [R, E+B]")
    B = cu_seqlens.shape[1] - E
    if B < 0:
        raise ValueError("cu_seqlens must have E+B columns")
    if x.numel() != R * S * K * H:
        raise ValueError("x must hold R*S*K rows of H")
    if B > 0:
        _need(w_slot, "w_slot", torch.bfloat16, (R, B, H, Hp), dev)
    if status is not None:
        _need(status, "status", torch.int32, (1,), dev)
    if y is None:
        y = torch.empty((R * S * K, Hp), dtype=torch.bfloat16, device=dev)
    else:
        _need(y, "y", torch.bfloat16, (R * S * K, Hp), dev)
    need = grouped_gemm_workspace_bytes(R, S, K, E, B)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        rc = load_library().mep_grouped_gemm(_ptr(x), _ptr(cu_seqlens), _ptr(w_home),
                                             _ptr(w_slot) if B > 0 else None, _ptr(status), R, S,
                                             K, E, B, H, Hp, _ptr(workspace), need, _ptr(y),
                                             _stream(dev))
    _check("mep_grouped_gemm", rc)
    return y


def mep_wait_selftest(limit_ns: int, device=None):
    """Run the bounded-wait self-test on the device; returns (status, elapsed_ns)
    tensors (int32 [1], int64 [1]) after it is enqueued (not synchronised)."""
    torch = _torch()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    elapsed = torch.zeros(1, dtype=torch.int64, device=dev)
    with torch.cuda.device(dev):
        rc = load_library().mep_wait_selftest(_ptr(status), int(limit_ns), _ptr(elapsed),
                                              _stream(dev))
    _check("mep_wait_selftest", rc)
    return status, elapsed
