"""Helpers for the GPU parity tests: numpy <-> torch device transfers."""

import numpy as np
import torch

DEV = torch.device("cuda:0")


def to_dev(a: np.ndarray):
    """numpy -> device tensor; uint16 arrays are treated as bf16 bit patterns."""
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def to_np(t) -> np.ndarray:
    """device tensor -> numpy; bf16 becomes uint16 bit patterns."""
    t = t.detach()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def bf16_ulp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """|a - b| in units of bf16 ulps, for finite bf16 bit patterns of equal sign."""
    def key(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, -(x & 0x7FFF), x)
    return np.abs(key(a) - key(b))
