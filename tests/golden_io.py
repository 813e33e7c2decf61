"""Reader for the small text fixtures under tests/golden/."""

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name: str) -> dict:
    """Parse ``key v1 v2 ...`` lines; '#' starts a comment line."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if len(vals) == 1 and not _is_num(vals[0]):
                out[key] = vals[0]
            elif all(_is_int(v) for v in vals):
                out[key] = np.array([int(v) for v in vals], dtype=np.int64)
            else:
                out[key] = np.array([float(v) for v in vals], dtype=np.float64)
    return out


def load_hex_pairs(name: str):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            a, b, *_ = line.split()
            rows.append((int(a, 16), int(b, 16)))
    return rows


def _is_int(s):
    try:
        int(s)
        return True
    except ValueError:
        return False


def _is_num(s):
    try:
        float(s)
        return True
    except ValueError:
        return False
