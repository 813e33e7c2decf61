"""Host-side checks of the C ABI: the library loads, exports every function
that include/mep.h declares, and rejects bad arguments before touching the GPU."""

import ctypes
import os
import re

import pytest

import load_balancing_topk_gb300 as mep
from load_balancing_topk_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return mep.load_library()


def declared_functions():
    names = []
    for f in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            names += re.findall(r"^MEP_API\s+[\w\s\*]+?\b(mep_\w+)\s*\(", text, re.M)
    return names


def test_header_declares_the_four_steps():
    names = declared_functions()
    for n in ("mep_plan", "mep_dispatch", "mep_combine", "mep_reduce_grad",
              "mep_plan_workspace_bytes", "mep_status_string", "mep_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n
    # the binding's signature table covers exactly the declared functions
    assert sorted(n for n, _, _ in mep.SIGNATURES) == sorted(declared_functions())


def test_status_strings(lib):
    for code in mep.STATUS:
        assert mep.status_string(code) != "unknown status"
    assert mep.status_string(99) == "unknown status"
    assert mep.version() >= (0, 1)


def test_plan_kernel_count(lib):
    # k_hist, k_plan, k_offsets; k_gsum too once the tile counts reach 128 KB
    assert mep.plan_kernel_count(8, 4096, 6, 64, 8) == 3      # 128 tiles x 64 experts
    assert mep.plan_kernel_count(8, 8192, 8, 256, 32) == 4    # 256 tiles x 256 experts
    assert mep.plan_kernel_count(2, 0, 2, 8, 4) == 1          # no tokens: the planner alone
    with pytest.raises(mep.MepError):
        mep.plan_kernel_count(3, 10, 2, 8, 4)


def test_workspace_bytes(lib):
    b = mep.plan_workspace_bytes(8, 8192, 8, 256, 32)
    # per-tile histograms: 128 tiles x 256 experts x 4 bytes, plus tables
    assert b >= 128 * 256 * 4
    assert mep.plan_workspace_bytes(2, 0, 2, 8, 4) > 0


@pytest.mark.parametrize("args", [
    (3, 10, 2, 8, 4),      # E % R != 0
    (2, 10, 9, 8, 4),      # K > E
    (2, 10, 0, 8, 4),      # K < 1
    (0, 10, 2, 8, 4),      # R < 1
    (2, -1, 2, 8, 4),      # S < 0
    (2, 10, 2, 8, -1),     # B < 0
    (2, 10, 2, 8192, 4),   # E > MEP_MAX_E
    (2, 10, 65, 128, 4),   # K > MEP_MAX_K
    (2, 2**30, 8, 8, 4),   # R*S*K overflows int32 rows
])
def test_plan_rejects_bad_sizes(lib, args):
    out = ctypes.c_size_t(0)
    assert lib.mep_plan_workspace_bytes(*args, ctypes.byref(out)) == mep.STATUS_CODE["MEP_ERR_INVALID_ARG"]
    R, S, K, E, B = args
    rc = lib.mep_plan(None, R, S, K, E, B, None, 0, None, None, None, None, None, None)
    assert rc == mep.STATUS_CODE["MEP_ERR_INVALID_ARG"]


def test_plan_rejects_null_and_small_workspace(lib):
    bad = mep.STATUS_CODE["MEP_ERR_INVALID_ARG"]
    # null workspace / outputs: refused before anything is launched
    assert lib.mep_plan(16, 2, 4, 2, 8, 4, None, 0, 16, 16, 16, 16, 16, None) == bad
    need = mep.plan_workspace_bytes(2, 4, 2, 8, 4)
    assert lib.mep_plan(16, 2, 4, 2, 8, 4, 256, need - 1, 16, 16, 16, 16, 16, None) == bad
    # misaligned topk_idx
    assert lib.mep_plan(18, 2, 4, 2, 8, 4, 256, need, 16, 16, 16, 16, 16, None) == bad


def test_permute_rejects_bad_args(lib):
    bad = mep.STATUS_CODE["MEP_ERR_INVALID_ARG"]
    assert lib.mep_dispatch(16, 16, None, 2, 4, 2, 12, 16, None) == bad        # H % 8
    assert lib.mep_dispatch(None, 16, None, 2, 4, 2, 16, 16, None) == bad      # null
    assert lib.mep_dispatch(24, 16, None, 2, 4, 2, 16, 16, None) == bad        # misaligned
    assert lib.mep_combine(16, None, 16, None, 2, 4, 2, 16, 16, None) == bad   # null weights
    assert lib.mep_combine(16, 16, 16, None, 2, 4, 0, 16, 16, None) == bad     # K < 1
    # empty input is a no-op that needs no pointers
    assert lib.mep_dispatch(None, None, None, 2, 0, 2, 16, None, None) == 0
    assert lib.mep_combine(None, None, None, None, 2, 0, 2, 16, None, None) == 0


def test_reduce_grad_rejects_bad_args(lib):
    bad = mep.STATUS_CODE["MEP_ERR_INVALID_ARG"]
    assert lib.mep_reduce_grad(16, 0, 2, 2, 8, 16, 16, None, None) == bad     # E < 1
    assert lib.mep_reduce_grad(16, 4, 2, 2, -1, 16, 16, None, None) == bad    # HHp < 0
    assert lib.mep_reduce_grad(None, 4, 2, 2, 8, 16, 16, None, None) == bad   # null map
    assert lib.mep_reduce_grad(16, 4, 2, 2, 8, 20, 16, None, None) == bad     # misaligned
    assert lib.mep_reduce_grad(None, 4, 2, 0, 8, None, None, None, None) == 0  # no slots


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    monkeypatch.setattr(mep, "_lib", None)
    monkeypatch.setattr(mep, "_PKG", str(tmp_path))
    with pytest.raises(RuntimeError, match="missing"):
        mep.load_library()


def test_prefetch_rejects_bad_args(lib):
    bad = mep.STATUS_CODE["MEP_ERR_INVALID_ARG"]
    assert lib.mep_prefetch(16, 0, 2, 2, 64, 16, 16, None, None) == bad     # E < 1
    assert lib.mep_prefetch(16, 4, 2, 2, 24, 16, 16, None, None) == bad     # bytes % 16
    assert lib.mep_prefetch(16, 4, 2, 2, -16, 16, 16, None, None) == bad    # bytes < 0
    assert lib.mep_prefetch(None, 4, 2, 2, 64, 16, 16, None, None) == bad   # null map
    assert lib.mep_prefetch(16, 4, 2, 2, 64, 24, 16, None, None) == bad     # misaligned
    assert lib.mep_prefetch(None, 4, 2, 0, 64, None, None, None, None) == 0  # no slots


def test_wait_selftest_rejects_bad_args(lib):
    bad = mep.STATUS_CODE["MEP_ERR_INVALID_ARG"]
    assert lib.mep_wait_selftest(None, 1000, 16, None) == bad          # null status
    assert lib.mep_wait_selftest(16, 1000, None, None) == bad          # null elapsed
    assert lib.mep_wait_selftest(16, -1, 16, None) == bad              # negative limit
    assert lib.mep_wait_selftest(16, 10**10 + 1, 16, None) == bad      # limit beyond 10 s

