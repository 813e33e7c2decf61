"""The package smoke check runs on the GPU and loads the in-tree library."""

import pytest

pytestmark = pytest.mark.gpu


def test_smoke():
    import __graft_entry__

    __graft_entry__.smoke()
    import load_balancing_topk_gb300 as mep

    assert mep._lib is not None and mep.library_path().endswith("libmep.so")
