"""Shared fixtures.  `-m gpu` tests need a CUDA device and the built library;
everything else runs on the CPU."""
import os
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the built CUDA library")


@pytest.fixture(scope="session")
def orc():
    """The oracle; ORACLE_LIB points the pins at another build of oracle.c
    (the planted-mistake test uses this)."""
    import oracle
    path = os.environ.get("ORACLE_LIB")
    return oracle.Oracle(path) if path else oracle.get()


@pytest.fixture(autouse=True)
def _checked_build_stays_in_bounds(request):
    """With WC_EXPECT_CHECKED=1 (the library named by WC_LIBRARY is the
    bounds-checked build), every GPU test must leave no skipped access."""
    yield
    if os.environ.get("WC_EXPECT_CHECKED") != "1" or request.node.get_closest_marker("gpu") is None:
        return
    import torch
    from weight_communication_gb300 import binding
    torch.cuda.synchronize()
    n = binding.checked_violations(reset=True)
    assert n == 0, binding.last_error()
