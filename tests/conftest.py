import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103) and the built library")
    config.addinivalue_line("markers", "slow: longer CPU-side checks")


def pytest_collection_modifyitems(config, items):
    # GPU tests need a device; skip them loudly (not silently pass) on a CPU host.
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device on this host")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session")
def lib():
    """The built C-ABI library (built here if stale; there is no fallback)."""
    from moe_router_gemm_gb300 import build as _build
    _build.build()
    import moe_router_gemm_gb300 as m
    m.load()
    return m
