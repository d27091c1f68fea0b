import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running case")


def _gpu_available():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # pragma: no cover
        return False


def pytest_collection_modifyitems(config, items):
    if _gpu_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device in this process")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(autouse=True)
def _guard_bands(request, monkeypatch):
    """GPU tests: every output and workspace the binding allocates, and the
    device tensors of tests/gpu_step.py's GpuStep, carry canary bands that
    are checked after every call (the stand-in for an out-of-bounds checker)."""
    if "gpu" not in request.keywords or not _gpu_available():
        yield
        return
    import gpu_step
    import paged_kv_cache_write_gb300 as pkv
    gpu_step.start_guarding(monkeypatch, pkv)
    yield
    gpu_step.stop_guarding()
