import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libvsf.so")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes)")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device in this process")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(autouse=True)
def _bounds_checked_on_close(monkeypatch):
    """Under the bounds-checking build (VSF_LIBRARY set), every ShardStep
    must close with no failed index check (bit 4 of its device error word)."""
    if not os.environ.get("VSF_LIBRARY"):
        yield
        return
    import torch
    from fsdp_buffer_layout_gb300 import step
    orig = step.ShardStep.close

    def close(self):
        if self.plan:
            torch.cuda.synchronize()
            assert self.device_error() & 4 == 0, "a kernel's index check failed"
        orig(self)

    monkeypatch.setattr(step.ShardStep, "close", close)
    yield
