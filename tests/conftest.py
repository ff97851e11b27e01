import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: CPU test that takes more than a few seconds")


def pytest_collection_modifyitems(config, items):
    # GPU tests cannot run without a device; fail loudly rather than skip
    # when the caller asked for them explicitly on a machine without one.
    pass


@pytest.fixture(autouse=True)
def _guard_regions(request, monkeypatch):
    """GPU tests: the layers' buffers (pipeline._u8 / pipeline._empty) get
    guard regions too, and every guard of the test is checked when it ends."""
    if request.node.get_closest_marker("gpu") is None:
        yield
        return
    from precision_moe_numerics_nvfp4_gb300 import pipeline as PL
    from tests import gpu_helpers as gh
    monkeypatch.setattr(PL, "_u8", lambda n, dev: gh.guarded_bytes(max(int(n), 16)))
    monkeypatch.setattr(PL, "_empty", lambda shape, dtype, dev: gh.gempty(shape, dtype=dtype, device=dev))
    try:
        yield
        gh.check_guards()
    finally:
        gh.clear_guards()
