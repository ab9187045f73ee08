import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    # GPU tests without a GPU are an error on a GPU machine, but here (no GPU) they
    # are only deselected by -m "not gpu"; if someone runs them anyway, skip.
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


@pytest.fixture(autouse=True)
def _guard_bands(request):
    """GPU tests: guard bands around the layer helpers' device buffers, checked after the test."""
    if "gpu" not in request.keywords:
        yield
        return
    try:
        import torch
        if not torch.cuda.is_available():
            yield
            return
    except Exception:  # pragma: no cover
        yield
        return
    from mamba_ssm_layer_gb300 import layer
    from tests.helpers import GuardBands
    g = GuardBands()
    prev = layer.set_allocator(g.alloc)
    try:
        yield
    finally:
        layer.set_allocator(prev)
    g.check()
