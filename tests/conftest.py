import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: longer CPU test")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA GPU in this process")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(autouse=True)
def _no_store_outside_buffers(request):
    """Against a bounds-checked library build (Q4_LIBRARY set), every GPU
    test ends with a q4_check that must not report a store outside its
    buffer."""
    yield
    if not os.environ.get("Q4_LIBRARY") or "gpu" not in request.node.keywords:
        return
    import weight_only_int4_group_gb300 as q4
    assert q4.check() != q4.ERR_BOUNDS, "a kernel store fell outside its buffer"
