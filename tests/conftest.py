import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


@pytest.fixture(autouse=True)
def _bounds_checked_build(request):
    """Under SDV_DEBUG_BOUNDS=1 (the bounds-checked library): after every GPU test that loaded the
    library, no bounds check may have failed (site numbers >= 100 in the status word)."""
    yield
    if os.environ.get("SDV_DEBUG_BOUNDS") != "1" or "gpu" not in request.keywords:
        return
    import speculative_decoding_verify_gb300 as m
    if m._lib is None:
        return
    assert m.build_flags() & 1, "SDV_DEBUG_BOUNDS=1 but the loaded library is the release build"
    st, site = m.device_status_site()
    assert site < 100, f"bounds check failed at site {site} (status {st})"
