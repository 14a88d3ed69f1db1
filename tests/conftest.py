import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU check")


def gpu_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if gpu_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.lib()


@pytest.fixture(autouse=True)
def _bounds_check_word(request):
    """With GS2D_CHECKED=1 (the bounds-checked library), every GPU test must
    leave the device check word at zero: no index taken from data fell
    outside the buffer it addresses."""
    yield
    if os.environ.get("GS2D_CHECKED") != "1" or request.node.get_closest_marker("gpu") is None:
        return
    from raster_gaussian_02_b300 import gs2d
    if gs2d._lib is None:
        return
    st, word = gs2d.gs2d_debug_check_word(clear=True)
    assert st == gs2d.GS2D_OK, gs2d.status_string(st)
    assert word == 0, f"bounds checks failed: word {word:#x}"
