import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running oracle comparison")


@pytest.fixture(scope="session")
def ost():
    """The built CUDA library's Python binding (GPU tests only)."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without CUDA; run with -m 'not gpu'")
    import __graft_entry__
    __graft_entry__.build()
    import online_softmax_tiled_gb300 as pkg
    pkg.lib()
    return pkg


@pytest.fixture(autouse=True)
def _device_status_clean(request):
    """After every GPU test the library's device error word must be clear."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    import online_softmax_tiled_gb300 as pkg
    assert pkg.attn_sync_status() == pkg.ATTN_OK
