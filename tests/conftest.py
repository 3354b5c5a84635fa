"""Shared pytest configuration: the ``gpu`` marker and the repository root on sys.path."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: CPU test that takes more than a few seconds")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


@pytest.fixture(autouse=True)
def _device_error_word(request):
    """GPU tests: the library's sticky device error word must be clear after every test (read and cleared)."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    import torch
    if not torch.cuda.is_available():
        return
    import medusa_tree_speculative_verify_gb300 as mv
    st, code, detail = mv.get_error(with_detail=True)
    assert st == 0, f"device error word set during {request.node.name}: {code:#x} (detail {detail:#x})"
