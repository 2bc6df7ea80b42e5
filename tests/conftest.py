import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the CUDA library")


def _has_gpu() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    # GPU tests fail loudly (never skip silently) when run with -m gpu on a box
    # without a GPU; on a CPU-only run they are deselected by -m "not gpu".
    pass


@pytest.fixture(scope="session")
def gpu_lib():
    """The CUDA library, loaded; GPU tests use it through its C ABI."""
    if not _has_gpu():
        pytest.fail("GPU test selected but torch.cuda.is_available() is False")
    import weight_only_int4_repack_gb300 as w4
    return w4
