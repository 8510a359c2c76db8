import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


def _has_gpu() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def native_lib():
    """The C-ABI library, built in-tree if it is missing or stale."""
    from gemm_conv_epilogues_gb300 import build as gbuild
    gbuild.build_library()
    from gemm_conv_epilogues_gb300 import binding
    return binding.lib()


@pytest.fixture(scope="session")
def cuda_ready(native_lib):
    if not _has_gpu():
        pytest.fail("GPU test selected but torch.cuda.is_available() is False")
    import torch
    torch.cuda.init()
    return native_lib
