import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 GPU (sm_103a) and the built CUDA library")


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library, built in-tree if missing (nvcc cross-compiles without a GPU)."""
    from mixture_experts_gemm_gb300 import _build
    _build.build()
    import mixture_experts_gemm_gb300 as m
    return m.lib()
