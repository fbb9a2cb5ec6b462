import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
for p in (ROOT, os.path.dirname(os.path.abspath(__file__))):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running case (full-size problems)")


@pytest.fixture(scope="session")
def lib():
    """The compiled C library (built in-tree on first use; nvcc cross-compiles without a GPU)."""
    from dense_fp32_gemm_04_gb300 import _build
    import dense_fp32_gemm_04_gb300 as sg

    _build.build()
    return sg.library()
