"""pytest configuration: the ``gpu`` marker and shared fixtures.

Tests marked ``gpu`` need a CUDA device and the compiled GPU library; everything else runs on
a host without a GPU (the CPU oracle and its pins, host-side argument checks, the library's
exported symbols, the two-rank gloo sharding check).
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the compiled GPU library")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle

    return oracle.default()


@pytest.fixture(scope="session")
def cuda_device():
    import torch

    if not torch.cuda.is_available():
        pytest.fail("a test marked gpu ran on a host without a CUDA device")
    return torch.device("cuda:0")


@pytest.fixture(scope="session")
def rrn(cuda_device):
    """The GPU library's Python binding (fails loudly if the library was not built)."""
    import residual_rmsnorm_row_gb300 as rrn_mod

    rrn_mod.load_library()
    return rrn_mod
