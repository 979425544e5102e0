"""Shared test configuration.

Markers: ``gpu`` -- needs a CUDA device and the built library; everything else
runs on the CPU (the oracle, its pins, the host logic, and the C-ABI symbol
check).
"""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: CPU test that takes more than a few seconds")


@pytest.fixture(scope="session")
def repo_root():
    return ROOT


@pytest.fixture(scope="session")
def built_library():
    """Path of libflashsample.so, (re)built in-tree if a source changed."""
    from lm_head_exact_gb300.build import build
    return build()


@pytest.fixture(scope="session")
def fs(built_library):
    """The ctypes binding on a CUDA device (GPU tests only): fails loudly --
    never skips -- when no device is present, so a GPU run cannot pass
    without executing the kernels."""
    import torch
    assert torch.cuda.is_available(), "GPU test run without a CUDA device"
    from lm_head_exact_gb300 import binding
    binding.library()
    binding.set_path(binding.FS_PATH_AUTO)
    return binding


@pytest.fixture(scope="session")
def torch_cuda():
    import torch
    assert torch.cuda.is_available(), "GPU test run without a CUDA device"
    return torch
