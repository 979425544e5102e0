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


def pytest_terminal_summary(terminalreporter):
    """Near-tie statistics of the oracle comparisons run by this session:
    rows compared, rows whose oracle top-two gap is inside the band, and id
    mismatches (all of which must be inside the band)."""
    try:
        from _helpers import BAND_LOG
    except ImportError:
        return
    big = [r for r in BAND_LOG if r[1] >= 256]
    if not big:
        return
    tr = terminalreporter
    tr.write_sep("-", "oracle comparisons of >= 256 rows: rows / in-band rows / id mismatches")
    for what, n, n_band, n_mis in big:
        tr.write_line(f"{what}: {n} rows, {n_band} in band, {n_mis} mismatches")
    tot = sum(r[1] for r in BAND_LOG)
    tr.write_line(f"all comparisons: {tot} rows, {sum(r[2] for r in BAND_LOG)} in band, "
                  f"{sum(r[3] for r in BAND_LOG)} mismatches")
