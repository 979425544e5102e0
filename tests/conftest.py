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
