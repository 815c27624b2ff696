"""Test configuration: the `gpu` marker and shared helpers.

Tests marked `gpu` need a CUDA device and the compiled library; everything
else runs on the CPU (oracle pins, host-side policy, ABI symbol checks).
"""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300) and the compiled libpd.so")


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device in this process")
    return torch.device("cuda:0")
