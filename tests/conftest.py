"""Shared test configuration.

Markers: ``gpu`` marks tests that need a GB300 (sm_103a) and the CUDA
library. Everything else runs on a CPU-only machine.
"""

from __future__ import annotations

import os
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

GOLDEN = Path(__file__).resolve().parent / "golden"


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs an sm_103a GPU and libbfp8.so")


@pytest.fixture(scope="session")
def bfp8():
    """The ctypes binding, building libbfp8.so first if it is missing or stale."""
    from block_scaled_fp8_token_gb300 import build

    build.build()
    from block_scaled_fp8_token_gb300 import bfp8 as mod

    return mod


@pytest.fixture(scope="session")
def cuda_device(bfp8):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    major, minor = torch.cuda.get_device_capability(0)
    if (major, minor) != (10, 3):
        pytest.skip(f"needs sm_103 (GB300), found sm_{major}{minor}")
    return torch.device("cuda:0")
