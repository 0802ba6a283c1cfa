"""Shared test set-up.

Markers:
  gpu -- needs a CUDA device (the parity tests proper, run through the C ABI).
Everything unmarked runs on a CPU-only host: the oracle against its pins,
the host-side argument checks of the C ABI, the exported-symbol check and the
multi-process (gloo) bench plumbing.
"""
from __future__ import annotations

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a); runs the CUDA path through the C ABI")


@pytest.fixture(scope="session")
def cuda_lib_path():
    """Path of the CUDA library, built in-tree if it is missing or stale."""
    from fp8_fine_grained_act_gb300 import build as b
    return b.build()


@pytest.fixture(scope="session")
def gpu_device():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("test marked gpu but no CUDA device is visible")
    from fp8_fine_grained_act_gb300 import build as b
    b.build()
    return torch.device("cuda:0")
