"""Test configuration: the ``gpu`` marker and shared helpers.

``-m "not gpu"`` runs the oracle's pins, the generators and the host-side
checks of the C-ABI library (it loads and exports its symbols; argument
validation that returns before any CUDA call).  ``-m gpu`` runs the parity
tests of the CUDA path against the oracle through the C-ABI.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_collection_modifyitems(config, items):
    # GPU tests fail loudly (not skip) when no GPU is present and they were selected.
    pass


def gpu_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False
