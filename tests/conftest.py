"""Shared pytest set-up.

Markers:
  gpu -- needs a CUDA device and the built ``libtm.so``; the CPU suite runs with
         ``-m "not gpu"``.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the built libtm.so")


def read_golden(name):
    """Rows of a golden fixture: whitespace-separated fields, '#' comments skipped."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


@pytest.fixture(scope="session")
def oracle():
    import oracle as _oracle
    _oracle.build()
    return _oracle


@pytest.fixture(scope="session")
def cuda():
    """Skip when no GPU is present; fail loudly when the GPU is present but the
    CUDA library cannot be loaded."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from masking_tm_affine_gb300 import tm
    tm.load()  # raises if libtm.so is missing or does not load
    return tm
