"""Shared pytest configuration.

Tests marked ``gpu`` need a CUDA device and the built ``libfp8q.so``; everything
else runs on the CPU.  The CPU oracle (``oracle/``) is compiled on first use.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workload check (minutes on the CPU oracle)")


@pytest.fixture(scope="session")
def oracle():
    import oracle as o
    o.lib()
    return o
