"""pytest configuration: markers and shared fixtures.

``-m "not gpu"`` runs the oracle pins, the host-side logic and the C-ABI
symbol checks; ``-m gpu`` runs the parity tests, which call the CUDA path
through the C-ABI and compare it with the fp64 oracle.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes)")


@pytest.fixture(scope="session")
def orc():
    """The fp64 oracle built from the committed source."""
    import oracle

    return oracle.default()
