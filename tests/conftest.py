import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds on the host")


def pytest_collection_modifyitems(config, items):
    """GPU tests fail loudly when no GPU is present: they are never silently skipped
    on a run that selected them with -m gpu, so a box without a working device shows
    up as failures rather than as a green run."""
    return None
