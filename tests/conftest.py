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


@pytest.fixture
def stream_k_on():
    """Turns the GEMM's stream-K tail on for one test (it is off by default) and off again."""
    import blackwell_tensor_core_fp16_gb300 as g
    assert g.gemm_f16_set_stream_k(1) == g.OK
    yield
    g.gemm_f16_set_stream_k(0)
