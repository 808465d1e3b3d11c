import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long CPU-side oracle work")


def pytest_collection_modifyitems(config, items):
    # GPU tests are skipped (not failed) on a machine without a CUDA device, so a bare
    # `pytest tests/` stays green on CPU; `-m gpu` on a GPU machine runs them for real.
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session")
def oracle_pool():
    """Spawned worker processes that run the oracle on every row of a full-size call."""
    from oracle_pool import OraclePool
    pool = OraclePool()
    yield pool
    pool.close()
