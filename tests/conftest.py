import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
for _p in (ROOT, os.path.dirname(os.path.abspath(__file__))):
    if _p not in sys.path:
        sys.path.insert(0, _p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running (exhaustive sweeps)")


@pytest.fixture(scope="session")
def orc():
    import oracle

    oracle.build()
    return oracle


from gpu_helpers import moe  # noqa: E402,F401  (session fixture for -m gpu tests)
