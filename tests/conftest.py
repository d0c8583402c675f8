import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.lib()  # build once per session
    return oracle


@pytest.fixture(scope="session")
def dep():
    """The library's Python binding, with the library built for sm_103a."""
    from skinny_bf16_split_gb300 import build as _b
    _b.build()
    import skinny_bf16_split_gb300 as d
    d.lib()
    return d
