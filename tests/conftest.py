import os
import sys

import pytest

_ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_TESTS = os.path.dirname(os.path.abspath(__file__))
for p in (_ROOT, _TESTS):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running test")


@pytest.fixture(scope="session")
def orc_lib():
    import oracle
    return oracle.load()


@pytest.fixture(autouse=True)
def _output_guard_bands():
    """After every test: no kernel wrote into the guard bands of the outputs it allocated."""
    yield
    gu = sys.modules.get("gpu_util")
    if gu is not None:
        gu.check_guards()
