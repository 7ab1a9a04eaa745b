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
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running check")
    # build (or refresh) the oracle and the CUDA library before collection;
    # both are no-ops when the built files are newer than their sources
    import oracle
    from draft_verification_02_b300 import build as cuda_build
    oracle.build()
    cuda_build.build()
    cuda_build.build(debug=True)


@pytest.fixture(scope="session")
def orc():
    """The C oracle (built on demand)."""
    import oracle
    oracle.load()
    return oracle


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(TESTS, "golden")
