import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size oracle comparisons (tens of seconds)")


@pytest.fixture(scope="session", autouse=True)
def _built_host_parts():
    """The oracle and the host generator are plain C: (re)build them once per session."""
    from gen import gen
    from oracle import oracle
    if os.environ.get("COLI_ORACLE_SO") or os.environ.get("COLI_TIER_HOST_SO"):
        yield  # a child run against prebuilt (sanitized) libraries: build nothing here
        return
    gen.build(cuda=False)
    oracle.build()
    yield
