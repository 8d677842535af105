import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running parity case")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(autouse=True)
def _parity_test_id(request):
    """Labels the parity comparisons a test makes (tests/parity.py)."""
    try:
        import parity
    except Exception:  # the CPU-only environment may lack torch's CUDA parts; parity needs none
        yield
        return
    parity.CURRENT["test"] = request.node.nodeid.split("::", 1)[-1]
    yield


def pytest_sessionfinish(session, exitstatus):
    path = os.environ.get("GDR_PARITY_REPORT")
    if not path:
        return
    try:
        import parity
    except Exception:
        return
    if parity.RECORDS:
        parity.write_report(path)
