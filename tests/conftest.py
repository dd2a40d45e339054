import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle._load()


# The test process loads several native runtimes at once (the CUDA runtime,
# with or without a driver; OpenMP through the oracle and through torch; gloo
# through the multi-rank tests). Interpreter teardown after a complete, passing
# session crashed intermittently in their destructors, so the session ends
# with the status pytest computed, without running them.
_EXIT_STATUS = None


def pytest_sessionfinish(session, exitstatus):
    global _EXIT_STATUS
    _EXIT_STATUS = int(exitstatus)


def pytest_unconfigure(config):
    if _EXIT_STATUS is None or os.environ.get("KVD_TEST_NORMAL_EXIT"):
        return
    sys.stdout.flush()
    sys.stderr.flush()
    os._exit(_EXIT_STATUS)
