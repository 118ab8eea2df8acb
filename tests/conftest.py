import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda", 0)


@pytest.fixture(autouse=True)
def _guard_bands():
    """Checks, when each test ends, the guard bands its buffers were given."""
    yield
    from tests import guards
    if guards.registered():
        guards.check_guards()


def pytest_sessionfinish(session, exitstatus):
    """Writes the list-verdict tallies when ASP_PARITY_REPORT names a file."""
    if "tests.parity" in sys.modules:
        sys.modules["tests.parity"].write_report()
