import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size parity case (minutes)")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.load()


@pytest.fixture(scope="session")
def kda():
    """The CUDA library binding; GPU tests fail loudly when it is missing."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without CUDA")
    import kda_gated_delta_chunkwise_gb300 as k
    k.load()  # raises if the shared library is missing
    k.device_errors(reset=True)
    return k


@pytest.fixture(autouse=True)
def _no_device_errors(request):
    """Every GPU test must leave the device error word clear (no kernel gave
    up on a bounded wait)."""
    yield
    if request.node.get_closest_marker("gpu") is not None:
        import kda_gated_delta_chunkwise_gb300 as k
        errs = k.device_errors(reset=True)
        assert errs == 0, f"a kernel reported device error {errs}"
