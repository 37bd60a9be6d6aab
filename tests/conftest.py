import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload parity (minutes)")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


@pytest.fixture(params=["single", "pair"])
def fwd_kernel(request):
    """Runs a bf16 forward test once with each forward kernel (one CTA per SM,
    and SM pairs); the choice is process-wide, so it is reset afterwards."""
    import ring_attention_fwd_gb300 as ra
    ra.set_fwd_kernel(request.param)
    yield request.param
    ra.set_fwd_kernel("single")
