import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HERE = os.path.dirname(os.path.abspath(__file__))
for p in (ROOT, HERE):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(autouse=True)
def _no_expired_device_wait(request):
    """After every GPU test that loaded the library: no bounded wait inside a
    kernel expired (the device flag reads clear)."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    from memory_bound_weight_gb300 import _binding

    if _binding._lib is not None:
        _binding.check_device_error()
