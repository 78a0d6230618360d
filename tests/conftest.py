import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but CUDA is not available")
    return torch.device("cuda:0")


@pytest.fixture(autouse=True)
def device_status_clean(request):
    """After every GPU test: no kernel may have raised a device status bit
    (an expired bounded wait).  A test that provokes one reads and clears the
    status itself."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    import torch
    if not torch.cuda.is_available():
        return
    import deterministic_w8a8_int8_gb300 as prism
    status = prism.prism_device_status()
    assert status == 0, f"device status bits raised during the test: {status:#x}"
