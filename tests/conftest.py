import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built liblora.so")


import pytest  # noqa: E402


@pytest.fixture(autouse=True)
def _no_device_error(request):
    """After every GPU test: no kernel may have flagged a device-side error
    (a bounded wait that ran out)."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    import torch
    if not torch.cuda.is_available():
        return
    from lora_rank_adapter_gb300 import binding
    torch.cuda.synchronize()
    assert binding.lora_device_error() == 0, "a kernel flagged a device-side error"
