import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def oracle():
    from oracle import Oracle
    return Oracle()


@pytest.fixture(scope="session")
def situ_lib():
    """libsitu built for sm_103a (rebuilt only when a source changed)."""
    from situ_glu_activation_gb300 import _native
    from situ_glu_activation_gb300.build import build

    build()
    return _native.lib()


@pytest.fixture(scope="session")
def cuda_dev(situ_lib):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _clean_device_status(request):
    """GPU tests start and end with a clear device status word."""
    if request.node.get_closest_marker("gpu") is None:
        yield
        return
    request.getfixturevalue("cuda_dev")
    import situ_glu_activation_gb300 as situ

    situ.device_status(clear=True)
    yield
    import torch

    torch.cuda.synchronize()
    assert situ.device_status(clear=True) == 0, "a kernel recorded a device-side failure"
