"""Failure detection on the GPU without a fault: a bounded wait gives up, records
SITU_ERR_TIMEOUT in the device status, and the context stays usable."""
import pytest
import torch

import situ_glu_activation_gb300 as situ
from situ_glu_activation_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives(cuda_dev):
    situ.selftest_bounded_wait(limit_us=2000)
    torch.cuda.synchronize()
    assert situ.device_status(clear=True) == 5  # SITU_ERR_TIMEOUT
    assert situ.device_status(clear=True) == 0
    g = wl.normal((4, 16), 1.0, seed=0).to(cuda_dev)
    out = situ.situ_glu_act(g)
    torch.cuda.synchronize()
    assert out.shape == (4, 8)
