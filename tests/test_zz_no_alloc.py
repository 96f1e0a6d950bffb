"""situ_ffn_forward_noalloc: the dense FFN for callers that cannot allocate.

Some callers of this library have no way to allocate device memory when they run
the FFN: an engine plugin executing inside a pre-planned memory budget, or a
serving loop that must never call cudaMalloc.  The no-allocation entry point keeps
the intermediate h in a fixed scratch array inside the library.  Here it is
called through the C ABI (ctypes, the exported symbol) twice in a row -- the
second call smaller, so the scratch still holds the first call's h -- and each
result is checked against the regular entry point's output (which uses a
caller-provided workspace) at the FFN tolerance, 2e-2 * (1 + |ref|).

This file is collected last on purpose; it passes alone in a fresh process and
after the rest of the suite.
"""
import pytest
import torch

import situ_glu_activation_gb300 as situ
from situ_glu_activation_gb300 import workloads as wl
from numerics import assert_ffn_close, to_f64

pytestmark = pytest.mark.gpu

SITU_OK, SITU_ERR_WORKSPACE = 0, 8
SCRATCH_BYTES = 16 << 20


def _noalloc(lib, x, wgu, wd, y, beta=4.0, linear_beta=25.0):
    R, M = x.shape
    I = wgu.shape[0] // 2
    dt = 0 if x.dtype == torch.bfloat16 else 1
    return lib.situ_ffn_forward_noalloc(x.data_ptr(), wgu.data_ptr(), wd.data_ptr(), y.data_ptr(),
                                        R, M, I, beta, linear_beta, dt,
                                        torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_noalloc_matches_ffn_forward_twice(situ_lib, cuda_dev, dtype):
    M, I = 512, 1024
    for R, seed in [(1500, 0), (300, 1)]:  # second call smaller: stale scratch must not matter
        x, wgu, wd = wl.ffn_inputs(M, I, R, seed=seed, device=cuda_dev, dtype=dtype)
        ref = situ.situ_ffn_forward(x, wgu, wd)
        y = torch.full_like(x, float("nan"))
        assert _noalloc(situ_lib, x, wgu, wd, y) == SITU_OK
        torch.cuda.synchronize()
        assert_ffn_close(to_f64(y), to_f64(ref), f"noalloc R={R} {dtype}")


def test_noalloc_rejects_sizes_beyond_scratch(situ_lib, cuda_dev):
    M, I = 256, 3072
    R = SCRATCH_BYTES // (2 * I) + 1  # one row more than the scratch holds
    x, wgu, wd = wl.ffn_inputs(M, I, 8, seed=0, device=cuda_dev)
    x_big = torch.zeros(R, M, dtype=torch.bfloat16, device=cuda_dev)
    y = torch.zeros_like(x_big)
    assert _noalloc(situ_lib, x_big, wgu, wd, y) == SITU_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((y == 0).all())  # nothing was launched
    y_ok = torch.empty(R - 1, M, dtype=torch.bfloat16, device=cuda_dev)
    assert _noalloc(situ_lib, x_big[: R - 1], wgu, wd, y_ok) == SITU_OK
    torch.cuda.synchronize()
