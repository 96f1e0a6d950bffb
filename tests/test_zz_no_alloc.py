"""situ_ffn_forward_noalloc: the dense FFN for callers that cannot allocate.

Some callers of this library have no way to allocate device memory when they run
the FFN: an engine plugin executing inside a pre-planned memory budget, or a
serving loop that must never call cudaMalloc.  The no-allocation entry point keeps
the intermediate h in a fixed scratch array inside the library.  Here it is
called through the C ABI (ctypes, the exported symbol) twice in a row -- the
second call smaller, so the scratch still holds the first call's h -- and each
result is checked against the regular entry point's output (which uses a
caller-provided workspace) and, on sampled rows, against the FP64 oracle, both at
the FFN tolerance, 2e-2 * (1 + |ref|).  The call that fills the scratch to within
one row of its end is checked the same way.

This file is collected last on purpose; it passes alone in a fresh process and
after the rest of the suite.
"""
import pytest
import torch

import situ_glu_activation_gb300 as situ
from situ_glu_activation_gb300 import workloads as wl
from numerics import assert_ffn_close, oracle_input, to_f64

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


def _check_rows(oracle, x, wgu, wd, y, rows, what):
    """Sampled rows of y against the FP64 oracle's FFN of the same inputs."""
    ref = oracle.ffn_forward(oracle_input(x[rows]), oracle_input(wgu), oracle_input(wd))
    assert_ffn_close(to_f64(y[rows]), ref, what)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_noalloc_matches_ffn_forward_twice(situ_lib, cuda_dev, oracle, dtype):
    M, I = 512, 1024
    for R, seed in [(1500, 0), (300, 1)]:  # second call smaller: stale scratch must not matter
        x, wgu, wd = wl.ffn_inputs(M, I, R, seed=seed, device=cuda_dev, dtype=dtype)
        ref = situ.situ_ffn_forward(x, wgu, wd)
        y = torch.full_like(x, float("nan"))
        assert _noalloc(situ_lib, x, wgu, wd, y) == SITU_OK
        torch.cuda.synchronize()
        assert_ffn_close(to_f64(y), to_f64(ref), f"noalloc R={R} {dtype}")
        rows = torch.cat([torch.arange(0, R, 97), torch.tensor([R - 1])])
        _check_rows(oracle, x, wgu, wd, y, rows, f"noalloc R={R} {dtype} vs oracle")
    assert situ.device_status(clear=True) == 0


def test_noalloc_rejects_sizes_beyond_scratch(situ_lib, cuda_dev, oracle):
    M, I = 256, 3072
    R = SCRATCH_BYTES // (2 * I) + 1  # one row more than the scratch holds
    x_big, wgu, wd = wl.ffn_inputs(M, I, R, seed=2, device=cuda_dev)
    y = torch.zeros_like(x_big)
    assert _noalloc(situ_lib, x_big, wgu, wd, y) == SITU_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((y == 0).all())  # nothing was launched
    # R - 1 rows fill the scratch to within one row of its end (a partial last
    # 128-row tile): the result must still be exact where a write past the end of the
    # scratch would show.
    x_ok = x_big[: R - 1]
    y_ok = torch.full_like(x_ok, float("nan"))
    assert _noalloc(situ_lib, x_ok, wgu, wd, y_ok) == SITU_OK
    torch.cuda.synchronize()
    ref = situ.situ_ffn_forward(x_ok, wgu, wd)
    torch.cuda.synchronize()
    assert_ffn_close(to_f64(y_ok), to_f64(ref), "noalloc at the scratch limit")
    rows = torch.tensor([0, 1, 128, R // 2, R - 130, R - 2])
    _check_rows(oracle, x_ok, wgu, wd, y_ok, rows, "noalloc at the scratch limit vs oracle")
    assert situ.device_status(clear=True) == 0
