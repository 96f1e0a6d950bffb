"""Seeded random shapes through the dense FFN, the grouped experts and the grouped MX
experts: many more combinations of row counts, ragged K and N, single-row and empty
experts, and one-CTA versus two-CTA schedules than the hand-picked cases.

  * dense: the one-launch forward against the FP64 oracle (2e-2 (1 + |ref|)), and the
    two-launch forward bitwise equal to it;
  * grouped bf16: against the FP64 oracle's per-(token, slot) loop;
  * grouped MX: each (token, slot) row bitwise equal to the dense MX FFN of its expert.
The shapes come from numpy's seeded generator; the inputs from the shared workload
generators."""
import numpy as np
import pytest
import torch

import situ_glu_activation_gb300 as situ
from situ_glu_activation_gb300 import workloads as wl
from numerics import assert_ffn_close, oracle_input, to_f64

pytestmark = pytest.mark.gpu


def _dense_shapes(n=10, seed=101):
    g = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        R = int(g.integers(1, 800))
        M = 8 * int(g.integers(8, 89))     # 64 .. 704
        I = 8 * int(g.integers(8, 89))
        out.append((R, M, I))
    return out


@pytest.mark.parametrize("R,M,I", _dense_shapes())
def test_dense_random_shape(oracle, cuda_dev, R, M, I):
    x, wgu, wd = wl.ffn_inputs(M, I, R, seed=R + 7 * M + 13 * I, device=cuda_dev)
    y = situ.situ_ffn_forward(x, wgu, wd)
    torch.cuda.synchronize()
    assert situ.ffn_last_path() == situ.FFN_PATH_FUSED
    ref = oracle.ffn_forward(oracle_input(x), oracle_input(wgu), oracle_input(wd))
    assert_ffn_close(to_f64(y), ref, f"dense {R}x{M}x{I}")
    assert situ.ffn_set_single_launch(False) is True
    try:
        y2 = situ.situ_ffn_forward(x, wgu, wd)
    finally:
        situ.ffn_set_single_launch(True)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def _routes(T, k, E, seed):
    gen = torch.Generator().manual_seed(seed)
    return torch.stack([torch.randperm(E, generator=gen)[:k] for _ in range(T)]).to(torch.int32)


def _grouped_shapes(n=8, seed=202, quantum=8, lo=8, hi=49):
    """(T, k, E, M, I); the first three route every token to each of 2 or 3 experts, so
    the experts hold 600 or more rows (two-CTA MMAs); the rest draw more, smaller experts."""
    g = np.random.default_rng(seed)
    out = []
    for i in range(n):
        if i < 3:
            E = int(g.integers(2, 4))
            T = int(g.integers(600, 1100))
            k = E
        else:
            E = int(g.integers(2, 13))
            T = int(g.integers(1, 400))
            k = int(g.integers(1, min(4, E) + 1))
        M = quantum * int(g.integers(lo, hi))
        I = quantum * int(g.integers(lo, hi))
        out.append((T, k, E, M, I))
    return out


@pytest.mark.parametrize("T,k,E,M,I", _grouped_shapes())
def test_grouped_random_shape(oracle, cuda_dev, T, k, E, M, I):
    ids = _routes(T, k, E, seed=T + E)
    x = wl.normal((T, M), 1.0, seed=T + M)
    wgu, wd = wl.expert_weights(E, M, I, seed=E + I)
    off, tix = situ.situ_moe_build_index(ids.to(cuda_dev), E)
    y = situ.situ_moe_grouped_forward(x.to(cuda_dev), off, tix, wgu.to(cuda_dev),
                                      wd.to(cuda_dev), k)
    torch.cuda.synchronize()
    ref = oracle.moe_grouped_forward(oracle_input(x), ids.numpy(), oracle_input(wgu),
                                     oracle_input(wd))
    assert_ffn_close(to_f64(y), ref, f"grouped T={T} k={k} E={E} M={M} I={I}")


@pytest.mark.parametrize("fmt", [situ.MX_E4M3, situ.MX_E2M1], ids=["mxfp8", "mxfp4"])
@pytest.mark.parametrize("T,k,E,M,I", _grouped_shapes(n=6, seed=303, quantum=128, lo=1, hi=5))
def test_grouped_mx_random_shape(cuda_dev, T, k, E, M, I, fmt):
    ids = _routes(T, k, E, seed=T + 3 * E)
    x = wl.normal((T, M), 1.0, seed=T + M + 1).to(cuda_dev)
    wgu, wd = wl.expert_weights(E, M, I, seed=E + I + 1, device=cuda_dev)
    wguq = situ.mx_quantize_weights(wgu, situ.MX_GATE_UP, fmt)
    wdq = situ.mx_quantize_weights(wd, situ.MX_DOWN, fmt)
    off, tix = situ.situ_moe_build_index(ids.to(cuda_dev), E)
    y = situ.situ_moe_grouped_forward_mxfp8(x, off, tix, wguq, wdq, k)
    torch.cuda.synchronize()
    y = y.cpu()
    for e in range(E):
        t_idx, s_idx = (ids == e).nonzero(as_tuple=True)
        if len(t_idx) == 0:
            continue
        we = situ.MxWeights(wguq[0][e].contiguous(), wguq[1].view(E, -1)[e].contiguous(), fmt)
        wde = situ.MxWeights(wdq[0][e].contiguous(), wdq[1].view(E, -1)[e].contiguous(), fmt)
        ye = situ.situ_ffn_forward_mxfp8(x, we, wde).cpu()
        assert torch.equal(y[t_idx, s_idx].view(torch.int16), ye[t_idx].view(torch.int16)), e


# ---------------------------------------------------------------------------
# Training paths and the dense MX FFN at random shapes, with the checks (and the
# tolerances derived there) of their own test modules.
# ---------------------------------------------------------------------------
from test_gpu_backward import _check_backward, _inputs as _bwd_inputs  # noqa: E402
from test_gpu_moe_backward import _check as _grouped_bwd_check  # noqa: E402
from test_gpu_moe_backward import _routes as _bwd_routes  # noqa: E402
from test_gpu_moe_backward import _train_step  # noqa: E402
from test_gpu_mx import test_ffn_forward_mxfp8 as _mx_ffn_check  # noqa: E402


@pytest.mark.parametrize("R,M,I", _dense_shapes(n=6, seed=404))
def test_dense_backward_random_shape(oracle, cuda_dev, R, M, I):
    R = max(1, R // 2)  # the oracle's FP64 backward is the slow side
    x, wgu, wd, dy, (xd, wgud, wdd, dyd) = _bwd_inputs(R, M, I, R + 3 * M, cuda_dev)
    _, gu, h = situ.situ_ffn_forward_train(xd, wgud, wdd)
    dx, dwg, dwd = situ.situ_ffn_backward(xd, wgud, wdd, gu, h, dyd)
    torch.cuda.synchronize()
    _check_backward(oracle, x, wgu, wd, dy, dx, dwg, dwd, what=f"{R}x{M}x{I}")


def _grouped_bwd_shapes(n=5, seed=505):
    """(T, k, E, M, I); the last expert has no routes.  The first two route 1600 or more
    rows to 2 experts (two-CTA dh and dx GEMMs)."""
    g = np.random.default_rng(seed)
    out = []
    for i in range(n):
        if i < 2:
            E, k, T = 3, 2, int(g.integers(800, 1000))
        else:
            E = int(g.integers(3, 10))
            k = int(g.integers(1, min(3, E - 1) + 1))
            T = int(g.integers(1, 200))
        out.append((T, k, E, 8 * int(g.integers(8, 41)), 8 * int(g.integers(8, 41))))
    return out


@pytest.mark.parametrize("T,k,E,M,I", _grouped_bwd_shapes())
def test_grouped_backward_random_shape(oracle, cuda_dev, T, k, E, M, I):
    ids = _bwd_routes(T, k, E, seed=T + k + E)
    x = wl.normal((T, M), 1.0, seed=T + 1)
    wgu, wd = wl.expert_weights(E, M, I, seed=E + 2)
    dy = wl.normal((T, k, M), 1.0, seed=T + 3)
    _, got = _train_step(x, ids, wgu, wd, dy, cuda_dev)
    _grouped_bwd_check(oracle, x, ids, wgu, wd, dy, got, what=f"T={T} k={k} E={E} M={M} I={I}")


def _mx_dense_shapes(n=4, seed=606):
    g = np.random.default_rng(seed)
    return [(int(g.integers(1, 700)), 128 * int(g.integers(1, 7)), 128 * int(g.integers(1, 7)))
            for _ in range(n)]


@pytest.mark.parametrize("fmt", [situ.MX_E4M3, situ.MX_E2M1], ids=["mxfp8", "mxfp4"])
@pytest.mark.parametrize("R,M,I", _mx_dense_shapes())
def test_dense_mx_random_shape(oracle, cuda_dev, R, M, I, fmt):
    _mx_ffn_check(oracle, cuda_dev, R, M, I, fmt)
