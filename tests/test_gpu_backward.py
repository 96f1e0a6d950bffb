"""Training pair of the dense FFN on the GPU (forward that keeps the
pre-activation, and the backward) against the FP64 oracle.

Tolerance, derived from the arithmetic (no tolerance is stated for the
backward).  Like an autograd pass in bf16, the GPU keeps gu, h and dgu in bf16:
each stored factor carries a relative rounding of 2^-9, and dgu is evaluated at
the rounded gu.  A gradient entry is a sum of products (over the rows for the
weight gradients, over 2I for dx) that can cancel to far below its terms, so the
bound is the FFN tolerance plus 2^-8 times the sum of the absolute terms:
    |err| <= 2e-2 (1 + |ref|) + 2^-8 sum_i |term_i|
(measured worst case: about 2^-11 of the absolute sum)."""
import numpy as np
import pytest
import torch

import situ_glu_activation_gb300 as situ
from situ_glu_activation_gb300 import workloads as wl
from numerics import assert_ffn_close, oracle_input, to_f64

pytestmark = pytest.mark.gpu
INF = float("inf")


def _close(got, ref, abs_terms, what):
    err = np.abs(to_f64(got) - ref)
    tol = 2e-2 * (1.0 + np.abs(ref)) + 2.0 ** -8 * abs_terms
    assert np.isfinite(to_f64(got)).all(), what
    assert (err <= tol).all(), f"{what}: worst err/tol {float((err / tol).max()):.3g}"


def _check_backward(oracle, x, wgu, wd, dy, dx, dwg, dwd, caps=(4.0, 25.0), what=""):
    rdx, rdwg, rdwd, rdgu = oracle.ffn_backward(oracle_input(x), oracle_input(wgu),
                                               oracle_input(wd), oracle_input(dy), *caps,
                                               want_dgu=True)
    _, rh = oracle.ffn_forward(oracle_input(x), oracle_input(wgu), oracle_input(wd), *caps,
                               want_h=True)
    ax, awg, awd, ady = (np.abs(to_f64(t)) for t in (x, wgu, wd, dy))
    _close(dx, rdx, np.abs(rdgu) @ awg, f"dx {what}")
    _close(dwg, rdwg, np.abs(rdgu).T @ ax, f"dW_gate_up {what}")
    _close(dwd, rdwd, ady.T @ np.abs(rh), f"dW_down {what}")


def _inputs(R, M, I, seed, dev):
    x, wgu, wd = wl.ffn_inputs(M, I, R, seed=seed)
    dy = wl.normal((R, M), 1.0, seed=seed + 7)
    return x, wgu, wd, dy, [t.to(dev) for t in (x, wgu, wd, dy)]


def test_forward_train_matches_forward(oracle, cuda_dev):
    R, M, I = 300, 512, 384
    x, wgu, wd, _, (xd, wgud, wdd, _) = _inputs(R, M, I, 1, cuda_dev)
    y, gu, h = situ.situ_ffn_forward_train(xd, wgud, wdd)
    ws = torch.empty(situ.ffn_workspace_bytes(R, M, I), dtype=torch.uint8, device=cuda_dev)
    y2 = situ.situ_ffn_forward(xd, wgud, wdd, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    h2 = ws[: R * I * 2].view(torch.bfloat16).view(R, I)
    assert torch.equal(h.view(torch.int16), h2.view(torch.int16))
    gu_ref = to_f64(x) @ to_f64(wgu).T  # library matmul of the exact bf16 values
    assert_ffn_close(to_f64(gu), gu_ref, "saved pre-activation", tol=2 ** -8)


@pytest.mark.parametrize("R,M,I", [(300, 512, 384), (77, 136, 200), (1, 128, 256),
                                   (260, 1024, 520), (129, 256, 128)])
def test_backward_small(oracle, cuda_dev, R, M, I):
    x, wgu, wd, dy, (xd, wgud, wdd, dyd) = _inputs(R, M, I, R + M, cuda_dev)
    _, gu, h = situ.situ_ffn_forward_train(xd, wgud, wdd)
    dx, dwg, dwd = situ.situ_ffn_backward(xd, wgud, wdd, gu, h, dyd)
    torch.cuda.synchronize()
    _check_backward(oracle, x, wgu, wd, dy, dx, dwg, dwd, what=f"{R}x{M}x{I}")


@pytest.mark.parametrize("caps", [(INF, INF), (4.0, INF)], ids=["swiglu", "up_uncapped"])
def test_backward_variants(oracle, cuda_dev, caps):
    R, M, I = 200, 256, 256
    x, wgu, wd, dy, (xd, wgud, wdd, dyd) = _inputs(R, M, I, 5, cuda_dev)
    _, gu, h = situ.situ_ffn_forward_train(xd, wgud, wdd, *caps)
    dx, dwg, dwd = situ.situ_ffn_backward(xd, wgud, wdd, gu, h, dyd, *caps)
    torch.cuda.synchronize()
    oc = tuple(0.0 if c == INF else c for c in caps)
    _check_backward(oracle, x, wgu, wd, dy, dx, dwg, dwd, caps=oc, what=str(caps))


@pytest.mark.parametrize("R,M,I,caps", [(300, 512, 384, (4.0, 25.0)),
                                         (77, 136, 200, (4.0, 25.0)),
                                         (130, 256, 256, (INF, INF)),
                                         (130, 256, 256, (4.0, INF)),
                                         (130, 256, 256, (INF, 25.0))],
                         ids=["situ", "situ_ragged", "swiglu", "up_uncapped", "gate_uncapped"])
def test_dgu_elementwise(oracle, cuda_dev, R, M, I, caps):
    """The dh GEMM's activation-derivative epilogue, element by element: d(g, u) (left in
    the workspace) against dh = dy W_down (library matmul of the exact bf16 values) times
    the oracle's partial derivatives at the saved bf16 (g, u).

    Bound: the bf16 rounding of the result and the relative error of the FP32 partials
    (2^-8 |ref| covers both); for dg, the error of a'(g)'s two terms, each with a relative
    error of about 2^-11 from the hardware tanh, taken against their absolute sizes
    sigmoid(g) + |a(g)| sigmoid(-g) (2^-9 |dh| |b(u)| times that, where a'(g) cancels);
    and the FP32 accumulation of dh (2^-12 of its sum of absolute terms)."""
    x, wgu, wd, dy, (xd, wgud, wdd, dyd) = _inputs(R, M, I, 3 * R + I, cuda_dev)
    _, gu, h = situ.situ_ffn_forward_train(xd, wgud, wdd, *caps)
    ws = torch.empty(situ.ffn_backward_workspace_bytes(R, M, I), dtype=torch.uint8,
                     device=cuda_dev)
    situ.situ_ffn_backward(xd, wgud, wdd, gu, h, dyd, *caps, workspace=ws)
    torch.cuda.synchronize()
    assert situ.device_status(clear=True) == 0
    dgu = to_f64(ws[: R * 2 * I * 2].view(torch.bfloat16).view(R, 2 * I).cpu())
    assert np.isfinite(dgu).all()
    b1, b2 = (0.0 if c == INF else c for c in caps)
    guf = to_f64(gu.cpu())
    dh = to_f64(dy) @ to_f64(wd)
    dh_abs = np.abs(to_f64(dy)) @ np.abs(to_f64(wd))
    pg = np.empty((R, I))
    pu = np.empty((R, I))
    gate_terms = np.empty((R, I))
    up_abs = np.empty((R, I))
    for r in range(R):
        for j in range(I):
            g, u = guf[r, j], guf[r, I + j]
            pg[r, j], pu[r, j] = oracle.pair_grad(g, u, b1, b2)
            gate_terms[r, j] = oracle.sigmoid(g) + abs(oracle.gate(g, b1)) * oracle.sigmoid(-g)
            up_abs[r, j] = abs(oracle.up(u, b2))
    for got, part, extra, what in ((dgu[:, :I], pg, 2.0 ** -9 * np.abs(dh) * up_abs * gate_terms,
                                    "dg"),
                                   (dgu[:, I:], pu, 0.0, "du")):
        ref = dh * part
        tol = 2.0 ** -8 * np.abs(ref) + extra + 2.0 ** -12 * dh_abs * np.abs(part)
        err = np.abs(got - ref)
        assert (err <= tol).all(), f"{what} {R}x{M}x{I} {caps}: worst err/tol " \
                                   f"{float((err / np.maximum(tol, 1e-300)).max()):.3g}"


def test_dgu_special_values(oracle, cuda_dev):
    """The derivative epilogue on a saved pre-activation pair built to hit the method's
    edges: zeros and tiny values, the caps' saturation (|g| or |u| up to 1e4), the gate's
    negative tail down to -100 (where sigmoid(g) and a(g) leave the FP32 normal range),
    large positive gates, mixed with N(0, 1).  d(g, u) against dh times the oracle's
    partial derivatives, with the bound of test_dgu_elementwise plus an absolute
    2^-120 * |dh| * (1 + |a(g)| + |b(u)|): the kernel's FP32 special-function ops flush
    results below 2^-126 to zero, where the exact partials are smaller still."""
    R, M, I = 160, 256, 256
    g = torch.Generator().manual_seed(77)
    special = torch.tensor([0.0, -0.0, 1e-20, -1e-20, 1e-3, -1e-3, 2.0, -2.0, 20.0, -20.0, 44.0,
                            -44.0, 87.0, -87.0, -88.0, -90.0, -100.0, 100.0, 1e3, -1e3, 1e4,
                            -1e4, 30.0, -30.0])
    pick = torch.randint(0, special.numel(), (R, 2 * I), generator=g)
    gu = torch.where(torch.rand(R, 2 * I, generator=g) < 0.5, special[pick],
                     torch.randn(R, 2 * I, generator=g)).to(torch.bfloat16)
    x, wgu, wd = wl.ffn_inputs(M, I, R, seed=78)
    dy = wl.normal((R, M), 1.0, seed=79)
    h = wl.normal((R, I), 1.0, seed=80)  # only dW_down reads h; d(g, u) is checked
    dev = cuda_dev
    ws = torch.empty(situ.ffn_backward_workspace_bytes(R, M, I), dtype=torch.uint8, device=dev)
    situ.situ_ffn_backward(x.to(dev), wgu.to(dev), wd.to(dev), gu.to(dev), h.to(dev), dy.to(dev),
                           workspace=ws)
    torch.cuda.synchronize()
    assert situ.device_status(clear=True) == 0
    dgu = to_f64(ws[: R * 2 * I * 2].view(torch.bfloat16).view(R, 2 * I).cpu())
    assert np.isfinite(dgu).all()
    guf = to_f64(gu)
    dh = to_f64(dy) @ to_f64(wd)
    dh_abs = np.abs(to_f64(dy)) @ np.abs(to_f64(wd))
    pg = np.empty((R, I))
    pu = np.empty((R, I))
    gate_terms = np.empty((R, I))
    a_abs = np.empty((R, I))
    b_abs = np.empty((R, I))
    for r in range(R):
        for j in range(I):
            gv, uv = guf[r, j], guf[r, I + j]
            pg[r, j], pu[r, j] = oracle.pair_grad(gv, uv, 4.0, 25.0)
            a_abs[r, j] = abs(oracle.gate(gv, 4.0))
            b_abs[r, j] = abs(oracle.up(uv, 25.0))
            gate_terms[r, j] = oracle.sigmoid(gv) + a_abs[r, j] * oracle.sigmoid(-gv)
    flush = 2.0 ** -120 * np.abs(dh) * (1.0 + a_abs + b_abs)
    for got, part, extra, what in ((dgu[:, :I], pg, 2.0 ** -9 * np.abs(dh) * b_abs * gate_terms,
                                    "dg"),
                                   (dgu[:, I:], pu, 0.0, "du")):
        ref = dh * part
        tol = 2.0 ** -8 * np.abs(ref) + extra + 2.0 ** -12 * dh_abs * np.abs(part) + flush
        err = np.abs(got - ref)
        bad = err > tol
        assert not bad.any(), f"{what}: {int(bad.sum())} outside the bound, e.g. gu = " \
                              f"{guf[np.nonzero(bad)[0][0]]}"


def test_backward_full_size_sparse_dy(oracle, cuda_dev):
    """The 16384-token workload (M=2048, I=3072) at full size, with dy nonzero on 16
    seeded rows only: every other row contributes exactly zero, so the oracle's
    backward over those 16 rows gives the full dW_gate_up and dW_down, and dx must
    be zero elsewhere."""
    w = wl.WORKLOADS["dense"]
    x, wgu, wd = wl.ffn_inputs(w.M, w.I, w.rows, seed=0, device=cuda_dev)
    g = torch.Generator().manual_seed(17)
    rows = torch.cat([torch.tensor([0, w.rows - 1]), torch.randperm(w.rows - 2, generator=g)[:14] + 1])
    dy = torch.zeros(w.rows, w.M, dtype=torch.bfloat16, device=cuda_dev)
    dy[rows.to(cuda_dev)] = wl.normal((16, w.M), 1.0, seed=9).to(cuda_dev)
    _, gu, h = situ.situ_ffn_forward_train(x, wgu, wd)
    dx, dwg, dwd = situ.situ_ffn_backward(x, wgu, wd, gu, h, dy)
    torch.cuda.synchronize()
    rd = rows.to(cuda_dev)
    mask = torch.ones(w.rows, dtype=torch.bool, device=cuda_dev)
    mask[rd] = False
    assert int((dx[mask] != 0).sum()) == 0
    _check_backward(oracle, x[rd].cpu(), wgu.cpu(), wd.cpu(), dy[rd].cpu(), dx[rd], dwg, dwd,
                    what="full size, 16 rows of dy")
