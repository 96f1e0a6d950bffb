"""Training step of the grouped experts on the GPU (forward that keeps the
pre-activation in expert order, and the backward) against the FP64 oracle.

Tolerance, derived from the arithmetic as for the dense backward: gu, h, d(g, u)
and the per-route dx rows are stored in bf16 (relative rounding 2^-9 each), and a
gradient entry is a sum of products that can cancel, so
    |err| <= 2e-2 (1 + |ref|) + 2^-8 sum_i |term_i|
where the terms are those of the entry's sum: over 2I and the token's slots for
dx, over the expert's routes for the weight gradients."""
import numpy as np
import pytest
import torch

import situ_glu_activation_gb300 as situ
from situ_glu_activation_gb300 import workloads as wl
from numerics import oracle_input, to_f64

pytestmark = pytest.mark.gpu
INF = float("inf")


def _close(got, ref, abs_terms, what):
    g = to_f64(got) if isinstance(got, torch.Tensor) else got
    err = np.abs(g - ref)
    tol = 2e-2 * (1.0 + np.abs(ref)) + 2.0 ** -8 * abs_terms
    assert np.isfinite(g).all(), what
    assert (err <= tol).all(), f"{what}: worst err/tol {float((err / tol).max()):.3g}"


def _routes(T, k, E, seed, unused_last=True):
    g = torch.Generator().manual_seed(seed)
    n = E - 1 if unused_last else E
    return torch.stack([torch.randperm(n, generator=g)[:k] for _ in range(T)]).to(torch.int32)


def _abs_terms(oracle, x, ids, wgu, wd, dy, caps):
    """Sums of absolute terms of every gradient entry, from the oracle's dense
    backward of each expert's routes (d(g, u) and h in FP64)."""
    T, k = ids.shape
    E = wgu.shape[0]
    M = x.shape[1]
    I = wgu.shape[1] // 2
    xa, wga, wda, dya = (np.abs(oracle_input(t)) for t in (x, wgu, wd, dy))
    dx_abs = np.zeros((T, M))
    dwg_abs = np.zeros((E, 2 * I, M))
    dwd_abs = np.zeros((E, M, I))
    ids_np = ids.numpy()
    for e in range(E):
        t_idx, s_idx = np.nonzero(ids_np == e)
        if len(t_idx) == 0:
            continue
        _, _, _, dgu = oracle.ffn_backward(oracle_input(x[t_idx]), oracle_input(wgu[e]),
                                           oracle_input(wd[e]), oracle_input(dy[t_idx, s_idx]),
                                           *caps, want_dgu=True)
        _, h = oracle.ffn_forward(oracle_input(x[t_idx]), oracle_input(wgu[e]),
                                  oracle_input(wd[e]), *caps, want_h=True)
        np.add.at(dx_abs, t_idx, np.abs(dgu) @ wga[e])
        dwg_abs[e] = np.abs(dgu).T @ xa[t_idx]
        dwd_abs[e] = dya[t_idx, s_idx].T @ np.abs(h)
    return dx_abs, dwg_abs, dwd_abs


def _train_step(x, ids, wgu, wd, dy, dev, caps=(4.0, 25.0)):
    E = wgu.shape[0]
    k = ids.shape[1]
    off, tix = situ.situ_moe_build_index(ids.to(dev).contiguous(), E)
    xd, wgud, wdd = x.to(dev), wgu.to(dev), wd.to(dev)
    y, gu, h = situ.situ_moe_grouped_forward_train(xd, off, tix, wgud, wdd, k, *caps)
    dx, dwg, dwd = situ.situ_moe_grouped_backward(xd, off, tix, wgud, wdd, gu, h, dy.to(dev),
                                                  *caps)
    torch.cuda.synchronize()
    assert situ.device_status(clear=True) == 0
    return (off, tix, y, gu, h), (dx, dwg, dwd)


def _check(oracle, x, ids, wgu, wd, dy, got, caps=(4.0, 25.0), what=""):
    dx, dwg, dwd = got
    rdx, rdwg, rdwd = oracle.moe_grouped_backward(oracle_input(x), ids.numpy(),
                                                  oracle_input(wgu), oracle_input(wd),
                                                  oracle_input(dy), *caps)
    adx, adwg, adwd = _abs_terms(oracle, x, ids, wgu, wd, dy, caps)
    _close(dx, rdx, adx, f"dx {what}")
    _close(dwg, rdwg, adwg, f"dW_gate_up {what}")
    _close(dwd, rdwd, adwd, f"dW_down {what}")


@pytest.mark.parametrize("T,k,E,M,I", [
    (50, 3, 6, 256, 384),    # experts with a single row, one unused expert
    (300, 2, 3, 128, 256),   # groups over several k-blocks with ragged last blocks
    (40, 4, 9, 136, 200),    # ragged M and I
    (130, 1, 2, 256, 128),   # one slot per token
])
def test_grouped_backward_small(oracle, cuda_dev, T, k, E, M, I):
    ids = _routes(T, k, E, seed=T * k + E)
    x = wl.normal((T, M), 1.0, seed=T)
    wgu, wd = wl.expert_weights(E, M, I, seed=E)
    dy = wl.normal((T, k, M), 1.0, seed=T + 11)
    _, got = _train_step(x, ids, wgu, wd, dy, cuda_dev)
    assert not got[1][E - 1].any() and not got[2][E - 1].any()  # unused expert: zero
    _check(oracle, x, ids, wgu, wd, dy, got, what=f"{T}x{k} E={E} M={M} I={I}")


@pytest.mark.parametrize("caps", [(INF, INF), (INF, 25.0)], ids=["swiglu", "gate_uncapped"])
def test_grouped_backward_variants(oracle, cuda_dev, caps):
    T, k, E, M, I = 64, 2, 4, 256, 256
    ids = _routes(T, k, E, seed=8, unused_last=False)
    x = wl.normal((T, M), 1.0, seed=9)
    wgu, wd = wl.expert_weights(E, M, I, seed=10)
    dy = wl.normal((T, k, M), 1.0, seed=12)
    _, got = _train_step(x, ids, wgu, wd, dy, cuda_dev, caps)
    oc = tuple(0.0 if c == INF else c for c in caps)
    _check(oracle, x, ids, wgu, wd, dy, got, caps=oc, what=str(caps))


def test_forward_train_matches_forward(oracle, cuda_dev):
    """y is bit-identical to the inference forward; gu in expert order is the
    pre-activation of each route's token and expert; h is the activation."""
    T, k, E, M, I = 70, 2, 5, 256, 384
    ids = _routes(T, k, E, seed=21)
    x = wl.normal((T, M), 1.0, seed=22)
    wgu, wd = wl.expert_weights(E, M, I, seed=23)
    dy = wl.normal((T, k, M), 1.0, seed=24)
    (off, tix, y, gu, h), _ = _train_step(x, ids, wgu, wd, dy, cuda_dev)
    y2 = situ.situ_moe_grouped_forward(x.to(cuda_dev), off, tix, wgu.to(cuda_dev),
                                       wd.to(cuda_dev), k)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    off_c, tix_c = off.cpu().numpy(), tix.cpu().numpy()
    xf, wgf = to_f64(x), to_f64(wgu)
    gu_c, h_c = to_f64(gu), to_f64(h)
    for e in range(E):
        rows = np.arange(off_c[e], off_c[e + 1])
        if len(rows) == 0:
            continue
        t = tix_c[rows] // k
        ref = xf[t] @ wgf[e].T  # library matmul of the exact bf16 values
        assert (np.abs(gu_c[rows] - ref) <= 2.0 ** -8 * (1 + np.abs(ref))).all()
        _, rh = oracle.ffn_forward(oracle_input(x[t]), oracle_input(wgu[e]), oracle_input(wd[e]),
                                   want_h=True)
        _close(h_c[rows], rh, 0.0, f"h of expert {e}")


@pytest.mark.parametrize("T", [333, 1200])
def test_grouped_backward_equals_dense_single_expert(cuda_dev, T):
    """One expert, one slot: the grouped backward runs the same tiles in the same
    order as the dense backward, so every output is bit-identical (333 rows: two-CTA
    grouped dh and dx GEMMs whose third m-tile is an M = 128 pair, against the dense
    kernels' M = 256 pair with a phantom half; 1200: whole pairs)."""
    M, I = 256, 384
    ids = torch.zeros(T, 1, dtype=torch.int32)
    x = wl.normal((T, M), 1.0, seed=31)
    wgu, wd = wl.expert_weights(1, M, I, seed=32)
    dy = wl.normal((T, 1, M), 1.0, seed=33)
    _, (dx, dwg, dwd) = _train_step(x, ids, wgu, wd, dy, cuda_dev)
    xd, wgd, wdd = x.to(cuda_dev), wgu[0].to(cuda_dev), wd[0].to(cuda_dev)
    _, gu, h = situ.situ_ffn_forward_train(xd, wgd, wdd)
    ddx, ddwg, ddwd = situ.situ_ffn_backward(xd, wgd, wdd, gu, h, dy[:, 0].to(cuda_dev))
    torch.cuda.synchronize()
    for a, b in ((dx, ddx), (dwg[0], ddwg), (dwd[0], ddwd)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("M,I", [(256, 384), (136, 200)])
def test_grouped_backward_two_cta_tails(oracle, cuda_dev, M, I):
    """Experts averaging >= 128 routes run the two-CTA dh and dx GEMMs: whole pairs, an
    expert's odd last m-tile as an M = 128 pair (333 routes: its second CTA holds 13
    rows; 129: one row; 64: no rows), an empty expert, and (I = 200) a ragged last
    32-column chunk of the saved (g, u).  Every gradient against the oracle."""
    sizes = [333, 129, 0, 200, 64]
    E = len(sizes)
    ids = torch.cat([torch.full((n,), e, dtype=torch.int32) for e, n in enumerate(sizes)])
    ids = ids[torch.randperm(ids.numel(), generator=torch.Generator().manual_seed(41))][:, None]
    T = ids.shape[0]
    assert T >= 128 * E
    x = wl.normal((T, M), 1.0, seed=42)
    wgu, wd = wl.expert_weights(E, M, I, seed=43)
    dy = wl.normal((T, 1, M), 1.0, seed=44)
    _, got = _train_step(x, ids, wgu, wd, dy, cuda_dev)
    assert not got[1][2].any() and not got[2][2].any()  # the empty expert
    _check(oracle, x, ids, wgu, wd, dy, got, what=f"two-CTA tails M={M} I={I}")


def test_grouped_backward_weight_gradient_k_tails(oracle, cuda_dev):
    """The weight gradients contract each expert over its own routes in 64-route
    k-blocks on two-CTA MMAs: experts of 1, 63, 64, 65, 130 and 191 routes (a last
    k-block of 1..64 valid routes, followed by the next expert's rows or, for the last
    expert, the end of the buffer), an empty expert, and output row counts (M = 128
    for dW_down, 2I = 384 for dW_gate_up) with an odd number of 128-row m-tiles, whose
    last pair has a second half past the rows."""
    sizes = [1, 63, 64, 65, 0, 130, 191]
    E, M, I = len(sizes), 128, 192
    ids = torch.cat([torch.full((n,), e, dtype=torch.int32) for e, n in enumerate(sizes)])
    ids = ids[torch.randperm(ids.numel(), generator=torch.Generator().manual_seed(51))][:, None]
    T = ids.shape[0]
    x = wl.normal((T, M), 1.0, seed=52)
    wgu, wd = wl.expert_weights(E, M, I, seed=53)
    dy = wl.normal((T, 1, M), 1.0, seed=54)
    _, got = _train_step(x, ids, wgu, wd, dy, cuda_dev)
    assert not got[1][4].any() and not got[2][4].any()  # the empty expert
    _check(oracle, x, ids, wgu, wd, dy, got, what="weight-gradient K tails")


@pytest.mark.parametrize("sizes,M,I", [
    ([1, 63, 64, 65, 0, 130, 191], 128, 192),   # K tails of every kind, odd m-tile counts
    ([5, 14, 0, 40, 700, 333], 256, 384),       # experts ending before row 32, a long one
])
def test_grouped_backward_weight_gradient_forms_agree(cuda_dev, sizes, M, I):
    """The two forms of the per-expert weight gradients, two-CTA MMAs through per-expert
    tensor maps that end at each expert's last row and one CTA per tile with the rows
    past the end zeroed in shared memory, produce the same bits."""
    E = len(sizes)
    ids = torch.cat([torch.full((n,), e, dtype=torch.int32) for e, n in enumerate(sizes)])
    ids = ids[torch.randperm(ids.numel(), generator=torch.Generator().manual_seed(61))][:, None]
    T = ids.shape[0]
    x = wl.normal((T, M), 1.0, seed=62)
    wgu, wd = wl.expert_weights(E, M, I, seed=63)
    dy = wl.normal((T, 1, M), 1.0, seed=64)
    _, two = _train_step(x, ids, wgu, wd, dy, cuda_dev)
    prev = situ.moe_set_kgrouped_two_cta(False)
    try:
        _, one = _train_step(x, ids, wgu, wd, dy, cuda_dev)
    finally:
        situ.moe_set_kgrouped_two_cta(prev)
    for a, b, what in zip(two, one, ("dx", "dW_gate_up", "dW_down")):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), what


def test_grouped_backward_no_routes(cuda_dev):
    E, M, I = 3, 64, 64
    x = torch.empty(0, M, dtype=torch.bfloat16, device=cuda_dev)
    wgu, wd = wl.expert_weights(E, M, I, seed=0, device=cuda_dev)
    off = torch.zeros(E + 1, dtype=torch.int32, device=cuda_dev)
    tix = torch.empty(0, dtype=torch.int32, device=cuda_dev)
    gu = torch.empty(0, 2 * I, dtype=torch.bfloat16, device=cuda_dev)
    h = torch.empty(0, I, dtype=torch.bfloat16, device=cuda_dev)
    dy = torch.empty(0, 2, M, dtype=torch.bfloat16, device=cuda_dev)
    dx, dwg, dwd = situ.situ_moe_grouped_backward(x, off, tix, wgu, wd, gu, h, dy)
    torch.cuda.synchronize()
    assert dx.shape == (0, M) and not dwg.any() and not dwd.any()


def test_grouped_backward_bad_offsets(cuda_dev):
    """Offsets that fail validation: SITU_ERR_INDEX, and no weight gradient written."""
    T, k, E, M, I = 8, 2, 3, 64, 64
    x = wl.normal((T, M), 1.0, seed=0, device=cuda_dev)
    wgu, wd = wl.expert_weights(E, M, I, seed=0, device=cuda_dev)
    off = torch.tensor([0, 10, 5, 16], dtype=torch.int32, device=cuda_dev)  # not monotone
    tix = torch.arange(T * k, dtype=torch.int32, device=cuda_dev)
    gu = torch.zeros(T * k, 2 * I, dtype=torch.bfloat16, device=cuda_dev)
    h = torch.zeros(T * k, I, dtype=torch.bfloat16, device=cuda_dev)
    dy = wl.normal((T, k, M), 1.0, seed=1, device=cuda_dev)
    R = T * k
    ws = torch.empty(situ.moe_backward_workspace_bytes(R, E, M, I), dtype=torch.uint8,
                     device=cuda_dev)
    lib = situ._native.lib()
    dx = torch.empty(T, M, dtype=torch.bfloat16, device=cuda_dev)
    dwg = torch.full((E, 2 * I, M), 7.0, dtype=torch.bfloat16, device=cuda_dev)
    dwd = torch.full((E, M, I), 7.0, dtype=torch.bfloat16, device=cuda_dev)
    st = lib.situ_moe_grouped_backward(
        x.data_ptr(), off.data_ptr(), tix.data_ptr(), wgu.data_ptr(), wd.data_ptr(),
        gu.data_ptr(), h.data_ptr(), dy.data_ptr(), dx.data_ptr(), dwg.data_ptr(), dwd.data_ptr(),
        ws.data_ptr(), ws.numel(), T, k, E, M, I, 4.0, 25.0, 0,
        torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 0
    assert situ.device_status(clear=True) == 7
    assert bool((dwg == 7.0).all()) and bool((dwd == 7.0).all())


def test_grouped_backward_full_size_sparse_dy(oracle, cuda_dev):
    """The E=64, 16384-token top-8 Zipf workload (M=2048, I=3072) at full size, with
    dy nonzero on 12 seeded routes only (among them routes of the most and of the
    least loaded experts): every other route contributes exactly zero, so the
    oracle's backward of those 12 routes gives dx and every dW, and the gradients
    of experts without a chosen route are exactly zero."""
    w = wl.WORKLOADS["grouped"]
    E, M, I, k = w.num_experts, w.M, w.I, w.k_eff
    ids = wl.routes(w, seed=0)
    x = wl.normal((w.T, M), 1.0, seed=0, device=cuda_dev)
    wgu, wd = wl.expert_weights(E, M, I, seed=0, device=cuda_dev)
    flat = ids.view(-1)
    counts = torch.bincount(flat.long(), minlength=E)
    used = torch.nonzero(counts > 0).view(-1)
    busiest = int(used[counts[used].argmax()])
    quietest = int(used[counts[used].argmin()])
    g = torch.Generator().manual_seed(5)
    pick = [int(torch.nonzero(flat == busiest)[0]), int(torch.nonzero(flat == busiest)[-1]),
            int(torch.nonzero(flat == quietest)[0])]
    pick += torch.randint(0, flat.numel(), (9,), generator=g).tolist()
    pick = sorted(set(pick))
    dy = torch.zeros(w.T * k, M, dtype=torch.bfloat16)
    dy[pick] = wl.normal((len(pick), M), 1.0, seed=6)
    dy = dy.view(w.T, k, M)
    off, tix = situ.situ_moe_build_index(ids.to(cuda_dev), E)
    _, gu, h = situ.situ_moe_grouped_forward_train(x, off, tix, wgu, wd, k)
    dx, dwg, dwd = situ.situ_moe_grouped_backward(x, off, tix, wgu, wd, gu, h, dy.to(cuda_dev))
    torch.cuda.synchronize()
    assert situ.device_status(clear=True) == 0
    # Sub-problem of the chosen routes: one slot each.
    tok = [p // k for p in pick]
    sub_ids = flat[pick].view(-1, 1)
    sub_x = x[torch.tensor(tok, device=cuda_dev)].cpu()
    sub_dy = dy.view(-1, M)[pick].view(-1, 1, M)
    sub_e = sorted(set(sub_ids.view(-1).tolist()))
    wgu_c = wgu[torch.tensor(sub_e, device=cuda_dev)].cpu()
    wd_c = wd[torch.tensor(sub_e, device=cuda_dev)].cpu()
    remap = torch.tensor([sub_e.index(e) for e in sub_ids.view(-1).tolist()],
                         dtype=torch.int32).view(-1, 1)
    rdx, rdwg, rdwd = oracle.moe_grouped_backward(oracle_input(sub_x), remap.numpy(),
                                                  oracle_input(wgu_c), oracle_input(wd_c),
                                                  oracle_input(sub_dy))
    adx, adwg, adwd = _abs_terms(oracle, sub_x, remap, wgu_c, wd_c, sub_dy, (4.0, 25.0))
    # dx: rows of the chosen tokens (a token chosen twice sums its routes).
    uniq = sorted(set(tok))
    want = np.zeros((len(uniq), M))
    want_abs = np.zeros((len(uniq), M))
    for i, t in enumerate(tok):
        want[uniq.index(t)] += rdx[i]
        want_abs[uniq.index(t)] += adx[i]
    _close(dx[torch.tensor(uniq, device=cuda_dev)], want, want_abs, "dx of the chosen tokens")
    mask = torch.ones(w.T, dtype=torch.bool, device=cuda_dev)
    mask[torch.tensor(uniq, device=cuda_dev)] = False
    assert int((dx[mask] != 0).sum()) == 0
    for j, e in enumerate(sub_e):
        _close(dwg[e], rdwg[j], adwg[j], f"dW_gate_up[{e}] ({int(counts[e])} routes)")
        _close(dwd[e], rdwd[j], adwd[j], f"dW_down[{e}] ({int(counts[e])} routes)")
    others = torch.ones(E, dtype=torch.bool, device=cuda_dev)
    others[torch.tensor(sub_e, device=cuda_dev)] = False
    assert int((dwg[others] != 0).sum()) == 0 and int((dwd[others] != 0).sum()) == 0
