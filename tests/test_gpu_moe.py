"""Expert index and grouped SiTU-GLU experts on the GPU against the FP64 oracle.

Indices: bit-exact.  Outputs: |y - ref| <= 2e-2 (1 + |ref|)."""
import numpy as np
import pytest
import torch

import situ_glu_activation_gb300 as situ
from situ_glu_activation_gb300 import workloads as wl
from numerics import assert_ffn_close, oracle_input, to_f64

pytestmark = pytest.mark.gpu


def _index(ids_cpu, E, dev):
    off, tix = situ.situ_moe_build_index(ids_cpu.to(dev).contiguous(), E)
    torch.cuda.synchronize()
    return off.cpu().numpy(), tix.cpu().numpy()


@pytest.mark.parametrize("name", ["grouped", "k3_decode", "k3_prefill"])
def test_index_bit_exact_full_size(oracle, cuda_dev, name):
    w = wl.WORKLOADS[name]
    ids = wl.routes(w, seed=0)
    off, tix = _index(ids, w.num_experts, cuda_dev)
    ref_off, ref_tix = oracle.moe_build_index(ids.numpy(), w.num_experts)
    assert np.array_equal(off, ref_off)
    assert np.array_equal(tix, ref_tix)
    if name == "grouped":
        assert (np.diff(off) == 0).sum() >= 4  # the forced-empty experts


@pytest.mark.parametrize("n,E", [(0, 5), (1, 1), (1000, 3), (1025, 17), (4097, 900), (3000, 16384)])
def test_index_edge_sizes(oracle, cuda_dev, n, E):
    g = torch.Generator().manual_seed(n + E)
    ids = torch.randint(0, E, (n,), generator=g, dtype=torch.int32)
    off, tix = _index(ids, E, cuda_dev)
    ref_off, ref_tix = oracle.moe_build_index(ids.numpy(), E)
    assert np.array_equal(off, ref_off) and np.array_equal(tix, ref_tix)


def test_index_bad_id_reported(cuda_dev):
    ids = torch.tensor([0, 1, 7, 1], dtype=torch.int32)
    off, tix = _index(ids, 3, cuda_dev)
    assert situ.device_status(clear=True) == 7  # SITU_ERR_INDEX
    assert off[-1] == 3  # the bad route was dropped


def _grouped(x, ids, wgu, wd, dev):
    E = wgu.shape[0]
    ids_d = ids.to(dev).contiguous()
    off, tix = situ.situ_moe_build_index(ids_d, E)
    y = situ.situ_moe_grouped_forward(x.to(dev), off, tix, wgu.to(dev), wd.to(dev), ids.shape[1])
    torch.cuda.synchronize()
    return y


@pytest.mark.parametrize("T,k,E,M,I", [
    (50, 3, 6, 256, 384),    # some experts with a single row
    (300, 2, 3, 128, 256),   # groups spanning several 128-row tiles with tails
    (40, 4, 9, 136, 200),    # ragged K and N
])
def test_grouped_small(oracle, cuda_dev, T, k, E, M, I):
    g = torch.Generator().manual_seed(T * k + E)
    ids = torch.stack([torch.randperm(E - 1, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    x = wl.normal((T, M), 1.0, seed=T)
    wgu, wd = wl.expert_weights(E, M, I, seed=E)
    y = _grouped(x, ids, wgu, wd, cuda_dev)
    ref = oracle.moe_grouped_forward(oracle_input(x), ids.numpy(), oracle_input(wgu),
                                     oracle_input(wd))
    assert_ffn_close(to_f64(y), ref, f"grouped {T}x{k} E={E}")


def test_grouped_swiglu_variant(oracle, cuda_dev):
    """The grouped epilogue with both caps removed (SwiGLU)."""
    T, k, E, M, I = 60, 2, 5, 256, 384
    g = torch.Generator().manual_seed(3)
    ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    x = wl.normal((T, M), 1.0, seed=4)
    wgu, wd = wl.expert_weights(E, M, I, seed=5)
    ids_d = ids.to(cuda_dev)
    off, tix = situ.situ_moe_build_index(ids_d, E)
    inf = float("inf")
    y = situ.situ_moe_grouped_forward(x.to(cuda_dev), off, tix, wgu.to(cuda_dev), wd.to(cuda_dev),
                                      k, inf, inf)
    torch.cuda.synchronize()
    ref = oracle.moe_grouped_forward(oracle_input(x), ids.numpy(), oracle_input(wgu),
                                     oracle_input(wd), 0.0, 0.0)
    assert_ffn_close(to_f64(y), ref, "grouped swiglu")


@pytest.mark.parametrize("T,k,E,M,I,skew", [
    (64, 2, 4, 256, 256, False),    # few rows per expert: one-CTA kernel
    # >= 128 rows per expert on average: two-CTA MMAs; skewed sizes give experts with
    # odd m-tile counts (an M = 128 pair tail), one expert with no rows
    (1024, 2, 4, 512, 384, True),
])
def test_grouped_equals_dense_per_expert(cuda_dev, T, k, E, M, I, skew):
    """Grouped vs naive on the GPU: each (token, slot) row equals the dense FFN of
    that expert applied to the token (same tiles, same rounding of h)."""
    g = torch.Generator().manual_seed(1)
    if skew:
        # slot 0: expert 0 (~70 %) or 1; slot 1: expert 2; expert 3 gets no rows
        first = torch.where(torch.rand(T, generator=g) < 0.7, 0, 1)
        ids = torch.stack([first, torch.full_like(first, 2)], 1).to(torch.int32)
    else:
        ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    x = wl.normal((T, M), 1.0, seed=2)
    wgu, wd = wl.expert_weights(E, M, I, seed=3)
    y = _grouped(x, ids, wgu, wd, cuda_dev).cpu()
    for e in range(E):
        ye = situ.situ_ffn_forward(x.to(cuda_dev), wgu[e].to(cuda_dev), wd[e].to(cuda_dev)).cpu()
        t_idx, s_idx = (ids == e).nonzero(as_tuple=True)
        assert torch.equal(y[t_idx, s_idx].view(torch.int16), ye[t_idx].view(torch.int16))


@pytest.mark.parametrize("sizes", [
    (228, 356, 300, 0, 77),   # odd m-tile counts with tails of 100, 44 and 77 rows
    (129, 192, 64, 385, 1),   # tails of 1 and 64 rows, a 64-row expert, one row
])
def test_grouped_half_pair_tails(oracle, cuda_dev, sizes):
    """Experts averaging >= 128 rows run two-CTA MMAs; an expert's odd last m-tile is an
    M = 128 pair (64 rows per CTA, the second CTA's rows possibly all past the expert's
    end).  Every row equals the dense FFN of its expert bit for bit, and sampled rows
    match the oracle."""
    E, M, I = len(sizes), 256, 384
    ids = torch.cat([torch.full((n,), e, dtype=torch.int32) for e, n in enumerate(sizes)])
    ids = ids[torch.randperm(ids.numel(), generator=torch.Generator().manual_seed(9))][:, None]
    T = ids.shape[0]
    assert T >= 128 * E  # the two-CTA schedule
    x = wl.normal((T, M), 1.0, seed=10)
    wgu, wd = wl.expert_weights(E, M, I, seed=11)
    y = _grouped(x, ids, wgu, wd, cuda_dev).cpu()
    for e in range(E):
        if sizes[e] == 0:
            continue
        ye = situ.situ_ffn_forward(x.to(cuda_dev), wgu[e].to(cuda_dev), wd[e].to(cuda_dev)).cpu()
        t_idx = (ids[:, 0] == e).nonzero(as_tuple=True)[0]
        assert torch.equal(y[t_idx, 0].view(torch.int16), ye[t_idx].view(torch.int16)), e
    rows = torch.arange(0, T, 7)
    ref = oracle.moe_grouped_forward(oracle_input(x[rows]), ids[rows].numpy(), oracle_input(wgu),
                                     oracle_input(wd))
    assert_ffn_close(to_f64(y[rows]), ref, "grouped half-pair tails")
    assert situ.device_status(clear=True) == 0


_WEIGHTS = {}


def _expert_weights(E, M, I, seed, dev):
    """Seeded expert weights, generated once per shape for this module (the
    898-expert set is 34 GB; the decode and prefill checks share it)."""
    key = (E, M, I, seed)
    if key not in _WEIGHTS:
        _WEIGHTS.clear()
        torch.cuda.empty_cache()
        _WEIGHTS[key] = wl.expert_weights(E, M, I, seed=seed, device=dev)
    return _WEIGHTS[key]


@pytest.fixture(scope="module", autouse=True)
def _free_weights():
    yield
    _WEIGHTS.clear()
    torch.cuda.empty_cache()


def _sample_check(oracle, w, dev, n_sample, seed=0):
    ids = wl.routes(w, seed=seed)
    E = w.num_experts
    x = wl.normal((w.T, w.M), 1.0, seed=seed, device=dev)
    wgu, wd = _expert_weights(E, w.M, w.I, seed, dev)
    off, tix = situ.situ_moe_build_index(ids.to(dev), E)
    y = situ.situ_moe_grouped_forward(x, off, tix, wgu, wd, w.k_eff)
    torch.cuda.synchronize()
    off_c = off.cpu().numpy()
    tix_c = tix.cpu().numpy()
    g = torch.Generator().manual_seed(seed + 99)
    # first and last row of several groups, plus random rows
    nonempty = np.flatnonzero(np.diff(off_c) > 0)
    pick = list(off_c[nonempty[:8]]) + list(off_c[nonempty[-8:] + 1] - 1)
    pick += torch.randint(0, w.T * w.k_eff, (n_sample - len(pick),), generator=g).tolist()
    for r in pick:
        flat = int(tix_c[r])
        t, s = divmod(flat, w.k_eff)
        e = int(ids[t, s])
        ref = oracle.ffn_forward(oracle_input(x[t:t + 1].cpu()), oracle_input(wgu[e].cpu()),
                                 oracle_input(wd[e].cpu()))
        assert_ffn_close(to_f64(y[t, s:s + 1]), ref, f"{w.name}: row {r} (t={t}, s={s}, e={e})")


def test_grouped_zipf_full_size_sampled(oracle, cuda_dev):
    _sample_check(oracle, wl.WORKLOADS["grouped"], cuda_dev, 40)


def test_k3_decode_full_size_sampled(oracle, cuda_dev):
    _sample_check(oracle, wl.WORKLOADS["k3_decode"], cuda_dev, 40)


def test_k3_prefill_full_size_sampled(oracle, cuda_dev):
    """The 32768-token K3-shaped layer (898 experts, 327680 routes) as the benchmark
    launches it; the oracle checks 40 routes (first and last rows of several experts,
    the shared experts' included, and random routes)."""
    _sample_check(oracle, wl.WORKLOADS["k3_prefill"], cuda_dev, 40)


def test_bad_offsets_write_nothing(cuda_dev):
    T, k, E, M, I = 8, 2, 3, 64, 64
    x = wl.normal((T, M), 1.0, seed=0, device=cuda_dev)
    wgu, wd = wl.expert_weights(E, M, I, seed=0, device=cuda_dev)
    off = torch.tensor([0, 10, 5, 16], dtype=torch.int32, device=cuda_dev)  # not monotone
    tix = torch.arange(T * k, dtype=torch.int32, device=cuda_dev)
    y = torch.full((T, k, M), 7.0, dtype=torch.bfloat16, device=cuda_dev)
    situ.situ_moe_grouped_forward(x, off, tix, wgu, wd, k, y=y)
    torch.cuda.synchronize()
    assert situ.device_status(clear=True) == 7
    assert bool((y == 7.0).all())


# ---------------------------------------------------------------------------
# Combine (router-weighted sum of a token's slot outputs)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("T,k,M,dtype", [(100, 10, 2048, torch.bfloat16), (7, 3, 12, torch.bfloat16),
                                         (33, 4, 64, torch.float32), (5, 1, 6, torch.float32)])
def test_combine_against_oracle(oracle, cuda_dev, T, k, M, dtype):
    """FP32 accumulation in slot order, one rounding: within 1 bf16 ulp of the FP64
    combine plus 1e-6 of sum |w y| (cancellation)."""
    y = wl.normal((T, k, M), 1.0, seed=T + k, dtype=dtype)
    w = wl.combine_weights(T, k - 1 if k > 1 else 1, 1 if k > 1 else 0, seed=k)
    out = situ.situ_moe_combine(y.to(cuda_dev), w.to(cuda_dev))
    torch.cuda.synchronize()
    ref = oracle.moe_combine(to_f64(y), w.numpy())
    slack = 1e-6 * np.einsum("tk,tkm->tm", np.abs(w.numpy().astype(np.float64)), np.abs(to_f64(y)))
    err = np.abs(to_f64(out) - ref)
    from numerics import bf16_ulp
    assert (err <= bf16_ulp(ref) + slack).all(), float((err - bf16_ulp(ref)).max())


def test_moe_layer_output(oracle, cuda_dev):
    """Index, grouped experts and combine together (a routed layer's output)
    against the oracle's grouped FFN and combine."""
    T, k, E, M, I = 40, 3, 6, 256, 384
    g = torch.Generator().manual_seed(31)
    ids = torch.stack([torch.randperm(E - 1, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    ids = torch.cat([ids, torch.full((T, 1), E - 1, dtype=torch.int32)], dim=1)  # a shared expert
    x = wl.normal((T, M), 1.0, seed=32)
    wgu, wd = wl.expert_weights(E, M, I, seed=33)
    w = wl.combine_weights(T, k, 1, seed=34)
    off, tix = situ.situ_moe_build_index(ids.to(cuda_dev), E)
    y = situ.situ_moe_grouped_forward(x.to(cuda_dev), off, tix, wgu.to(cuda_dev), wd.to(cuda_dev),
                                      k + 1)
    out = situ.situ_moe_combine(y, w.to(cuda_dev))
    torch.cuda.synchronize()
    yref = oracle.moe_grouped_forward(oracle_input(x), ids.numpy(), oracle_input(wgu),
                                      oracle_input(wd))
    ref = oracle.moe_combine(yref, w.numpy())
    assert_ffn_close(to_f64(out), ref, "moe layer output")


# ---------------------------------------------------------------------------
# Combine fused into the down projection (FP32 scatter-add)
# ---------------------------------------------------------------------------
def _layer_case(T, k, E, M, I, seed, dev):
    g = torch.Generator().manual_seed(seed)
    ids = torch.stack([torch.randperm(E - 1, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    ids = torch.cat([ids, torch.full((T, 1), E - 1, dtype=torch.int32)], dim=1)  # a shared expert
    x = wl.normal((T, M), 1.0, seed=seed + 1)
    wgu, wd = wl.expert_weights(E, M, I, seed=seed + 2)
    w = wl.combine_weights(T, k, 1, seed=seed + 3)
    off, tix = situ.situ_moe_build_index(ids.to(dev), E)
    return ids, x, wgu, wd, w, off, tix


@pytest.mark.parametrize("T,k,E,M,I", [(40, 3, 6, 256, 384), (300, 2, 4, 136, 200)])
def test_fused_combine_against_oracle(oracle, cuda_dev, T, k, E, M, I):
    ids, x, wgu, wd, w, off, tix = _layer_case(T, k, E, M, I, T + E, cuda_dev)
    out = situ.situ_moe_grouped_forward_combined(x.to(cuda_dev), off, tix, wgu.to(cuda_dev),
                                                 wd.to(cuda_dev), w.to(cuda_dev))
    torch.cuda.synchronize()
    assert situ.device_status(clear=True) == 0
    yref = oracle.moe_grouped_forward(oracle_input(x), ids.numpy(), oracle_input(wgu),
                                      oracle_input(wd))
    assert_ffn_close(to_f64(out), oracle.moe_combine(yref, w.numpy()), "fused combine")


def test_fused_combine_matches_unfused(cuda_dev):
    """The fused and the separate combine add the same weighted rows; they differ by
    the bf16 rounding of each route's row in the separate path (2^-9 |w y| a route),
    the order of the FP32 additions (2^-22 sum |w y|) and the output rounding (one
    bf16 ulp of either result): |fused - unfused| <= 2^-8 sum_s |w_s y_s| + 2^-7 |out|."""
    T, k, E, M, I = 256, 4, 8, 512, 384
    ids, x, wgu, wd, w, off, tix = _layer_case(T, k, E, M, I, 77, cuda_dev)
    xd, wgud, wdd, wdv = x.to(cuda_dev), wgu.to(cuda_dev), wd.to(cuda_dev), w.to(cuda_dev)
    fused = situ.situ_moe_grouped_forward_combined(xd, off, tix, wgud, wdd, wdv)
    y = situ.situ_moe_grouped_forward(xd, off, tix, wgud, wdd, k + 1)
    sep = situ.situ_moe_combine(y, wdv)
    torch.cuda.synchronize()
    absum = np.einsum("tk,tkm->tm", np.abs(w.numpy().astype(np.float64)), np.abs(to_f64(y)))
    f, u = to_f64(fused), to_f64(sep)
    tol = 2.0 ** -8 * absum + 2.0 ** -7 * np.maximum(np.abs(f), np.abs(u))
    assert (np.abs(f - u) <= tol).all(), float((np.abs(f - u) / tol).max())


def test_fused_combine_full_size(oracle, cuda_dev):
    """The 64-expert Zipf workload (16384 tokens, top-8, M=2048, I=3072) at full size
    through the fused combine, 16 sampled tokens against the oracle's layer output."""
    wk = wl.WORKLOADS["grouped"]
    E = wk.num_experts
    ids = wl.routes(wk, seed=0)
    x = wl.normal((wk.T, wk.M), 1.0, seed=0, device=cuda_dev)
    wgu, wd = wl.expert_weights(E, wk.M, wk.I, seed=0, device=cuda_dev)
    w = wl.combine_weights(wk.T, wk.k, 0, seed=0)
    off, tix = situ.situ_moe_build_index(ids.to(cuda_dev), E)
    out = situ.situ_moe_grouped_forward_combined(x, off, tix, wgu, wd, w.to(cuda_dev))
    torch.cuda.synchronize()
    assert situ.device_status(clear=True) == 0
    g = torch.Generator().manual_seed(6)
    toks = [0, wk.T - 1] + torch.randint(1, wk.T - 1, (14,), generator=g).tolist()
    for t in toks:
        ref = np.zeros(wk.M)
        for s in range(wk.k):
            e = int(ids[t, s])
            ref += float(w[t, s]) * oracle.ffn_forward(oracle_input(x[t:t + 1].cpu()),
                                                        oracle_input(wgu[e].cpu()),
                                                        oracle_input(wd[e].cpu()))[0]
        assert_ffn_close(to_f64(out[t]), ref, f"fused combine token {t}")
