"""The seeded input generators (CPU): shapes, determinism and the routing
constructions stated in the recipe."""
import torch

from situ_glu_activation_gb300 import workloads as wl


def test_normal_is_seeded_and_scaled():
    a = wl.normal((1000, 64), 3.0, seed=5, dtype=torch.float32)
    b = wl.normal((1000, 64), 3.0, seed=5, dtype=torch.float32)
    c = wl.normal((1000, 64), 3.0, seed=6, dtype=torch.float32)
    assert torch.equal(a, b) and not torch.equal(a, c)
    assert abs(float(a.std()) - 3.0) < 0.05 and abs(float(a.mean())) < 0.05
    h = wl.normal((4, 8), 1.0, seed=5)
    assert h.dtype == torch.bfloat16


def test_outliers_fraction_and_range():
    w = wl.WORKLOADS["act"]
    g = wl.gate_up_input(w, seed=0, rows=512).float()
    big = g.abs() >= 50.0
    frac = float(big.float().mean())
    assert 0.008 < frac < 0.012  # p = 0.01 (plus a negligible N(0,3) tail beyond 50)
    assert float(g.abs().max()) <= 5000.0 * (1 + 2 ** -8)
    assert float((g[big] > 0).float().mean()) > 0.4 and float((g[big] < 0).float().mean()) > 0.4


def test_zipf_routes():
    w = wl.WORKLOADS["grouped"]
    ids = wl.routes(w, seed=0)
    assert ids.shape == (16384, 8) and ids.dtype == torch.int32
    srt = ids.sort(dim=1).values
    assert bool((srt[:, 1:] != srt[:, :-1]).all())  # distinct experts per token
    counts = torch.bincount(ids.view(-1).long(), minlength=64)
    assert int((counts == 0).sum()) == 4             # the forced-empty experts
    # Zipf popularity: the busiest expert takes a large share of the routes
    assert int(counts.max()) > 0.1 * ids.numel()
    assert torch.equal(ids, wl.routes(w, seed=0))


def test_uniform_routes_with_shared():
    w = wl.WORKLOADS["k3_decode"]
    ids = wl.routes(w, seed=0)
    assert ids.shape == (512, 10)
    assert bool((ids[:, 8] == 896).all()) and bool((ids[:, 9] == 897).all())
    assert int(ids[:, :8].max()) < 896
    srt = ids.sort(dim=1).values
    assert bool((srt[:, 1:] != srt[:, :-1]).all())


def test_special_rows():
    row = wl.special_gate_up(torch.float32)
    n = len(wl.SPECIAL_PAIRS)
    assert row.shape == (1, 2 * n)
    assert float(row[0, 0]) == 2.0 and float(row[0, n]) == 2.0
    assert wl.special_gate_up(torch.float32, pad_to=16).shape == (1, 32)
