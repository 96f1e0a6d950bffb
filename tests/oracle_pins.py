"""Pins for the FP64 oracle: checks that tie it to what the SiTU-GLU pages print and
to closed forms of the mathematics, never to a second copy of its own formula.

Each pin is a function ``pin(o)`` taking an ``oracle.Oracle`` and raising
AssertionError when the oracle disagrees.  ``test_oracle_pins.py`` runs them on
the real oracle; ``test_oracle_mutants.py`` runs them on deliberately broken
builds of the oracle and requires every mistake to be caught by at least one.

Page titles cited below:
  problem page  "SiTU-GLU" (ai-engineer-exhaustive.pages.dev)
  chapter       "SiTU-GLU" architecture chapter (mkdocs.reaper.mx, French)
  docs page     "DenseFFN and SituGLU - Docs - Kimi K3 from Scratch"
  bound page    "Kimi K3 - Bound the up branch" (atlas.klimoza.dev)
"""
from __future__ import annotations

import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
B1, B2 = 4.0, 25.0  # chapter, "Les valeurs chez Kimi K3"


def load_golden(name: str) -> dict:
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, value, half = line.split()
            vals[key] = (float(value), float(half))
    return vals


def _close(got, want, half, what):
    assert abs(got - want) <= half, f"{what}: oracle {got!r}, page prints {want} (+-{half})"


# ---------------------------------------------------------------------------
# Scalar pins
# ---------------------------------------------------------------------------
def pin_worked_example(o):
    """problem page "A scalar example" and chapter "Verification de comprehension"."""
    gv = load_golden("worked_example.txt")
    g, u = gv["g"][0], gv["u"][0]
    b1, b2 = gv["beta"][0], gv["linear_beta"][0]
    _close(o.softcap(g, b1) / b1, *gv["tanh_half"], "tanh(2/4)")
    _close(o.sigmoid(g), *gv["sigmoid_two"], "sigmoid(2)")
    _close(o.gate(g, b1), *gv["gate_branch"], "gate branch at g=2")
    _close(o.up(u, b2), *gv["up_branch"], "up branch at u=2")
    _close(o.pair(g, u, b1, b2), *gv["product"], "SiTU-GLU at g=u=2")


def pin_swiglu_gate_and_gaps(o):
    """chapter: SwiGLU's gate at x=2 is 1.762; the caps cost about 8 % on the gate
    and 0.2 % on the up branch.  A cap of 1e12 reaches the SwiGLU gate."""
    gv = load_golden("worked_example.txt")
    _close(o.gate(2.0, 1e12), *gv["swiglu_gate"], "uncapped gate (SwiGLU) at 2")
    gap_gate = 1.0 - o.gate(2.0, B1) / o.gate(2.0, 1e12)
    gap_up = 1.0 - o.up(2.0, B2) / 2.0
    _close(gap_gate, *gv["gate_gap_vs_swiglu"], "relative gate gap")
    _close(gap_up, *gv["up_gap_vs_linear"], "relative up gap")


def pin_bound(o):
    """chapter "La borne de sortie": |SiTU-GLU| <= beta1*beta2 = 100 for every input;
    reached at saturation (g -> +inf, |u| -> inf)."""
    gv = load_golden("worked_example.txt")
    bound = gv["bound"][0]
    assert B1 * B2 == bound
    rng = np.random.default_rng(1234)
    samples = np.concatenate([
        rng.normal(0, 3, 2000), rng.normal(0, 1000, 2000),
        rng.choice([-1, 1], 2000) * 10.0 ** rng.uniform(-30, 30, 2000),
        np.array([1e4, -1e4, 1e30, -1e30, 0.0, 88.0, -88.0, 1e-30]),
    ])
    gs = rng.permutation(samples)
    us = rng.permutation(samples)
    for g, u in zip(gs, us):
        h = o.pair(g, u, B1, B2)
        assert abs(h) <= bound, f"|h({g}, {u})| = {abs(h)} > {bound}"
    assert o.pair(1e4, 1e4, B1, B2) == bound
    assert o.pair(1e4, -1e4, B1, B2) == -bound
    assert o.pair(-1e4, 1e4, B1, B2) == 0.0


def pin_saturation_limits(o):
    """problem page "Why scaled tanh is useful": beta*tanh(x/beta) -> +-beta for large
    |x|; the gate cap is beta1 and the up cap is beta2 ("The two caps are
    independent"); for large positive g the sigmoid goes to one."""
    assert o.gate(1e4, B1) == B1
    assert o.up(1e4, B2) == B2 and o.up(-1e4, B2) == -B2
    assert o.softcap(1e6, 7.0) == 7.0 and o.softcap(-1e6, 7.0) == -7.0
    # just short of saturation the soft cap is strictly inside (unlike a clamp)
    assert 0 < o.gate(10.0, B1) < B1 and 0 < o.up(40.0, B2) < B2


def pin_negative_tail(o):
    """problem page: for a large negative gate the sigmoid moves toward zero (Swish's
    vanishing negative side); chapter "Les proprietes": negative tail kept.
    Closed form: for g << 0, tanh(g/4) -> -1 and sigmoid(g) = e^g/(1+e^g), so
    a(g) = -4 e^g (1 + O(e^{g/2}))."""
    for g, rel in [(-80.0, 1e-12), (-40.0, 1e-7), (-200.0, 1e-12)]:
        a = o.gate(g, B1)
        ref = -B1 * math.exp(g)
        assert a < 0, f"a({g}) = {a} should be negative"
        assert abs(a / ref - 1) <= rel, f"a({g}) = {a}, closed form {ref}"
    assert o.sigmoid(-800.0) == 0.0 and o.gate(-1e4, B1) == 0.0


def pin_odd_in_up(o):
    """h is odd in u (the up branch is a scaled tanh, with no sigmoid -- problem page
    "Common mistakes": sigmoid belongs only to the gate)."""
    rng = np.random.default_rng(7)
    for g, u in rng.normal(0, 20, (200, 2)):
        assert o.pair(g, -u, B1, B2) == -o.pair(g, u, B1, B2)
        assert o.up(-u, B2) == -o.up(u, B2)
    assert o.up(-30.0, B2) < -20.0


def pin_first_order(o):
    """chapter: beta*tanh(z/beta) = z + O(z^3/beta^2); SiTU-GLU agrees with SwiGLU to
    first order at the origin.  Closed form of the ratio to SwiGLU:
      h / (g sigmoid(g) u) = [1 - g^2/(3 beta1^2) + ...][1 - u^2/(3 beta2^2) + ...]
                           = 1 - g^2/48 - u^2/1875 + O(4th order)."""
    rng = np.random.default_rng(11)
    for g, u in rng.uniform(1e-3, 2e-2, (200, 2)) * rng.choice([-1, 1], (200, 2)):
        swish = g / (1.0 + math.exp(-g))
        ratio = o.pair(g, u, B1, B2) / (swish * u)
        resid = ratio - (1.0 - g * g / 48.0 - u * u / 1875.0)
        assert abs(resid) <= 1e-9, f"second-order term wrong at g={g}, u={u}: {resid}"


def pin_swiglu_limit(o):
    """chapter "Les proprietes": exactly SwiGLU as beta1, beta2 -> infinity."""
    rng = np.random.default_rng(3)
    for g, u in rng.normal(0, 5, (300, 2)):
        swiglu = g / (1.0 + math.exp(-g)) * u
        h = o.pair(g, u, 1e8, 1e8)
        assert abs(h - swiglu) <= 1e-12 * (abs(swiglu) + 1e-300), (g, u, h, swiglu)


def pin_caps_independent(o):
    """problem page "The two caps are independent": swapping or sharing caps must
    change the result.  At g = u the product is symmetric in the two caps whenever
    sigmoid(g) factors out, so the check uses g = 2, u = 30."""
    h = o.pair(2.0, 30.0, B1, B2)
    assert abs(o.pair(2.0, 30.0, B2, B1) - h) > 1.0
    assert abs(o.pair(2.0, 30.0, B1, B1) - h) > 1.0
    assert abs(o.pair(2.0, 30.0, B2, B2) - h) > 1.0


def pin_bf16_decode(o):
    """Input decoding: bfloat16 bit patterns are the top half of binary32."""
    bits = np.array([[0x4000, 0x4000],  # g = 2, u = 2
                     [0x3F80, 0xC000],  # 1, -2
                     [0x0001, 0x3F80],  # 2^-133 (subnormal), 1
                     [0x4049, 0x7F7F],  # 3.140625, max finite
                     [0xC2B4, 0x4000]],  # -90, 2
                    dtype=np.uint16)
    vals = np.array([[2.0, 2.0], [1.0, -2.0], [2.0 ** -133, 1.0],
                     [3.140625, 3.3895313892515355e38], [-90.0, 2.0]])
    got = o.situ_glu_act(bits.reshape(5, 2))
    want = o.situ_glu_act(vals)
    assert np.array_equal(got, want), (got, want)
    gv = load_golden("worked_example.txt")
    _close(got[0, 0], *gv["product"], "bf16 worked example")


def pin_act_split_order(o):
    """docs page "one split, two softly bounded branches": the first half of the
    last dimension is the gate, the second half the up projection."""
    gate_up = np.array([[2.0, 30.0, 30.0, 2.0],
                        [-5.0, 0.5, 1.0, -7.0]])
    out = o.situ_glu_act(gate_up)
    assert out.shape == (2, 2)
    for r in range(2):
        for j in range(2):
            g, u = gate_up[r, j], gate_up[r, 2 + j]
            assert out[r, j] == o.pair(g, u, B1, B2)
    # pair(2, 30) and pair(30, 2) differ: the halves are not interchangeable
    assert abs(out[0, 0] - o.pair(30.0, 2.0)) > 1.0
    # empty inputs are a no-op
    assert o.situ_glu_act(np.zeros((0, 8))).shape == (0, 4)


# ---------------------------------------------------------------------------
# FFN pins
# ---------------------------------------------------------------------------
def pin_ffn_basis(o):
    """docs page "Two linear maps": gate_up_proj M -> 2I (rows 0..I-1 gate, I..2I-1
    up), down_proj I -> M, [out, in] orientation, no bias.  With a one-hot input and
    a weight that routes the input to gate column c and up column c with value 2,
    h is zero except h[c] = the worked example (about 3.25), and y = h[c] W_down[:, c]."""
    gv = load_golden("worked_example.txt")
    M, I = 6, 4
    rng = np.random.default_rng(5)
    wd = rng.normal(size=(M, I))
    for k in range(M):
        for c in range(I):
            x = np.zeros(M)
            x[k] = 1.0
            wgu = np.zeros((2 * I, M))
            wgu[c, k] = 2.0
            wgu[I + c, k] = 2.0
            y, h = o.ffn_forward(x[None], wgu, wd, want_h=True)
            assert np.count_nonzero(h) == 1 and h[0, c] != 0, h
            _close(h[0, c], *gv["product"], "h at the routed column")
            assert np.array_equal(y[0], h[0, c] * wd[:, c]), (y, h[0, c] * wd[:, c])
    # gate 2 / up 30 at column 1: split order decides the value
    x = np.zeros(M)
    x[0] = 1.0
    wgu = np.zeros((2 * I, M))
    wgu[1, 0] = 2.0
    wgu[I + 1, 0] = 30.0
    _, h = o.ffn_forward(x[None], wgu, wd, want_h=True)
    assert h[0, 1] == o.pair(2.0, 30.0)


def pin_ffn_packed_equals_separate(o):
    """docs page: the packed gate_up_proj is a storage layout, not a coupling of the
    two projections; bound page, KimiBlockSparseMLP: separate gate (w1) and up (w3)
    outputs concatenated.  On small-integer data every FP64 sum is exact, so the
    packed oracle's h must equal the activation of the two separate products
    exactly, and y must equal h W_down^T to rounding."""
    rng = np.random.default_rng(9)
    for (R, M, I) in [(3, 5, 4), (4, 7, 3), (1, 2, 6)]:
        x = rng.integers(-3, 4, (R, M)).astype(np.float64)
        wg = rng.integers(-2, 3, (I, M)).astype(np.float64)
        wu = rng.integers(-2, 3, (I, M)).astype(np.float64)
        wd = rng.normal(size=(M, I))
        y, h = o.ffn_forward(x, np.concatenate([wg, wu]), wd, want_h=True)
        gate_up = np.concatenate([x @ wg.T, x @ wu.T], axis=1)
        assert np.array_equal(h, o.situ_glu_act(gate_up))
        np.testing.assert_allclose(y, h @ wd.T, rtol=1e-13, atol=1e-13)
        assert y.shape == (R, M)


def pin_ffn_dtypes(o):
    """Inputs of any accepted precision decode exactly: float32 and bf16 inputs give
    the same FFN output as their float64 values."""
    rng = np.random.default_rng(2)
    M, I, R = 8, 4, 3
    x32 = rng.normal(size=(R, M)).astype(np.float32)
    wgu32 = rng.normal(size=(2 * I, M)).astype(np.float32)
    wd32 = rng.normal(size=(M, I)).astype(np.float32)
    y32 = o.ffn_forward(x32, wgu32, wd32)
    y64 = o.ffn_forward(x32.astype(np.float64), wgu32.astype(np.float64),
                        wd32.astype(np.float64))
    assert np.array_equal(y32, y64)
    # bf16: truncate float32 bits to their upper half
    tob = lambda a: (a.view(np.uint32) >> 16).astype(np.uint16)
    frm = lambda b: (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    xb, wgb, wdb = tob(x32), tob(wgu32), tob(wd32)
    assert np.array_equal(o.ffn_forward(xb, wgb, wdb), o.ffn_forward(frm(xb), frm(wgb), frm(wdb)))


# ---------------------------------------------------------------------------
# Expert index and grouped pins
# ---------------------------------------------------------------------------
def pin_build_index(o):
    """Stable counting sort, checked by brute-force recount: group sizes are the
    per-expert counts, each group lists exactly that expert's flat routes in
    ascending order, and empty experts give empty groups."""
    rng = np.random.default_rng(4)
    for (n, E) in [(0, 3), (1, 1), (17, 5), (200, 9), (64, 64)]:
        ids = rng.integers(0, E, n).astype(np.int32)
        if n > 10:
            ids[ids == 2] = 3  # force expert 2 empty
        off, tix = o.moe_build_index(ids, E)
        assert off[0] == 0 and off[-1] == n
        for e in range(E):
            want = np.flatnonzero(ids == e)
            assert off[e + 1] - off[e] == want.size
            assert np.array_equal(tix[off[e]:off[e + 1]], want)


def pin_grouped_equals_naive(o):
    """Grouped over experts = one dense FFN per (token, slot) with that slot's expert
    ("grouped vs naive", docs page "Verification"); the y row of (t, s) is flat
    index t*k_eff + s; no combine weights."""
    rng = np.random.default_rng(6)
    T, k_eff, E, M, I = 5, 3, 4, 6, 4
    x = rng.normal(size=(T, M))
    wgu = rng.normal(size=(E, 2 * I, M)) / math.sqrt(M)
    wd = rng.normal(size=(E, M, I)) / math.sqrt(I)
    ids = np.stack([rng.choice([0, 1, 3], k_eff, replace=False) for _ in range(T)]).astype(np.int32)
    y = o.moe_grouped_forward(x, ids, wgu, wd)
    assert y.shape == (T, k_eff, M)
    for t in range(T):
        for s in range(k_eff):
            want = o.ffn_forward(x[t:t + 1], wgu[ids[t, s]], wd[ids[t, s]])[0]
            assert np.array_equal(y[t, s], want), (t, s)


def pin_combine(o):
    """Combine of a routed layer, checked by brute force: one-hot weights pick a
    slot exactly, unit weights give the plain sum over slots (exact on integer
    data), and the result is linear in the weights."""
    rng = np.random.default_rng(12)
    T, k, M = 5, 4, 6
    y = rng.integers(-5, 6, (T, k, M)).astype(np.float64)
    for s in range(k):
        w = np.zeros((T, k))
        w[:, s] = 1.0
        assert np.array_equal(o.moe_combine(y, w), y[:, s, :])
    assert np.array_equal(o.moe_combine(y, np.ones((T, k))), y.sum(axis=1))
    w = rng.integers(-3, 4, (T, k)).astype(np.float64)
    want = np.array([[sum(w[t, s] * y[t, s, m] for s in range(k)) for m in range(M)]
                     for t in range(T)])
    assert np.array_equal(o.moe_combine(y, w), want)
    assert np.array_equal(o.moe_combine(y, 2.0 * w), 2.0 * want)
    w32 = w.astype(np.float32)
    assert np.array_equal(o.moe_combine(y, w32), want)


def pin_pair_grad_finite_differences(o):
    """The derivatives against central differences of the (separately pinned)
    forward: error O(eps^2), far below 1e-6 relative at eps = 1e-5."""
    rng = np.random.default_rng(21)
    pts = list(rng.normal(0, 5, (60, 2))) + [(2.0, 2.0), (0.3, -40.0), (-30.0, 7.0), (60.0, 60.0)]
    for b1, b2 in [(B1, B2), (1.0, 3.0), (0.0, 0.0), (B1, 0.0)]:
        for g, u in pts:
            dg, du = o.pair_grad(g, u, b1, b2)
            eps = 1e-5 * max(1.0, abs(g))
            fg = (o.pair(g + eps, u, b1, b2) - o.pair(g - eps, u, b1, b2)) / (2 * eps)
            eps = 1e-5 * max(1.0, abs(u))
            fu = (o.pair(g, u + eps, b1, b2) - o.pair(g, u - eps, b1, b2)) / (2 * eps)
            assert abs(dg - fg) <= 1e-6 * (1 + abs(fg)), (b1, b2, g, u, dg, fg)
            assert abs(du - fu) <= 1e-6 * (1 + abs(fu)), (b1, b2, g, u, du, fu)


def pin_pair_grad_closed_forms(o):
    """At g = 0: a'(0) = sech^2(0) sigmoid(0) = 1/2, so dh/dg = b(u)/2 and dh/du = 0
    (a(0) = 0).  At u = 0: b'(0) = 1, so dh/du = a(g).  As the caps grow, a'
    becomes Swish's derivative sigmoid(g) (1 + g (1 - sigmoid(g))).  Far out, the
    soft caps keep the gradient nonzero (chapter, soft cap vs hard clamp)."""
    for u in [0.5, 2.0, -7.0, 100.0]:
        dg, du = o.pair_grad(0.0, u)
        assert dg == o.up(u) / 2 and du == 0.0
    for g in [-3.0, 0.25, 2.0, 9.0]:
        dg, du = o.pair_grad(g, 0.0)
        assert du == o.gate(g) and dg == 0.0
    for g in [-2.0, 0.7, 3.0]:
        s = 1.0 / (1.0 + math.exp(-g))
        swish_prime = s * (1 + g * (1 - s))
        dg, _ = o.pair_grad(g, 1.0, 1e8, 1e8)
        assert abs(dg - swish_prime) <= 1e-9, (g, dg, swish_prime)
    dg, du = o.pair_grad(30.0, 60.0)
    assert dg > 0 and du > 0


def pin_ffn_backward_structure(o):
    """The backward's linear algebra by brute force on integer-valued data (exact
    sums): dx = dgu W_gate_up, dW_down = dy^T h, dW_gate_up = dgu^T x, with dgu from
    the pair derivatives and h from the forward oracle."""
    rng = np.random.default_rng(22)
    R, M, I = 3, 5, 4
    x = rng.integers(-2, 3, (R, M)).astype(np.float64)
    wgu = rng.integers(-1, 2, (2 * I, M)).astype(np.float64)
    wd = rng.integers(-2, 3, (M, I)).astype(np.float64)
    dy = rng.integers(-3, 4, (R, M)).astype(np.float64)
    dx, dwg, dwd, dgu = o.ffn_backward(x, wgu, wd, dy, want_dgu=True)
    gu = x @ wgu.T
    _, h = o.ffn_forward(x, wgu, wd, want_h=True)
    dh = dy @ wd
    for r in range(R):
        for j in range(I):
            pg, pu = o.pair_grad(gu[r, j], gu[r, I + j])
            assert dgu[r, j] == dh[r, j] * pg and dgu[r, I + j] == dh[r, j] * pu
    np.testing.assert_allclose(dx, dgu @ wgu, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(dwd, dy.T @ h, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(dwg, dgu.T @ x, rtol=1e-13, atol=1e-13)


def pin_ffn_backward_finite_differences(o):
    """The FFN gradients against central differences of the forward oracle's loss
    L = sum(dy * y) on a tiny random problem."""
    rng = np.random.default_rng(23)
    R, M, I = 2, 3, 2
    x = rng.normal(size=(R, M))
    wgu = rng.normal(size=(2 * I, M))
    wd = rng.normal(size=(M, I))
    dy = rng.normal(size=(R, M))
    dx, dwg, dwd = o.ffn_backward(x, wgu, wd, dy)
    loss = lambda x_, g_, d_: float((dy * o.ffn_forward(x_, g_, d_)).sum())
    eps = 1e-6
    for arr, grad, idx in [(x, dx, 0), (wgu, dwg, 1), (wd, dwd, 2)]:
        for pos in np.ndindex(arr.shape):
            args = [x.copy(), wgu.copy(), wd.copy()]
            args[idx][pos] += eps
            lp = loss(*args)
            args[idx][pos] -= 2 * eps
            lm = loss(*args)
            fd = (lp - lm) / (2 * eps)
            assert abs(grad[pos] - fd) <= 1e-6 * (1 + abs(fd)), (idx, pos, grad[pos], fd)


def pin_grouped_backward(o):
    """The grouped backward against the dense backward, brute force: one expert and
    one slot reproduce the dense backward exactly (same sums in the same order); in
    general dx[t] is the sum over the token's slots of the dense dx of its expert,
    and dW[e] the sum over expert e's routes; unused experts get zero gradients."""
    rng = np.random.default_rng(24)
    T, M, I = 4, 5, 3
    x = rng.normal(size=(T, M))
    wgu = rng.normal(size=(1, 2 * I, M))
    wd = rng.normal(size=(1, M, I))
    dy = rng.normal(size=(T, 1, M))
    gdx, gdwg, gdwd = o.moe_grouped_backward(x, np.zeros((T, 1), np.int32), wgu, wd, dy)
    ddx, ddwg, ddwd = o.ffn_backward(x, wgu[0], wd[0], dy[:, 0, :])
    assert np.array_equal(gdx, ddx) and np.array_equal(gdwg[0], ddwg) and np.array_equal(gdwd[0], ddwd)
    E, k = 4, 2
    ids = np.array([[0, 2], [2, 0], [2, 3], [3, 0]], dtype=np.int32)  # expert 1 unused
    wgu = rng.normal(size=(E, 2 * I, M))
    wd = rng.normal(size=(E, M, I))
    dy = rng.normal(size=(T, k, M))
    gdx, gdwg, gdwd = o.moe_grouped_backward(x, ids, wgu, wd, dy)
    want_dx = np.zeros((T, M))
    want_dwg = np.zeros((E, 2 * I, M))
    want_dwd = np.zeros((E, M, I))
    for t in range(T):
        for s in range(k):
            e = ids[t, s]
            a, b, c = o.ffn_backward(x[t:t + 1], wgu[e], wd[e], dy[t:t + 1, s, :])
            want_dx[t] += a[0]
            want_dwg[e] += b
            want_dwd[e] += c
    np.testing.assert_allclose(gdx, want_dx, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(gdwg, want_dwg, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(gdwd, want_dwd, rtol=1e-12, atol=1e-12)
    assert not gdwg[1].any() and not gdwd[1].any()


def _e4m3_reference_grid():
    """Every finite E4M3 value written out from its definition (sign, 4-bit biased
    exponent, 3-bit mantissa, subnormals m/8 * 2^-6, the all-ones pattern NaN), by
    enumeration rather than through the oracle."""
    vals = {}
    for code in range(256):
        e, m = (code >> 3) & 15, code & 7
        if e == 15 and m == 7:
            continue
        mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
        vals[code] = -mag if code & 0x80 else mag
    return vals


def pin_e4m3_codes(o):
    """E4M3 decoding against the format's definition for all 256 codes: the printed
    landmarks (1.0 = 0x38, 448 the largest, 2^-6 the smallest normal, 2^-9 the
    smallest subnormal), NaN only at S.1111.111, and encode(decode(c)) = c for every
    finite code (no two codes share a value but +0 / -0)."""
    grid = _e4m3_reference_grid()
    dec = o.e4m3_decode(np.arange(256, dtype=np.uint8))
    for c in range(256):
        if c in grid:
            assert dec[c] == grid[c], hex(c)
        else:
            assert np.isnan(dec[c]), hex(c)
    assert dec[0x38] == 1.0 and dec[0x7E] == 448.0 and dec[0x08] == 2.0 ** -6
    assert dec[0x01] == 2.0 ** -9 and dec[0xB8] == -1.0 and dec[0x3C] == 1.5
    codes = np.array(sorted(grid), dtype=np.uint8)
    assert np.array_equal(o.e4m3_encode(dec[codes]), codes)
    pos = np.array([grid[c] for c in range(0x7F)])
    assert (np.diff(pos) > 0).all()  # monotone in the code


def _brute_e4m3(x, pos):
    """Code of the nearest finite E4M3 value to x by brute force over the positive
    grid `pos` (list of (value, code)): ties to the even mantissa, magnitudes from
    448 up clamped to 448, the sign bit kept."""
    a = abs(x)
    if a >= 448.0:
        want = 0x7E
    else:
        d = [abs(a - p[0]) for p in pos]
        best = min(d)
        cands = [pos[i][1] for i in range(len(pos)) if d[i] == best]
        want = cands[0] if len(cands) == 1 else [k for k in cands if k % 2 == 0][0]
    if x < 0 or (x == 0 and np.signbit(x)):
        want |= 0x80
    return want


def pin_e4m3_rounding(o):
    """Rounding to E4M3 by brute force: the nearest finite value of the enumerated
    grid, ties to the even mantissa, magnitudes from 448 up clamped to 448, tiny
    values to a signed zero."""
    grid = _e4m3_reference_grid()
    pos = sorted((v, c) for c, v in grid.items() if c < 0x80)
    rng = np.random.default_rng(40)
    v = np.concatenate([rng.uniform(-500, 500, 3000), rng.uniform(-0.05, 0.05, 3000),
                        np.array([p[0] for p in pos]) * 1.0,
                        [(pos[i][0] + pos[i + 1][0]) / 2 for i in range(len(pos) - 1)],
                        [448.0, 449.0, 464.0, 1e9, -1e9, 2.0 ** -10, -(2.0 ** -10), 2.0 ** -11]])
    got = o.e4m3_encode(v)
    for x, c in zip(v, got):
        assert int(c) == _brute_e4m3(x, pos), (x, hex(int(c)))


def pin_mx_scale(o):
    """The block scale 2^(floor(log2 amax) - 8): amax in [2^e, 2^(e+1)) gives code
    e - 8 + 127, so the block's largest scaled magnitude lies in [256, 512); zero
    blocks and exponents below -127 take code 0."""
    for e in (-100, -9, -1, 0, 1, 6, 7, 8, 100):
        for f in (1.0, 1.5, 1.999):
            assert o.mx_scale_code(f * 2.0 ** e) == e - 8 + 127
    assert o.mx_scale_code(0.0) == 0
    assert o.mx_scale_code(2.0 ** -130) == 0
    assert o.mx_scale_code(2.0 ** 200) == 254
    assert o.e8m0_decode(127) == 1.0 and o.e8m0_decode(0) == 2.0 ** -127
    assert np.isnan(o.e8m0_decode(255))


def pin_mx_quantize(o):
    """MX quantization of bf16 rows against its definition, recomputed here with the
    enumerated E4M3 grid: per 32-column block the scale from the largest magnitude,
    then each element's nearest grid value (clamped to 448) times the scale; plus
    the error bound |dequant - v| <= max(2^-3 |v|, 2^-10 X) (clamping costs at most
    an eighth, rounding a sixteenth, the subnormal quantum 2^-9 X)."""
    rng = np.random.default_rng(41)
    x = rng.normal(0, 3, (6, 96))
    x[0, :32] = 0.0                     # a zero block
    x[1, 32:64] *= 1e-38                # a block of subnormal bf16 values
    x[2, 64:96] = 1.9 * 2.0 ** 5        # clamping: 1.9 * 256 > 448 after scaling
    x[3, 5] = 5000.0                    # one outlier flattens the rest of its block
    xb = o.round_bf16(x)
    xf = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    codes, scales = o.mx_quantize(xb)
    grid = _e4m3_reference_grid()
    pos = sorted((v, c) for c, v in grid.items() if c < 0x80)
    deq = o.mx_dequantize(codes, scales)
    for r in range(6):
        for b in range(3):
            blk = xf[r, 32 * b:32 * b + 32]
            amax = np.abs(blk).max()
            e = int(np.floor(np.log2(amax))) - 8 if amax > 0 else -127
            e = max(-127, min(127, e))
            assert scales[r, b] == e + 127
            X = 2.0 ** e
            for i, v in enumerate(blk):
                assert codes[r, 32 * b + i] == _brute_e4m3(v / X, pos), (r, b, i, v)
                err = abs(deq[r, 32 * b + i] - v)
                assert err <= max(2.0 ** -3 * abs(v), 2.0 ** -10 * X), (r, b, i, v)
    assert (codes[0, :32] == 0).all() and scales[0, 0] == 0
    assert scales[1, 1] == 0
    assert (np.abs(deq[2, 64:96]) == 448.0 * 2.0 ** -3).all()   # clamped: 1.9 * 2^5 -> 448 * 2^-3


def pin_round_bf16(o):
    """bf16 rounding against the bit-level rule on float32 inputs (add 0x7FFF plus
    the kept last bit, drop 16 bits), including ties; doubles between two bf16
    values round to the nearer one (no double rounding through float32)."""
    rng = np.random.default_rng(42)
    f = rng.normal(0, 10, 5000).astype(np.float32)
    bits = f.view(np.uint32).astype(np.uint64)
    ties = ((rng.integers(0, 2 ** 15, 200, dtype=np.uint64) << 16) | 0x8000).astype(np.uint32)
    allf = np.concatenate([f, ties.view(np.float32)]).astype(np.float32)
    bits = allf.view(np.uint32).astype(np.uint64)
    want = ((bits + 0x7FFF + ((bits >> 16) & 1)) >> 16).astype(np.uint16)
    assert np.array_equal(o.round_bf16(allf.astype(np.float64)), want)
    # 1 + 2^-8 + 2^-30 is above the tie between 1 and 1 + 2^-7: rounds up; through
    # float32 it would first become the tie 1 + 2^-8 and then round down to 1.
    assert o.round_bf16(np.array([1.0 + 2.0 ** -8 + 2.0 ** -30]))[0] == 0x3F81


def pin_mx_ffn_exact_inputs(o):
    """The MX FFN on operands whose MX quantization is exact (every block's values
    on the E4M3 grid times a power of two, its largest magnitude in the top binade)
    equals the plain FFN on those values up to the bf16 cast and MX quantization of
    h, which are applied to the plain FFN's h here by the pinned functions."""
    rng = np.random.default_rng(43)
    grid = np.array(sorted(v for c, v in _e4m3_reference_grid().items() if c < 0x80))
    def exact(shape, e):
        v = rng.choice(grid[grid >= 2.0 ** -3], shape) * rng.choice([-1.0, 1.0], shape)
        v = v.reshape(shape[0], -1, 32)
        v[:, :, 0] = 448.0  # top binade: the block scale is 2^0 before the 2^e factor
        return (v * 2.0 ** e).reshape(shape)
    M, I, R = 64, 96, 5
    x = exact((R, M), -8)
    wgu = exact((2 * I, M), -10)
    wd = exact((M, I), -11)
    xq, wguq, wdq = o.mx_quantize(x), o.mx_quantize(wgu), o.mx_quantize(wd)
    for a, q in ((x, xq), (wgu, wguq), (wd, wdq)):
        assert np.array_equal(o.mx_dequantize(*q), a)
    y, hb, (hc, hs) = o.mx_ffn_forward(xq, wguq, wdq)
    _, h = o.ffn_forward(x, wgu, wd, want_h=True)
    assert np.array_equal(hb, o.round_bf16(h))
    hc2, hs2 = o.mx_quantize(hb)
    assert np.array_equal(hc, hc2) and np.array_equal(hs, hs2)
    ref = o.mx_dequantize(hc2, hs2) @ wd.T
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-13)


def pin_e2m1(o):
    """E2M1 against its definition (sign, 2-bit exponent with bias 1, 1-bit mantissa,
    exponent 0 the subnormal m * 0.5): the eight magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6;
    rounding by brute force over them with ties to the even mantissa (0.25 -> 0,
    0.75 -> 1, 2.5 -> 2, 5 -> 4) and magnitudes past 6 clamped."""
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for c in range(16):
        want = mags[c & 7] * (-1.0 if c & 8 else 1.0)
        assert o.e2m1_decode(c) == want, c
    v = np.concatenate([np.linspace(-8, 8, 3201), [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, 1e9,
                                                    -0.25, -5.0, -0.0, 0.0, 1e-30]])
    got = o.e2m1_encode(v)
    for x, c in zip(v, got):
        a = min(abs(x), 6.0)
        d = [abs(a - m) for m in mags]
        best = min(d)
        cands = [i for i in range(8) if d[i] == best]
        want = cands[0] if len(cands) == 1 else [i for i in cands if i % 2 == 0][0]
        if x < 0 or (x == 0 and np.signbit(x)):
            want |= 8
        assert int(c) == want, (x, int(c), want)


def pin_mxfp4_quantize(o):
    """MXFP4 quantization against its definition: scale 2^(floor(log2 amax) - 2) (the
    block maximum lands in [4, 8) before clamping to 6), codes by brute force, packing
    with the even element in the low nibble; dequantize inverts the packing."""
    rng = np.random.default_rng(44)
    x = rng.normal(0, 1, (5, 64))
    x[0, :32] = 0.0
    x[1, 0] = 7.9                      # clamps after scaling
    xb = o.round_bf16(x)
    xf = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    codes, scales = o.mxfp4_quantize(xb)
    assert codes.shape == (5, 32) and scales.shape == (5, 2)
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    deq = o.mxfp4_dequantize(codes, scales)
    for r in range(5):
        for b in range(2):
            blk = xf[r, 32 * b:32 * b + 32]
            amax = np.abs(blk).max()
            e = max(-127, int(np.floor(np.log2(amax))) - 2) if amax > 0 else -127
            assert scales[r, b] == e + 127
            X = 2.0 ** e
            for i, v in enumerate(blk):
                byte = codes[r, (32 * b + i) // 2]
                c = (byte & 15) if i % 2 == 0 else (byte >> 4)
                assert c == o.e2m1_encode(np.array([v / X]))[0], (r, b, i)
                assert deq[r, 32 * b + i] == mags[c & 7] * (-1 if c & 8 else 1) * X
    assert (codes[0, :16] == 0).all() and scales[0, 0] == 0


ALL_PINS = [
    pin_worked_example,
    pin_swiglu_gate_and_gaps,
    pin_bound,
    pin_saturation_limits,
    pin_negative_tail,
    pin_odd_in_up,
    pin_first_order,
    pin_swiglu_limit,
    pin_caps_independent,
    pin_bf16_decode,
    pin_act_split_order,
    pin_ffn_basis,
    pin_ffn_packed_equals_separate,
    pin_ffn_dtypes,
    pin_build_index,
    pin_grouped_equals_naive,
    pin_combine,
    pin_pair_grad_finite_differences,
    pin_pair_grad_closed_forms,
    pin_ffn_backward_structure,
    pin_ffn_backward_finite_differences,
    pin_grouped_backward,
    pin_e4m3_codes,
    pin_e4m3_rounding,
    pin_mx_scale,
    pin_mx_quantize,
    pin_round_bf16,
    pin_mx_ffn_exact_inputs,
    pin_e2m1,
    pin_mxfp4_quantize,
]


def run_all(o) -> list:
    """Run every pin; return the names of those that fail (any exception)."""
    failed = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except Exception:
            failed.append(pin.__name__)
    return failed


if __name__ == "__main__":
    # Child-process entry used by the mutation tests: a planted mistake may
    # corrupt memory, so each broken build runs in a process of its own.
    import json
    import sys

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    from oracle import Oracle, load

    print("PINS_FAILED " + json.dumps(run_all(Oracle(load(sys.argv[1])))), flush=True)
