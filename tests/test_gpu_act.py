"""Standalone SiTU-GLU activation on the GPU against the FP64 oracle.

Tolerance: 1 bf16 ulp of the oracle value, and |out| <= beta1*beta2 exactly."""
import math

import numpy as np
import pytest
import torch

import situ_glu_activation_gb300 as situ
from situ_glu_activation_gb300 import workloads as wl
from numerics import assert_within_ulp, oracle_input, to_f64

pytestmark = pytest.mark.gpu


def _all_bf16():
    return torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)


def _bits(v):
    return torch.tensor([v], dtype=torch.int32).to(torch.int16).view(torch.bfloat16).item()


OTHER = [2.0, -3.0, 0.5, 25.0, -1e4, 1e-3, -1e-30, 100.0, 7.5, -60.0,
         _bits(0x0001), _bits(0x8080), float("inf")]


INF = float("inf")
# The variants: up branch uncapped (linear_beta None), gate uncapped, SwiGLU.
VARIANTS = [(4.0, INF), (INF, 25.0), (INF, INF)]


def _oracle_caps(b1, b2):
    """The oracle writes "no cap" as a cap of 0."""
    return (0.0 if b1 == INF else b1), (0.0 if b2 == INF else b2)


def _run(gate_up_cpu, dev, beta=4.0, lbeta=25.0):
    out = situ.situ_glu_act(gate_up_cpu.to(dev), beta, lbeta)
    torch.cuda.synchronize()
    return to_f64(out)


@pytest.mark.parametrize("half", ["gate", "up"])
def test_exhaustive_bf16(oracle, cuda_dev, half):
    """Every bf16 value as g (or as u), against a set of fixed partners."""
    allv = _all_bf16()
    n = allv.numel()
    rows = []
    for v in OTHER:
        fixed = torch.full((n,), v, dtype=torch.bfloat16)
        rows.append(torch.cat([allv, fixed]) if half == "gate" else torch.cat([fixed, allv]))
    gate_up = torch.stack(rows)  # [len(OTHER), 2 * 65536]
    got = _run(gate_up, cuda_dev)
    ref = oracle.situ_glu_act(oracle_input(gate_up))
    assert_within_ulp(got, ref, f"exhaustive {half}")


# Partners for the uncapped variants: finite and within the variants' stated
# domain |u| <= 2^50.  The gate branch is carried as 2^64 a (a FP32 number), so a
# gate value below about 2^-188 (g < -131) is zero there; times |u| <= 2^50 the
# exact product is below half the smallest bf16 subnormal, so the output is still
# correctly rounded.  Beyond 2^50, or with an infinite u (0 * inf = NaN, as in an
# FP32 evaluation of the pages' formula), the variants are not graded.
OTHER_FINITE = [v for v in OTHER if math.isfinite(v)] + [1e10, 2.0 ** 50, -(2.0 ** 50)]


@pytest.mark.parametrize("caps", VARIANTS, ids=["up_uncapped", "gate_uncapped", "swiglu"])
@pytest.mark.parametrize("half", ["gate", "up"])
def test_exhaustive_bf16_variants(oracle, cuda_dev, caps, half):
    """The uncapped variants on every bf16 value of one branch (no bound applies)."""
    allv = _all_bf16()
    n = allv.numel()
    rows = []
    for v in OTHER_FINITE:
        fixed = torch.full((n,), v, dtype=torch.bfloat16)
        rows.append(torch.cat([allv, fixed]) if half == "gate" else torch.cat([fixed, allv]))
    gate_up = torch.stack(rows)
    got = _run(gate_up, cuda_dev, *caps)
    ref = oracle.situ_glu_act(oracle_input(gate_up), *_oracle_caps(*caps))
    assert_within_ulp(got, ref, f"exhaustive {half} {caps}", bound=INF)


@pytest.mark.parametrize("caps", VARIANTS, ids=["up_uncapped", "gate_uncapped", "swiglu"])
def test_fp32_variants(oracle, cuda_dev, caps):
    g = wl.gate_up_input(wl.WORKLOADS["act"], seed=8, rows=64).float()
    got = _run(g, cuda_dev, *caps)
    ref = oracle.situ_glu_act(oracle_input(g), *_oracle_caps(*caps))
    err = np.abs(got - ref)
    assert (err <= 1e-5 * np.abs(ref) + 1e-40).all(), float((err / (np.abs(ref) + 1e-40)).max())


def test_act_workload_slab(oracle, cuda_dev):
    """2048 rows of the memory-bound workload (N(0,3) + 1% outliers), every output."""
    w = wl.WORKLOADS["act"]
    gate_up = wl.gate_up_input(w, seed=0, rows=2048)
    got = _run(gate_up, cuda_dev)
    ref = oracle.situ_glu_act(oracle_input(gate_up))
    assert_within_ulp(got, ref, "act slab")
    # the outliers reach both saturation and the subnormal tail
    assert (np.abs(ref) > 99.0).any() and ((ref != 0) & (np.abs(ref) < 2.0 ** -126)).any()


def test_act_full_size_sampled(oracle, cuda_dev):
    """The full [65536, 6144] workload in the launch the benchmark times; the oracle
    checks a seeded sample of 256 whole rows (first and last included)."""
    w = wl.WORKLOADS["act"]
    gate_up = wl.gate_up_input(w, seed=0, device=cuda_dev)
    out = situ.situ_glu_act(gate_up)
    torch.cuda.synchronize()
    g = torch.Generator().manual_seed(5)
    rows = torch.cat([torch.tensor([0, w.rows - 1]), torch.randint(0, w.rows, (254,), generator=g)])
    rows_d = rows.to(cuda_dev)
    ref = oracle.situ_glu_act(oracle_input(gate_up[rows_d].cpu()))
    assert_within_ulp(to_f64(out[rows_d]), ref, "act full size sample")
    assert float(out.abs().max()) <= 100.0


@pytest.mark.parametrize("rows,I", [(1, 1), (3, 5), (7, 12), (33, 8), (129, 3072), (5, 4100)])
def test_ragged_shapes(oracle, cuda_dev, rows, I):
    """Odd widths take the scalar path, multiples of 8 the vector path."""
    gate_up = wl.normal((rows, 2 * I), 3.0, seed=rows * 1000 + I)
    got = _run(gate_up, cuda_dev)
    assert got.shape == (rows, I)
    assert_within_ulp(got, oracle.situ_glu_act(oracle_input(gate_up)), f"{rows}x{I}")


def test_unaligned_pointer_scalar_path(oracle, cuda_dev):
    """A view starting 2 bytes into an allocation cannot use 16-byte vectors."""
    base = wl.normal((8 * 64 + 1,), 3.0, seed=3).to(cuda_dev)
    gate_up = base[1:].view(8, 64)
    out = situ.situ_glu_act(gate_up)
    torch.cuda.synchronize()
    assert_within_ulp(to_f64(out), oracle.situ_glu_act(oracle_input(gate_up.cpu())), "unaligned")


def test_leading_dims_and_empty(oracle, cuda_dev):
    gate_up = wl.normal((2, 3, 4, 16), 2.0, seed=9)
    got = _run(gate_up, cuda_dev)
    assert got.shape == (2, 3, 4, 8)
    assert_within_ulp(got.reshape(-1, 8), oracle.situ_glu_act(oracle_input(gate_up.reshape(-1, 16))),
                      "leading dims")
    empty = situ.situ_glu_act(torch.empty(0, 16, dtype=torch.bfloat16, device=cuda_dev))
    assert empty.shape == (0, 8)


def test_fp32_special_rows(oracle, cuda_dev):
    """The tiny configuration's scalar rows: worked example, the bound at +-1e4, one
    saturated branch, the subnormal tail; float32 in and out."""
    for pad in (None, 16):
        gate_up = wl.special_gate_up(torch.float32, pad_to=pad)
        got = _run(gate_up, cuda_dev)
        ref = oracle.situ_glu_act(oracle_input(gate_up))
        assert_within_ulp(got, ref, "fp32 special rows")
        assert abs(got[0, 0] - 3.2493226) < 1e-5          # worked example
        assert got[0, 1] == 100.0 and got[0, 2] == -100.0  # the bound, reached


def test_fp32_relative_accuracy(oracle, cuda_dev):
    """float32 outputs take the accurate exponential form: relative error below
    1e-5 (far inside a bf16 ulp), absolute 1e-40 near zero."""
    g = wl.gate_up_input(wl.WORKLOADS["act"], seed=3, rows=256).float()
    got = _run(g, cuda_dev)
    ref = oracle.situ_glu_act(oracle_input(g))
    err = np.abs(got - ref)
    assert (err <= 1e-5 * np.abs(ref) + 1e-40).all(), float((err / (np.abs(ref) + 1e-40)).max())


def test_caps_are_arguments(oracle, cuda_dev):
    gate_up = wl.normal((64, 256), 10.0, seed=4)
    for b1, b2 in [(25.0, 4.0), (1.0, 1.0), (8.0, 50.0)]:
        got = _run(gate_up, cuda_dev, b1, b2)
        assert_within_ulp(got, oracle.situ_glu_act(oracle_input(gate_up), b1, b2),
                          f"caps {b1},{b2}", bound=b1 * b2)


def test_inputs_not_mutated(cuda_dev):
    gate_up = wl.normal((16, 64), 3.0, seed=2).to(cuda_dev)
    before = gate_up.clone()
    situ.situ_glu_act(gate_up)
    torch.cuda.synchronize()
    assert torch.equal(gate_up.view(torch.int16), before.view(torch.int16))
