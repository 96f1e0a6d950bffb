"""Comparison helpers for the GPU parity tests (test code, not the oracle).

Tolerances (the stated targets):
  * standalone activation: |gpu - ref| <= 1 bf16 ulp of the FP64 oracle value ref,
    ulp(ref) = 2^(floor(log2|ref|) - 7) for |ref| >= 2^-126, else 2^-133 (the bf16
    subnormal spacing; gradual underflow assumed), sign of zero ignored; and
    |gpu| <= beta1 * beta2 exactly.
  * FFN / grouped outputs (FP32 accumulation): |gpu - ref| <= 2e-2 * (1 + |ref|).
  * indices: bit-exact.
"""
from __future__ import annotations

import numpy as np
import torch

FFN_TOL = 2e-2


def bf16_ulp(ref: np.ndarray) -> np.ndarray:
    mag = np.abs(np.asarray(ref, dtype=np.float64))
    normal = mag >= 2.0 ** -126
    e = np.floor(np.log2(np.where(normal, mag, 1.0)))
    return np.where(normal, 2.0 ** (e - 7), 2.0 ** -133)


def to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 copy of a bf16 / fp32 tensor."""
    return t.detach().float().cpu().double().numpy()


def oracle_input(t: torch.Tensor) -> np.ndarray:
    """The array the oracle takes for a tensor: bf16 as raw bits, fp32 as is."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy()
    return t.double().numpy()


BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def assert_within_ulp(got: np.ndarray, ref: np.ndarray, what: str = "", bound: float = 100.0,
                      max_finite: float = BF16_MAX):
    """|got - ref| <= 1 bf16 ulp of ref; where |ref| exceeds the output type's largest
    finite value, +-inf of ref's sign is also accepted (round-to-nearest overflow)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    nan_ref = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan_ref), f"{what}: NaN pattern differs"
    g, r = got[~nan_ref], ref[~nan_ref]
    overflow_ok = (np.abs(r) > max_finite) & np.isinf(g) & (np.sign(g) == np.sign(r))
    with np.errstate(invalid="ignore"):
        err = np.abs(g - r)
    ulp = bf16_ulp(r)
    bad = ~(err <= ulp) & ~overflow_ok
    if bad.any():
        i = np.flatnonzero(bad)[:8]
        raise AssertionError(f"{what}: {bad.sum()} of {r.size} outputs off by more than 1 bf16 "
                             f"ulp; e.g. got {g[i]}, ref {r[i]}, ulp {ulp[i]}")
    assert np.abs(g).max(initial=0.0) <= bound, f"{what}: bound {bound} exceeded"


def assert_ffn_close(got: np.ndarray, ref: np.ndarray, what: str = "", tol: float = FFN_TOL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    scaled = np.abs(got - ref) / (1.0 + np.abs(ref))
    assert scaled.max(initial=0.0) <= tol, (
        f"{what}: max |err|/(1+|ref|) = {scaled.max():.4g} > {tol} at "
        f"{np.unravel_index(scaled.argmax(), scaled.shape)}")
    return float(scaled.max(initial=0.0))
