"""Acceptance metrics for a GPU result against the oracle (host-side numpy only).

For FP32 inputs drawn at random the bar is
  * normwise:    ||C - C_ref||_F / ||C_ref||_F <= 1e-5  (norms in FP64),
  * elementwise: max |C - C_ref| <= 1e-4 * sqrt(K),
with C_ref the oracle's FP64-accumulated product.  Sequential FP32
accumulation of K terms has a random-walk relative error of about
2^-24 * sqrt(K / 6), 1.6e-6 at K = 4096, so the normwise bar leaves a margin
of several times for any summation order.  For integer-valued inputs every
partial sum is exact in FP32, so the result must equal the oracle rounded to
FP32 bit for bit.
"""
from __future__ import annotations

import math

import numpy as np

NORMWISE_TOL = 1e-5


def elementwise_tol(K: int) -> float:
    return 1e-4 * math.sqrt(max(K, 1))


def errors(C: np.ndarray, ref: np.ndarray):
    """(normwise relative error, max abs error) of float32 C against float64 ref."""
    d = C.astype(np.float64) - ref
    denom = np.linalg.norm(ref)
    norm_err = np.linalg.norm(d) / denom if denom > 0 else np.linalg.norm(d)
    max_err = float(np.max(np.abs(d))) if d.size else 0.0
    return float(norm_err), max_err


def assert_close(C: np.ndarray, ref: np.ndarray, K: int, what: str = ""):
    assert C.shape == ref.shape, (C.shape, ref.shape)
    assert np.all(np.isfinite(C)), f"{what}: non-finite entries"
    norm_err, max_err = errors(C, ref)
    assert norm_err <= NORMWISE_TOL, f"{what}: normwise error {norm_err:.3e} > {NORMWISE_TOL}"
    tol = elementwise_tol(K)
    assert max_err <= tol, f"{what}: max abs error {max_err:.3e} > {tol:.3e}"
    return norm_err, max_err


def assert_bit_exact(C: np.ndarray, ref: np.ndarray, what: str = ""):
    want = ref.astype(np.float32)
    assert C.shape == want.shape
    bad = np.flatnonzero(C.view(np.uint32) != want.view(np.uint32))
    assert bad.size == 0, (f"{what}: {bad.size} entries differ, first at "
                           f"{np.unravel_index(bad[0], C.shape)}: {C.flat[bad[0]]} vs {want.flat[bad[0]]}")


def assert_close_few_outputs(C: np.ndarray, A: np.ndarray, B: np.ndarray, what: str = ""):
    """For products with only a handful of outputs, where the normwise ratio is a
    single entry's relative error and cancellation (an entry far smaller than its
    terms) can put any FP32 summation order above 1e-5: every entry within the
    elementwise bar 1e-4 sqrt(K) and within the classical bound of an FP32 dot
    product summed in any order, K 2^-24 sum_k |A_ik B_kj|."""
    K = A.shape[1]
    ref = A.astype(np.float64) @ B.astype(np.float64)
    mag = np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64))
    assert np.all(np.isfinite(C)), f"{what}: non-finite entries"
    err = np.abs(C.astype(np.float64) - ref)
    assert np.all(err <= elementwise_tol(K)), f"{what}: max abs error {err.max():.3e}"
    assert np.all(err <= K * 2.0 ** -24 * mag), f"{what}: beyond the FP32 dot-product bound"
