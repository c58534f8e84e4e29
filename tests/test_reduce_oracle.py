"""The reduction and softmax oracles ("Tiling Strategies", section 5) against
closed forms, exact brute force, independent library routines and the
invariants that define softmax (CPU only); planted mistakes must be caught."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle


# ---------------------------------------------------------------- array sum

def pin_sum_closed_forms(total):
    assert total(np.zeros(0, np.float32)) == 0.0
    for n in (1, 2, 7, 1000, 4097):
        assert total(np.ones(n, np.float32)) == n
        assert total(np.arange(n, dtype=np.float32)) == n * (n - 1) / 2
        alt = np.where(np.arange(n) % 2 == 0, 1.0, -1.0).astype(np.float32)
        assert total(alt) == n % 2


def pin_sum_bruteforce_exact(total):
    rng = np.random.default_rng(70)
    for n in (1, 3, 17, 256, 1001):
        x = (rng.integers(-512, 513, n) / 64).astype(np.float32)
        want = sum((Fraction(float(v)) for v in x), Fraction(0))
        assert Fraction(total(x)) == want, n


def pin_sum_against_fsum(total):
    # math.fsum is correctly rounded; an ascending FP64 sum of n terms is within
    # (n - 1) 2^-53 sum|x| of the exact value.
    rng = np.random.default_rng(71)
    for n in (10, 10_000, 300_001):
        x = rng.standard_normal(n, dtype=np.float32) * np.float32(1e3)
        want = math.fsum(float(v) for v in x)
        bound = (n - 1) * 2.0 ** -53 * float(np.abs(x.astype(np.float64)).sum())
        assert abs(total(x) - want) <= bound + 1e-300, n


SUM_PINS = [pin_sum_closed_forms, pin_sum_bruteforce_exact, pin_sum_against_fsum]


@pytest.mark.parametrize("pin", SUM_PINS, ids=lambda f: f.__name__)
def test_sum_pin(pin):
    pin(oracle.array_sum)


# ---------------------------------------------------------------- softmax

def pin_softmax_constant_rows(sm):
    for cols in (1, 2, 3, 10, 1000):
        x = np.repeat(np.arange(-3, 4, dtype=np.float32)[:, None], cols, axis=1)
        y = sm(x)
        assert y.shape == (7, cols)
        assert np.all(y == 1.0 / cols), cols


def pin_softmax_two_columns_is_logistic(sm):
    # softmax([a, b])_0 = 1 / (1 + e^(b - a)), the logistic function of a - b.
    rng = np.random.default_rng(72)
    x = (rng.standard_normal((200, 2)) * 8).astype(np.float32)
    y = sm(x)
    for r in range(200):
        a, b = float(x[r, 0]), float(x[r, 1])
        want0 = 1.0 / (1.0 + math.exp(b - a))
        want1 = 1.0 / (1.0 + math.exp(a - b))
        assert math.isclose(y[r, 0], want0, rel_tol=1e-14, abs_tol=1e-300)
        assert math.isclose(y[r, 1], want1, rel_tol=1e-14, abs_tol=1e-300)


def pin_softmax_defining_invariants(sm):
    # Rows sum to 1; every ratio y_j / y_k equals e^(x_j - x_k); adding a constant
    # to a row changes nothing (integer values keep x + c exact in float).
    rng = np.random.default_rng(73)
    x = rng.integers(-20, 21, (64, 97)).astype(np.float32)
    y = sm(x)
    assert np.all(np.abs(y.sum(axis=1) - 1.0) <= 97 * 2.0 ** -52)
    for r in range(64):
        j, k = rng.integers(0, 97, 2)
        ratio = y[r, j] / y[r, k]
        assert math.isclose(ratio, math.exp(float(x[r, j]) - float(x[r, k])), rel_tol=1e-13)
    shifted = sm(x + np.float32(1000.0))
    assert np.array_equal(shifted, y)


def pin_softmax_extreme_rows(sm):
    # A gap of 1000 underflows e^(-1000) to 0 in double: the result is one-hot,
    # wherever the maximum sits.  A gap of 30 gives the closed form
    # 1 / (1 + (c - 1) e^-30) on the maximum.
    x = np.zeros((3, 5), np.float32)
    x[0, 0] = 1000.0
    x[1, 4] = 1000.0
    x[2, :] = -1000.0
    x[2, 2] = 0.0
    y = sm(x)
    assert np.array_equal(y, np.eye(5)[[0, 4, 2]])
    x = np.zeros((1, 9), np.float32)
    x[0, 3] = 30.0
    y = sm(x)
    top = 1.0 / (1.0 + 8 * math.exp(-30.0))
    assert math.isclose(y[0, 3], top, rel_tol=1e-15)
    assert math.isclose(y[0, 0], math.exp(-30.0) * top, rel_tol=1e-14)


def pin_softmax_against_library(sm):
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(74)
    for rows, cols in ((5, 1), (33, 513), (4, 20_000)):
        x = (rng.standard_normal((rows, cols)) * 4).astype(np.float32)
        want = special.softmax(x.astype(np.float64), axis=1)
        assert np.allclose(sm(x), want, rtol=1e-12, atol=1e-300), (rows, cols)


def pin_softmax_row_stride(sm):
    # A padded row stride: the padding holds values that would change every
    # result if they were read.
    rng = np.random.default_rng(75)
    x = rng.standard_normal((17, 40)).astype(np.float32)
    padded = np.full((17, 48), 1e30, np.float32)
    padded[:, :40] = x
    assert np.array_equal(sm(padded[:, :40]), sm(np.ascontiguousarray(x)))
    assert sm(np.zeros((0, 5), np.float32)).shape == (0, 5)


SOFTMAX_PINS = [pin_softmax_constant_rows, pin_softmax_two_columns_is_logistic,
                pin_softmax_defining_invariants, pin_softmax_extreme_rows,
                pin_softmax_against_library, pin_softmax_row_stride]


@pytest.mark.parametrize("pin", SOFTMAX_PINS, ids=lambda f: f.__name__)
def test_softmax_pin(pin):
    pin(oracle.softmax_rows)


# ---------------------------------------------------------------- planted mistakes

MUTANTS = {
    "sum_drops_last": ("for (int64_t i = 0; i < n; ++i) s += (double)x[i];",
                       "for (int64_t i = 0; i + 1 < n; ++i) s += (double)x[i];"),
    "sum_single_precision": ("s += (double)x[i];", "s = (float)(s + (double)x[i]);"),
    "softmax_no_max_shift": ("yr[j] = exp((double)xr[j] - m);", "yr[j] = exp((double)xr[j]);"),
    "softmax_min_not_max": ("if ((double)xr[j] > m)", "if ((double)xr[j] < m)"),
    "softmax_sign": ("yr[j] = exp((double)xr[j] - m);", "yr[j] = exp(m - (double)xr[j]);"),
    "softmax_short_sum": ("s += yr[j];", "if (j + 1 < cols) s += yr[j];"),
    "softmax_ignores_ldx": ("const float *xr = x + r * ldx;", "const float *xr = x + r * cols;"),
}


def _mutant_lib(name, tmp_path):
    src_path = os.path.join(os.path.dirname(oracle.SOURCE), "reduce_oracle.c")
    old, new = MUTANTS[name]
    src = open(src_path).read()
    assert old in src
    c = os.path.join(tmp_path, "m.c")
    open(c, "w").write(src.replace(old, new, 1))
    others = [s for s in oracle.SOURCES if not s.endswith("reduce_oracle.c")]
    so = oracle.compile_source(others + [c], os.path.join(tmp_path, "m.so"))
    return oracle.OracleLib(so)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    lib = _mutant_lib(name, tmp_path)
    if name.startswith("sum"):
        pins, fn = SUM_PINS, lib.array_sum
    else:
        pins, fn = SOFTMAX_PINS, lib.softmax_rows
    failed = []
    for pin in pins:
        try:
            with np.errstate(all="ignore"):
                pin(fn)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, name
