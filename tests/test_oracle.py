"""The CPU oracle against its pins, and the pins against planted mistakes.

CPU only.  The first group runs every pin of ``oracle_pins`` on the oracle as
built from ``oracle/gemm_oracle.c``.  The second compiles copies of that
source with one plausible mistake planted each (a dropped term, a wrong sign,
a wrong stride, an FP32-rounded product, a non-zero start value, a reversed
index) and checks that at least one pin rejects every copy, so the pins do
catch the mistakes they are meant to catch.
"""
import os

import numpy as np
import pytest

import oracle
import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_GEMM_PINS, ids=lambda f: f.__name__)
def test_oracle_gemm_pin(pin):
    pin(oracle.gemm)


@pytest.mark.parametrize("pin", P.ALL_ENTRY_PINS, ids=lambda f: f.__name__)
def test_oracle_entries_pin(pin):
    pin(oracle.gemm_entries)


def test_entries_agree_with_full_product():
    rng = np.random.default_rng(21)
    A = rng.standard_normal((50, 70), dtype=np.float32)
    B = rng.standard_normal((70, 40), dtype=np.float32)
    full = oracle.gemm(A, B)
    ii = rng.integers(0, 50, 200)
    jj = rng.integers(0, 40, 200)
    # Same definition, same ascending-k order: the doubles must be identical.
    assert np.array_equal(oracle.gemm_entries(A, B, ii, jj), full[ii, jj])


def test_thread_count_does_not_change_bits():
    rng = np.random.default_rng(22)
    A = rng.standard_normal((33, 65), dtype=np.float32)
    B = rng.standard_normal((65, 17), dtype=np.float32)
    assert np.array_equal(oracle.gemm(A, B, threads=1), oracle.gemm(A, B, threads=5))


def test_empty_shapes():
    assert oracle.gemm(np.zeros((0, 3), np.float32), np.zeros((3, 4), np.float32)).shape == (0, 4)
    assert oracle.gemm(np.zeros((2, 3), np.float32), np.zeros((3, 0), np.float32)).shape == (2, 0)
    C = oracle.gemm(np.zeros((2, 0), np.float32), np.zeros((0, 3), np.float32))
    assert C.shape == (2, 3) and np.all(C == 0)


def test_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.gemm(np.zeros((2, 3), np.float32), np.zeros((4, 2), np.float32))
    with pytest.raises(TypeError):
        oracle.gemm(np.zeros((2, 3), np.float64), np.zeros((3, 2), np.float32))
    with pytest.raises(ValueError):
        oracle.gemm_entries(np.zeros((2, 3), np.float32), np.zeros((3, 2), np.float32),
                            [2], [0])


def test_fp32_rounding_is_round_to_nearest_even():
    # 1 + 2^-24 is a tie between 1 and 1 + 2^-23; nearest-even gives 1.
    A = np.array([[1.0, 2.0 ** -12]], np.float32)
    B = np.array([[1.0], [2.0 ** -12]], np.float32)
    assert oracle.gemm(A, B)[0, 0] == 1.0 + 2.0 ** -24
    assert oracle.gemm_f32(A, B)[0, 0] == np.float32(1.0)
    # 1 + 3*2^-24 is a tie between 1 + 2^-23 and 1 + 2^-22; nearest-even gives the latter.
    B2 = np.array([[1.0], [3.0 * 2.0 ** -12]], np.float32)
    assert oracle.gemm_f32(A, B2)[0, 0] == np.float32(1.0 + 2.0 ** -22)


# -- planted mistakes ------------------------------------------------------------------

MUTANTS = {
    # full product: first term dropped
    "drop_first_term": ("for (int64_t k = 0; k < K; ++k) {\n            const double a_ik",
                        "for (int64_t k = 1; k < K; ++k) {\n            const double a_ik"),
    # full product: last term dropped
    "drop_last_term": ("for (int64_t k = 0; k < K; ++k) {\n            const double a_ik",
                       "for (int64_t k = 0; k < K - 1; ++k) {\n            const double a_ik"),
    "wrong_sign": ("c_row[j] += a_ik", "c_row[j] -= a_ik"),
    "product_rounded_to_fp32": ("c_row[j] += a_ik * (double)b_row[j];",
                                "c_row[j] += (float)(a_ik * (double)b_row[j]);"),
    "nonzero_start": ("c_row[j] = 0.0;", "c_row[j] = 1.0;"),
    "a_stride_ignores_lda": ("(double)A[i * lda + k];", "(double)A[i * K + k];"),
    "b_stride_ignores_ldb": ("B + k * ldb;", "B + k * N;"),
    "a_reversed_k": ("(double)A[i * lda + k];", "(double)A[i * lda + (K - 1 - k)];"),
    "entries_wrong_sign": ("acc += (double)A", "acc -= (double)A"),
    "entries_b_index_swapped": ("(double)B[k * ldb + j]", "(double)B[k * ldb + (N - 1 - j)]"),
}


def _failing_pins(lib):
    failed = []
    for pin in P.ALL_GEMM_PINS:
        try:
            pin(lib.gemm)
        except AssertionError:
            failed.append(pin.__name__)
    for pin in P.ALL_ENTRY_PINS:
        try:
            pin(lib.gemm_entries)
        except AssertionError:
            failed.append(pin.__name__)
    return failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    with open(oracle.SOURCE) as f:
        src = f.read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new, 1)
    c_path = os.path.join(tmp_path, f"{name}.c")
    with open(c_path, "w") as f:
        f.write(mutated)
    lib = oracle.OracleLib(oracle.compile_source(c_path, os.path.join(tmp_path, f"{name}.so")))
    assert _failing_pins(lib), f"no pin caught the planted mistake {name}"
