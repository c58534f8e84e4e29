"""Checks that pin a matrix-product routine to facts fixed outside itself.

Each ``pin_*`` takes ``gemm(A, B) -> float64 ndarray`` (and, where named,
``entries(A, B, ii, jj) -> float64 ndarray``) and raises AssertionError when the
routine disagrees with what the pages or plain mathematics fix:

* the worked outer-product example of "CMU DLSys Lecture 12: GPU
  Acceleration", section 4 (fixture in ``golden/``);
* closed forms: A I = A, I B = B, permutation matrices gather rows/columns,
  all-ones operands give C = K, integer rank-1 factors give
  C = (w . x) u v^T;
* exact rational brute force (``fractions.Fraction``) on every shape up to
  4 x 4 x 4 with dyadic entries, where the double result must be exact;
* an independent FP64 library product (numpy) within FP64 rounding;
* Freivalds' identity C x = A (B x) on a larger random case;
* padded leading dimensions whose padding holds NaN (never read).

The set is chosen so that a dropped term, a wrong sign, a wrong index or
stride, a transposed operand, or an FP32-rounded product each fails at least
one check; ``test_oracle.py`` plants such mistakes in compiled copies of the
oracle source to show it.
"""
from __future__ import annotations

import itertools
import os
from fractions import Fraction

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_matrix_fixture(name: str):
    """Parse a golden fixture: header lines 'M m', 'N n', 'K k', then A, B, C blocks."""
    dims, blocks, cur = {}, {}, None
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            if parts[0] in ("M", "N", "K") and len(parts) == 2:
                dims[parts[0]] = int(parts[1])
            elif parts[0] in ("A", "B", "C") and len(parts) == 1:
                cur = parts[0]
                blocks[cur] = []
            else:
                blocks[cur].append([float(v) for v in parts])
    M, N, K = dims["M"], dims["N"], dims["K"]
    A = np.array(blocks["A"], dtype=np.float32).reshape(M, K)
    B = np.array(blocks["B"], dtype=np.float32).reshape(K, N)
    C = np.array(blocks["C"], dtype=np.float64).reshape(M, N)
    return A, B, C


def pin_worked_example(gemm):
    A, B, C = load_matrix_fixture("dlsys_lecture12_s4_outer_product.txt")
    got = gemm(A, B)
    assert got.shape == C.shape
    assert np.array_equal(got, C), (got, C)


def pin_identity(gemm):
    rng = np.random.default_rng(11)
    A = rng.random((7, 5), dtype=np.float32) * 2 - 1
    assert np.array_equal(gemm(A, np.eye(5, dtype=np.float32)), A.astype(np.float64))
    assert np.array_equal(gemm(np.eye(7, dtype=np.float32), A), A.astype(np.float64))


def pin_permutation(gemm):
    rng = np.random.default_rng(12)
    perm = rng.permutation(6)
    P = np.zeros((6, 6), dtype=np.float32)
    P[np.arange(6), perm] = 1.0          # (P X)[r] = X[perm[r]]
    X = rng.standard_normal((6, 4), dtype=np.float32)
    assert np.array_equal(gemm(P, X), X[perm].astype(np.float64))
    Y = rng.standard_normal((3, 6), dtype=np.float32)
    inv = np.argsort(perm)               # (Y P)[:, c] = Y[:, inv[c]]
    assert np.array_equal(gemm(Y, P), Y[:, inv].astype(np.float64))


def pin_all_ones(gemm):
    for (M, N, K) in [(1, 1, 1), (3, 5, 7), (9, 2, 300), (4, 4, 0)]:
        C = gemm(np.ones((M, K), np.float32), np.ones((K, N), np.float32))
        assert C.shape == (M, N)
        assert np.all(C == K), (M, N, K)


def pin_rank1_integer(gemm):
    rng = np.random.default_rng(13)
    M, N, K = 5, 6, 9
    u = rng.integers(-5, 6, M)
    v = rng.integers(-5, 6, N)
    w = rng.integers(-5, 6, K)
    x = rng.integers(-5, 6, K)
    A = np.outer(u, w).astype(np.float32)   # A[i][k] = u_i w_k
    B = np.outer(x, v).astype(np.float32)   # B[k][j] = x_k v_j
    want = (np.outer(u, v) * int(np.dot(w, x))).astype(np.float64)
    assert np.array_equal(gemm(A, B), want)


def _fraction_product(A, B):
    M, K = A.shape
    N = B.shape[1]
    return [[sum((Fraction(float(A[i, k])) * Fraction(float(B[k, j])) for k in range(K)),
                 Fraction(0)) for j in range(N)] for i in range(M)]


def pin_bruteforce_exact(gemm):
    rng = np.random.default_rng(14)
    for M, N, K in itertools.product(range(1, 5), repeat=3):
        A = (rng.integers(-16, 17, (M, K)) / 8).astype(np.float32)
        B = (rng.integers(-16, 17, (K, N)) / 8).astype(np.float32)
        want = _fraction_product(A, B)
        got = gemm(A, B)
        for i in range(M):
            for j in range(N):
                assert Fraction(float(got[i, j])) == want[i][j], (M, N, K, i, j)


def pin_library_fp64(gemm):
    rng = np.random.default_rng(15)
    A = rng.random((37, 129), dtype=np.float32) * 2 - 1
    B = rng.random((129, 53), dtype=np.float32) * 2 - 1
    want = A.astype(np.float64) @ B.astype(np.float64)
    got = gemm(A, B)
    # Both are FP64 sums of exact products; only their order differs.
    assert np.max(np.abs(got - want)) <= 129 * 2.0 ** -52 * 129


def pin_freivalds(gemm):
    rng = np.random.default_rng(16)
    A = rng.standard_normal((300, 500), dtype=np.float32)
    B = rng.standard_normal((500, 200), dtype=np.float32)
    x = rng.standard_normal(200)
    C = gemm(A, B)
    lhs = C @ x
    rhs = A.astype(np.float64) @ (B.astype(np.float64) @ x)
    assert np.max(np.abs(lhs - rhs)) <= 1e-9 * np.max(np.abs(rhs))


def pin_padded_leading_dims(gemm):
    rng = np.random.default_rng(17)
    A = rng.random((6, 5), dtype=np.float32)
    B = rng.random((5, 7), dtype=np.float32)
    Ap = np.full((6, 9), np.nan, np.float32)
    Ap[:, :5] = A
    Bp = np.full((5, 12), np.nan, np.float32)
    Bp[:, :7] = B
    got = gemm(Ap[:, :5], Bp[:, :7])
    assert np.all(np.isfinite(got))
    assert np.array_equal(got, gemm(A, B))


def pin_integer_exact(gemm):
    rng = np.random.default_rng(18)
    A = rng.integers(-4, 5, (64, 96))
    B = rng.integers(-4, 5, (96, 48))
    want = (A @ B).astype(np.float64)
    assert np.array_equal(gemm(A.astype(np.float32), B.astype(np.float32)), want)


ALL_GEMM_PINS = [pin_worked_example, pin_identity, pin_permutation, pin_all_ones,
                 pin_rank1_integer, pin_bruteforce_exact, pin_library_fp64,
                 pin_freivalds, pin_padded_leading_dims, pin_integer_exact]


def pin_entries_exact(entries):
    """Sampled entries against exact rational dot products (shapes up to 4 x 4 x 5)."""
    rng = np.random.default_rng(19)
    for M, N, K in [(1, 1, 1), (3, 4, 5), (4, 2, 3), (2, 3, 1)]:
        A = (rng.integers(-16, 17, (M, K)) / 8).astype(np.float32)
        B = (rng.integers(-16, 17, (K, N)) / 8).astype(np.float32)
        want = _fraction_product(A, B)
        ii, jj = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
        got = entries(A, B, ii.ravel(), jj.ravel())
        for t, (i, j) in enumerate(zip(ii.ravel(), jj.ravel())):
            assert Fraction(float(got[t])) == want[i][j], (M, N, K, i, j)


def pin_entries_padded(entries):
    rng = np.random.default_rng(20)
    Ap = np.full((5, 8), np.nan, np.float32)
    Ap[:, :6] = rng.integers(-4, 5, (5, 6))
    Bp = np.full((6, 9), np.nan, np.float32)
    Bp[:, :3] = rng.integers(-4, 5, (6, 3))
    A, B = Ap[:, :6], Bp[:, :3]
    want = A.astype(np.int64) @ B.astype(np.int64)
    ii = np.array([0, 4, 2, 3]); jj = np.array([2, 0, 1, 2])
    got = entries(A, B, ii, jj)
    assert np.array_equal(got, want[ii, jj].astype(np.float64))


ALL_ENTRY_PINS = [pin_entries_exact, pin_entries_padded]
