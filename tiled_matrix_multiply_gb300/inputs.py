"""Seeded synthetic operands for the FP32 product C = A x B.

This module only draws random numbers: it holds none of the product's
arithmetic, and it is the one piece of code that both the CUDA path's tests
and the CPU oracle's tests use.

Recipe (NumPy ``default_rng``, PCG64; A is drawn first, then B, from one
generator):

* ``uniform``: ``rng.random(shape, float32) * 2 - 1``, exactly in [-1, 1);
* ``normal``:  ``rng.standard_normal(shape, float32)``;
* ``int4``:    integers drawn uniformly from {-4, ..., 4}, stored as float32,
  from a separate generator seeded ``[seed, 1]``.  With |a|, |b| <= 4 every
  partial sum of a K-term product is an integer of magnitude <= 16 K < 2^24,
  so any FP32 summation order gives the exact result.

The workloads (shapes, seeds, distributions) are the matrix sizes the tiling
pages reason about -- square 4096^3 as the running example of "Tiling
Hierarchy on GPUs" and "Tiling Strategies" section 2, N = 1024 as in the
counting table of "CMU DLSys Lecture 12" section 5 -- together with ragged
and rectangular shapes that exercise tile tails and aspect ratios.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    dist: str
    seed: int

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    def describe(self) -> str:
        d = {"uniform": "uniform[-1,1)", "normal": "standard normal",
             "int4": "integers in {-4..4}"}[self.dist]
        return (f"FP32 GEMM M={self.M} N={self.N} K={self.K} row-major, "
                f"A and B i.i.d. {d} from seed {self.seed}")


#: The parity and benchmark workloads.  ``square4096`` is the headline.
WORKLOADS = {
    "square256": Workload("square256", 256, 256, 256, "uniform", 0),
    "square256_int": Workload("square256_int", 256, 256, 256, "int4", 0),
    "square1024": Workload("square1024", 1024, 1024, 1024, "uniform", 1),
    "square4096": Workload("square4096", 4096, 4096, 4096, "normal", 2),
    "ragged4000x3001x2047": Workload("ragged4000x3001x2047", 4000, 3001, 2047, "uniform", 3),
    "rect8192x8192x1024": Workload("rect8192x8192x1024", 8192, 8192, 1024, "uniform", 4),
    "rect16384x1024x4096": Workload("rect16384x1024x4096", 16384, 1024, 4096, "uniform", 4),
    "rect1024x16384x4096": Workload("rect1024x16384x4096", 1024, 16384, 4096, "uniform", 4),
    "square8192": Workload("square8192", 8192, 8192, 8192, "uniform", 4),
}

HEADLINE = "square4096"


def draw(rng: np.random.Generator, shape, dist: str) -> np.ndarray:
    """One float32 array of the given shape and distribution."""
    if dist == "uniform":
        return rng.random(shape, dtype=np.float32) * np.float32(2) - np.float32(1)
    if dist == "normal":
        return rng.standard_normal(shape, dtype=np.float32)
    if dist == "int4":
        return rng.integers(-4, 5, size=shape, dtype=np.int32).astype(np.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def generator(seed: int, dist: str) -> np.random.Generator:
    """The generator a workload draws from (integer variants use seed [seed, 1])."""
    return np.random.default_rng([seed, 1] if dist == "int4" else seed)


def make_operands(M: int, N: int, K: int, dist: str, seed: int,
                  lda: int | None = None, ldb: int | None = None):
    """Draw A (M x K) then B (K x N).

    With ``lda > K`` (``ldb > N``) the operand is a view into a wider row-major
    buffer whose padding columns hold NaN, so a kernel that reads past a row's
    end poisons its result.
    """
    rng = generator(seed, dist)
    A = draw(rng, (M, K), dist)
    B = draw(rng, (K, N), dist)
    if lda is not None and lda != K:
        A = _pad(A, lda)
    if ldb is not None and ldb != N:
        B = _pad(B, ldb)
    return A, B


def _pad(x: np.ndarray, ld: int) -> np.ndarray:
    rows, cols = x.shape
    if ld < cols:
        raise ValueError("leading dimension shorter than the row")
    buf = np.full((rows, ld), np.nan, dtype=np.float32)
    buf[:, :cols] = x
    return buf[:, :cols]


def workload_operands(w: Workload | str):
    """Operands of a named workload (compact row-major: lda = K, ldb = N)."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    return make_operands(w.M, w.N, w.K, w.dist, w.seed)
