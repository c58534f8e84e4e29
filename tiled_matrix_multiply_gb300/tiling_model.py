"""Analytical counts of the tiling hierarchy for C = A x B (host-side arithmetic only).

These are the logical counts the tiling pages reason with, generalised from
square N x N x N to M x N x K and from square tiles to BM x BN block tiles and
TM x TN thread tiles.  The benchmark uses them for the algorithmic work per
launch (FLOPs, compulsory bytes) and for the traffic a kernel's tiling predicts,
which ncu's L2 and DRAM counters are compared with.

Sources:
* "Tiling Hierarchy on GPUs": sections "Where the FLOPs come from" (FMA
  throughput per SM), "Inner Product"/"Outer Product" (arithmetic intensity),
  "Register Tiling" (required intensity, 8 x 8 thread tile, register budget),
  "Eliminating Idle slots"/"Register prefetching" (issue-slot efficiency),
  "Reducing Overhead Slots" (larger tiles, threads per CTA).
* "CMU DLSys Lecture 12: GPU Acceleration", sections 4 and 5 (Q counts,
  the N = 1024 table, FLOPs per byte).
"""
from __future__ import annotations

FP32_BYTES = 4


def fma_count(M: int, N: int, K: int) -> int:
    """M*N*K multiply-adds: K per output ("Inner Product")."""
    return M * N * K


def flops(M: int, N: int, K: int) -> int:
    """2*M*N*K: every FMA is one multiply and one add."""
    return 2 * fma_count(M, N, K)


def compulsory_bytes(M: int, N: int, K: int) -> int:
    """Each operand read once and C written once: 4 (MK + KN + MN) bytes."""
    return FP32_BYTES * (M * K + K * N + M * N)


def inner_product_intensity() -> float:
    """FMAs per loaded value when each output walks its own row and column: K / 2K."""
    return 0.5


def outer_product_intensity(m: int, n: int) -> float:
    """FMAs per loaded value of one rank-1 step over an m x n output: m n / (m + n).

    The page's formula is missing from the extracted text; this is the ratio its
    prose defines (m n FMAs from m + n loads), which gives 0.5 m at m = n.
    """
    return m * n / (m + n)


def required_intensity(fma_per_clk: int = 128, values_per_clk: int = 32) -> float:
    """FMAs each register-file load must feed to keep the FMA pipes busy."""
    return fma_per_clk / values_per_clk


def min_square_thread_tile(required: float) -> int:
    """Smallest m with m/2 >= required (m x m tile from 2m loads)."""
    m = 1
    while outer_product_intensity(m, m) < required:
        m += 1
    return m


def thread_tile_registers(m: int, n: int, prefetch: bool) -> int:
    """Accumulators plus one (or, with register prefetch, two) sets of m + n operands."""
    return m * n + (2 if prefetch else 1) * (m + n)


def issue_efficiency(useful: int, overhead: int, idle: int) -> float:
    """eta = slots that issued an FMA / all slots."""
    return useful / (useful + overhead + idle)


def issue_ceiling(m: int, n: int) -> float:
    """eta with no idle slots and one load slot per operand value: mn / (mn + m + n)."""
    return m * n / (m * n + m + n)


def threads_per_cta(bm: int, bn: int, m: int, n: int) -> int:
    """Outputs of the block tile divided by outputs per thread."""
    return (bm * bn) // (m * n)


def q_input_to_reg(M: int, N: int, K: int, tm: int, tn: int) -> int:
    """Operand values loaded into registers by thread tiles: M N K (1/tn + 1/tm).

    For square N and V x V thread tiles this is 2 N^3 / V.
    """
    return (M * N * K) // tn + (M * N * K) // tm


def q_global_to_shared(M: int, N: int, K: int, bm: int, bn: int) -> int:
    """Values staged from global into shared memory by BM x BN block tiles.

    Each block stages BM rows of A and BN columns of B over the whole K depth:
    M N K (1/BN + 1/BM); for square N and L x L blocks, 2 N^3 / L.  The stage
    depth S cancels.
    """
    return (M * N * K) // bn + (M * N * K) // bm


def q_naive(M: int, N: int, K: int) -> int:
    """One output per thread: two operand loads per FMA, 2 M N K values."""
    return 2 * M * N * K


def two_level_flop_per_byte(N: int, L: int, with_output: bool) -> float:
    """2 N^3 FLOPs over the global input bytes of L x L block tiling (plus the N^2 store)."""
    moved = q_global_to_shared(N, N, N, L, L) + (N * N if with_output else 0)
    return flops(N, N, N) / (FP32_BYTES * moved)


def block_threads(L: int, V: int) -> int:
    """(L/V)^2 threads for an L x L block of V x V thread tiles."""
    return (L // V) ** 2


def stage_floats(S: int, L: int) -> int:
    """Two S x L slabs per reduction stage."""
    return 2 * S * L


def predicted_l2_to_sm_bytes(M: int, N: int, K: int, bm: int, bn: int) -> int:
    """Bytes the block tiling pulls through L2 into shared memory, plus the C store."""
    return FP32_BYTES * (q_global_to_shared(M, N, K, bm, bn) + M * N)
