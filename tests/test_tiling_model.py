"""The analytical tiling counts against the numbers the pages print (CPU only)."""
from fractions import Fraction

import pytest

from tiled_matrix_multiply_gb300 import tiling_model as T

GiB = 1 << 30
MiB = 1 << 20


def test_fma_and_flop_counts_running_example():
    # "Tiling Hierarchy on GPUs", "Inner Product": M N K FMAs, 2 M N K FLOPs.
    assert T.fma_count(4096, 4096, 4096) == 4096 ** 3
    assert T.flops(4096, 4096, 4096) == 2 * 4096 ** 3


def test_single_fma_and_inner_product_intensity():
    # "Arithmetic Intensity": 2 FLOPs / 8 bytes = 0.25 FLOP/B; inner product 0.5 FMA/load.
    assert 2 / (2 * T.FP32_BYTES) == 0.25
    assert T.inner_product_intensity() == 0.5


def test_outer_product_intensity_square_is_half_m():
    # "Outer Product": with M = N the intensity is 0.5 M FMAs per load.
    for m in (2, 8, 128, 4096):
        assert T.outer_product_intensity(m, m) == 0.5 * m
    # "Maximizing this requires M = N": for a fixed M + N the square split is best.
    assert T.outer_product_intensity(8, 8) > T.outer_product_intensity(4, 12)


def test_register_tiling_needs_8x8_and_80_or_96_registers():
    # "Register Tiling": 128 FMAs / 32 loaded values = 4 per load -> m = 8, 80 registers.
    req = T.required_intensity(128, 32)
    assert req == 4
    assert T.min_square_thread_tile(req) == 8
    assert T.thread_tile_registers(8, 8, prefetch=False) == 80
    # "Register prefetching": two operand sets, 96 registers.
    assert T.thread_tile_registers(8, 8, prefetch=True) == 96
    # "Reducing Overhead Slots": 8 x 16 needs 176, 16 x 16 needs 320 (> 255, spills).
    assert T.thread_tile_registers(8, 16, prefetch=True) == 176
    assert T.thread_tile_registers(16, 16, prefetch=True) == 320


def test_issue_slot_efficiency_traces():
    # "Eliminating Idle slots": 16 LDS + ~22 idle + 64 FFMA = ~102 cycles, eta ~ 63%.
    eta0 = T.issue_efficiency(64, 16, 22)
    assert round(eta0 * 100) == 63
    # "Register prefetching": 16 + 64 = 80 cycles, eta = 80%.
    assert T.issue_efficiency(64, 16, 0) == 0.8


def test_larger_thread_tile_raises_ceiling_by_about_four_points():
    # "Reducing Overhead Slots": 8 x 8 -> 8 x 16 raises the ceiling by only ~4%.
    gain = T.issue_ceiling(8, 16) - T.issue_ceiling(8, 8)
    assert T.issue_ceiling(8, 8) == 0.8
    assert 0.035 < gain < 0.045


def test_threads_per_cta_for_128x128_block():
    # 16,384 / 64 = 256 threads for 8 x 8; 16,384 / 128 = 128 threads for 8 x 16.
    assert T.threads_per_cta(128, 128, 8, 8) == 256
    assert T.threads_per_cta(128, 128, 8, 16) == 128


def test_dlsys_counting_table_n1024():
    # "CMU DLSys Lecture 12", section 5 table, N = 1024, L = 32, V = 4, S = 8.
    N, L, V = 1024, 32, 4
    assert T.q_naive(N, N, N) == 2_147_483_648
    assert T.q_naive(N, N, N) * T.FP32_BYTES == 8 * GiB
    assert T.q_input_to_reg(N, N, N, V, V) == 536_870_912          # register tile only
    assert T.q_input_to_reg(N, N, N, V, V) * T.FP32_BYTES == 2 * GiB
    assert T.q_global_to_shared(N, N, N, L, L) == 67_108_864       # two-level, global
    assert T.q_global_to_shared(N, N, N, L, L) * T.FP32_BYTES == 256 * MiB
    assert T.q_input_to_reg(N, N, N, V, V) == 536_870_912          # two-level, shared->reg
    # Output write: 4 MiB.
    assert N * N * T.FP32_BYTES == 4 * MiB


def test_dlsys_flop_per_byte():
    # Section 5: L/4 = 8 FLOP/B, 512/65 ~ 7.88 FLOP/B including the output write.
    assert T.two_level_flop_per_byte(1024, 32, with_output=False) == 8
    got = T.two_level_flop_per_byte(1024, 32, with_output=True)
    assert Fraction(got).limit_denominator(1000) == Fraction(512, 65)


def test_dlsys_block_and_stage_sizes():
    # Sections 5 and 6: 64 threads, 512 floats = 2 KiB per stage.
    assert T.block_threads(32, 4) == 64
    assert T.stage_floats(8, 32) == 512
    assert T.stage_floats(8, 32) * T.FP32_BYTES == 2048


def test_stage_depth_cancels():
    # The Q counts do not depend on S; only on the tile extents.
    a = T.q_global_to_shared(512, 256, 128, 64, 32)
    assert a == 512 * 256 * 128 // 32 + 512 * 256 * 128 // 64


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 4096), (4000, 3001, 2047)])
def test_compulsory_bytes(M, N, K):
    assert T.compulsory_bytes(M, N, K) == 4 * (M * K + K * N + M * N)
