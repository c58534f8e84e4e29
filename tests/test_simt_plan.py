"""The tiled FFMA path's work split, on the host (no GPU): tmm_testing_simt_plan.

gemm_f32 divides an M x N x K product among its blocks in one of five ways --
whole tiles; whole tiles then a stream-K tail split over K (two blocks per
split tile); a small problem's tiles in unequal K-parts chained through C; a
small problem in equal shares chained through C; a small problem in equal
shares reduced together from partial-sum slots.  These tests check, over a
grid of shapes, the invariants each way relies on (every K-slice covered,
shares long enough, the flag region large enough, the grid no larger than the
resident blocks when the blocks wait on one another), and the choices between
them that the measurements picked.
"""
import ctypes
import itertools

import pytest

from tiled_matrix_multiply_gb300 import _abi, build

BM, BK = 64, 16
MAX_FLAG_BLOCKS = 4096   # flags of one call's region


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _abi.load()


def plan(lib, M, N, K, wide=0, vec_c=1, may_reduce=1, slots=304):
    out = (ctypes.c_int64 * 9)()
    rc = lib.tmm_testing_simt_plan(M, N, K, wide, vec_c, may_reduce, slots, out)
    assert rc == _abi.TMM_OK, _abi.last_error()
    keys = ("grid", "coop", "partial_slots", "dp_tiles", "sk_iters", "parts", "part_base",
            "part_step", "part_rem")
    return dict(zip(keys, list(out)))


def geometry(M, N, K, wide):
    BN = 512 if wide else 256
    tiles = -(-M // BM) * -(-N // BN)
    return tiles, -(-K // BK)


def part_lengths(p, S):
    """Slices of each unequal part (the kernel's part_begin, restated)."""
    P, base, step, rem = p["parts"], p["part_base"], p["part_step"], p["part_rem"]
    return [base + (P - 1 - q) * step + (rem if q == 0 else 0) for q in range(P)]


def check_invariants(p, M, N, K, wide, slots):
    tiles, S = geometry(M, N, K, wide)
    g = p["grid"]
    assert g >= 1
    if p["partial_slots"] > 0:                       # reduced together
        T = tiles * S
        assert p["partial_slots"] == 2 * g and 2 * g <= MAX_FLAG_BLOCKS
        assert g <= slots and tiles < slots and g * 8 >= tiles * 9
        assert p["sk_iters"] == T and p["dp_tiles"] == 0 and p["coop"] == 1
        assert T // g >= 4, "shares of at least four slices"
        assert -(-T // g) <= S, "at most two segments per share"
    elif p["coop"] and p["parts"] > 0:               # unequal parts, chained
        P = p["parts"]
        assert 2 <= P <= 4 and g == tiles * P and g <= slots
        lengths = part_lengths(p, S)
        assert sum(lengths) == S and min(lengths) >= 4
        assert all(a >= b for a, b in zip(lengths, lengths[1:])), "earlier parts no shorter"
        assert p["dp_tiles"] == 0 and p["sk_iters"] == tiles * S
    elif p["coop"] and tiles < slots:                # equal shares, chained
        T = tiles * S
        assert p["dp_tiles"] == 0 and p["sk_iters"] == T
        assert g <= slots and g * 8 >= tiles * 9 and g <= MAX_FLAG_BLOCKS
        assert T // g >= 3, "shares of about four slices or more"
    elif p["coop"]:                                  # stream-K tail
        assert g == slots and g <= MAX_FLAG_BLOCKS and tiles > slots
        sk_tiles = tiles - p["dp_tiles"]
        assert p["sk_iters"] == sk_tiles * S and p["dp_tiles"] % slots == 0
        assert p["sk_iters"] // g >= S, "every share at least one tile: two contributors"
        assert sk_tiles < 2 * slots
    else:                                            # whole tiles
        assert g == tiles and p["dp_tiles"] == tiles and p["sk_iters"] == 0


SHAPES = list(itertools.product([1, 63, 64, 65, 300, 1024, 2048, 4000, 4096, 8192],
                                [1, 255, 256, 257, 1000, 3001, 4096],
                                [1, 15, 16, 17, 64, 256, 1001, 2047, 4096, 65536]))


@pytest.mark.parametrize("wide,slots", [(0, 304), (1, 152), (0, 100)])
@pytest.mark.parametrize("vec_c", [0, 1])
def test_every_split_keeps_its_invariants(lib, wide, slots, vec_c):
    for M, N, K in SHAPES:
        for may_reduce in (0, 1):
            p = plan(lib, M, N, K, wide, vec_c, may_reduce, slots)
            check_invariants(p, M, N, K, wide, slots)
            if not may_reduce:
                assert p["partial_slots"] == 0


def test_headline_takes_a_stream_k_tail(lib):
    # 4096^3 on 64 x 512 tiles: 512 tiles over 152 blocks, 3.37 waves.
    p = plan(lib, 4096, 4096, 4096, wide=1, slots=152)
    assert p["coop"] == 1 and p["grid"] == 152 and p["partial_slots"] == 0
    assert p["dp_tiles"] == 304 and p["sk_iters"] == (512 - 304) * 256


def test_small_problems_choose_chains_or_reduction_as_measured(lib):
    # 1024^3: 64 tiles, four unequal parts each (256 of 304 slots busy) -> chains.
    p = plan(lib, 1024, 1024, 1024)
    assert p["parts"] == 4 and p["grid"] == 256 and p["partial_slots"] == 0
    assert part_lengths(p, 64) == [19, 16, 15, 14]
    # The same product with C rows off 16-byte boundaries -> reduced together.
    p = plan(lib, 1024, 1023, 1024, vec_c=0)
    assert p["partial_slots"] > 0 and p["grid"] == 304
    # Few tiles (16, at most 64 blocks chained) -> reduced together over 304 blocks.
    p = plan(lib, 512, 512, 4096)
    assert p["partial_slots"] == 2 * p["grid"] and p["grid"] == 304
    # ... unless the reduction's scratch is not available: chains then.
    p = plan(lib, 512, 512, 4096, may_reduce=0)
    assert p["partial_slots"] == 0 and p["parts"] == 4 and p["grid"] == 64
    # 2048^3: 256 tiles -> equal shares chained through C, one block per slot.
    p = plan(lib, 2048, 2048, 2048)
    assert p["partial_slots"] == 0 and p["parts"] == 0 and p["grid"] == 304
    # 256^3: 4 tiles of 16 slices -> 16 blocks of 4 slices, reduced together.
    p = plan(lib, 256, 256, 256)
    assert p["partial_slots"] == 32 and p["grid"] == 16


def test_products_too_short_to_split_run_whole_tiles(lib):
    for M, N, K in [(256, 256, 16), (64, 256, 63), (1, 1, 1)]:
        p = plan(lib, M, N, K)
        tiles, _ = geometry(M, N, K, 0)
        assert p["coop"] == 0 and p["grid"] == tiles


def test_plan_rejects_bad_arguments(lib):
    out = (ctypes.c_int64 * 9)()
    for args in [(0, 1, 1), (1, 0, 1), (1, 1, 0), (1 << 31, 1, 1)]:
        assert lib.tmm_testing_simt_plan(*args, 0, 1, 1, 304, out) == _abi.TMM_ERR_INVALID_ARG
    assert lib.tmm_testing_simt_plan(1, 1, 1, 0, 1, 1, 0, out) == _abi.TMM_ERR_INVALID_ARG
    assert lib.tmm_testing_simt_plan(1, 1, 1, 0, 1, 1, 304, None) == _abi.TMM_ERR_INVALID_ARG
