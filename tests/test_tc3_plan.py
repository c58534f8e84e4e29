"""The tensor-core path's work list, on the host (no GPU): tmm_testing_tc3_plan.

gemm_f32_tc3 lists whole tiles first and then the K-parts of the tiles it
splits: the last, partly filled round of a large product in two halves, or
every tile of a small product in up to four parts of at least two 256-value
chunks.  A part waits only for the parts listed before it, and all parts run
in one round beside their partners; these tests check that the list keeps
those properties (whole tiles a multiple of the resident slots whenever parts
exist, the parts of a round no more than the slots, parts on chunk
boundaries, the parts within the flag capacity) over a grid of shapes, and
the choices the measurements picked.
"""
import ctypes
import itertools

import pytest

from tiled_matrix_multiply_gb300 import _abi, build

SLICES_PER_CHUNK = 16          # 256 values of K in slices of 16
MAX_UNITS = {1: 512, 0: 1024}  # split units a call's flags hold (pairs, single blocks)


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _abi.load()


def plan(lib, M, N, K, pairs=1, slots=76):
    out = (ctypes.c_int64 * 6)()
    rc = lib.tmm_testing_tc3_plan(M, N, K, pairs, slots, out)
    assert rc == _abi.TMM_OK, _abi.last_error()
    return dict(zip(("tiles", "items", "dp_tiles", "parts", "chunks", "slices"), list(out)))


SHAPES = list(itertools.product([1, 128, 129, 256, 1000, 2048, 4000, 4096, 8192, 16384],
                                [1, 256, 257, 1000, 3001, 4096, 16384],
                                [1, 31, 32, 256, 257, 512, 1024, 2047, 4096, 8192]))


@pytest.mark.parametrize("pairs,slots", [(1, 76), (0, 152), (1, 40)])
def test_work_list_keeps_its_invariants(lib, pairs, slots):
    for M, N, K in SHAPES:
        p = plan(lib, M, N, K, pairs, slots)
        bm, bn = (256, 256) if pairs else (128, 256)
        tiles = -(-M // bm) * -(-N // bn)
        slices = -(-K // 32) * 32 // 16
        assert p["tiles"] == tiles and p["slices"] == slices
        assert p["chunks"] == -(-slices // SLICES_PER_CHUNK)
        parts, dp = p["parts"], p["dp_tiles"]
        assert p["items"] == dp + parts * (tiles - dp)
        if parts == 1:
            assert dp == tiles
            continue
        units = parts * (tiles - dp)
        assert 2 <= parts <= 4 and units <= MAX_UNITS[pairs]
        assert p["chunks"] >= 2 * parts if dp == 0 else p["chunks"] >= 2
        assert units <= slots, "all parts in one round"
        assert dp % slots == 0, "whole tiles fill whole rounds before the parts"
        if dp > 0:
            assert parts == 2 and tiles - dp == tiles % slots


def test_choices_at_the_measured_sizes(lib):
    # 4096^3 on pairs: 256 tiles over 76 pairs, the last 28 tiles in halves.
    p = plan(lib, 4096, 4096, 4096)
    assert (p["tiles"], p["dp_tiles"], p["parts"], p["items"]) == (256, 228, 2, 284)
    # 8192^3: 1024 tiles, 36 left over -> halves (72 parts in the last round).
    p = plan(lib, 8192, 8192, 8192)
    assert (p["dp_tiles"], p["parts"]) == (988, 2)
    # 1024^3: 16 tiles of four chunks -> two parts of two chunks each.
    p = plan(lib, 1024, 1024, 1024)
    assert (p["tiles"], p["parts"], p["items"], p["chunks"]) == (16, 2, 32, 4)
    # 256^3: one tile of one chunk -> not split.
    p = plan(lib, 256, 256, 256)
    assert (p["tiles"], p["parts"], p["items"]) == (1, 1, 1)
    # A last round more than half full is not split (208 tiles: 56 left, 112 > 76).
    p = plan(lib, 3328, 4096, 4096)
    assert p["tiles"] == 13 * 16 and p["parts"] == 1


def test_plan_rejects_bad_arguments(lib):
    out = (ctypes.c_int64 * 6)()
    for args in [(0, 1, 1), (1, 0, 1), (1, 1, 0), (1 << 31, 1, 1)]:
        assert lib.tmm_testing_tc3_plan(*args, 1, 76, out) == _abi.TMM_ERR_INVALID_ARG
    assert lib.tmm_testing_tc3_plan(1, 1, 1, 1, 0, out) == _abi.TMM_ERR_INVALID_ARG
    assert lib.tmm_testing_tc3_plan(1, 1, 1, 1, 76, None) == _abi.TMM_ERR_INVALID_ARG
