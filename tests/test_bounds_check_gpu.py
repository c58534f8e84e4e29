"""Parity subsets through the bounds-checked debug build of the library.

The library compiled with -DTMM_BOUNDS_CHECK checks every global address of
the product kernels against its matrix's stored extent (rows, columns, never a
row gap) and every shared-memory offset against its slab; a failed check skips
the access and makes tmm_check_device return TMM_ERR_BOUNDS.  These tests run
the shapes most likely to expose an index error -- tile edges, padded and
unaligned leading dimensions and base pointers, the ragged workload, the
transposed layouts, and the small problems split over K -- through every
product entry point of that build, and require both the usual parity with the
oracle and a clean status (TMM_OK).  The checked library is its own file, so
its device state is separate from the normal build's.
"""
import itertools

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import parity  # noqa: E402
from tiled_matrix_multiply_gb300 import _abi, build, inputs  # noqa: E402

pytestmark = pytest.mark.gpu

ENTRIES = ("gemm_f32", "gemm_f32_naive", "gemm_f32_tc3")


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return _abi.load(build.build_checked())


def _run(lib, entry, A, B, **k):
    from gpu_util import run_entry
    return run_entry(entry, A, B, lib=lib, **k)


@pytest.mark.parametrize("entry", ENTRIES)
def test_tile_edges_integer_exact(lib, entry):
    rng = np.random.default_rng(70)
    for M, N, K in itertools.product([1, 127, 129, 257], [1, 3, 129, 131], [1, 17, 33]):
        A = rng.integers(-4, 5, (M, K)).astype(np.float32)
        B = rng.integers(-4, 5, (K, N)).astype(np.float32)
        parity.assert_bit_exact(_run(lib, entry, A, B), oracle.gemm(A, B), f"{entry} {M}x{N}x{K}")


LAYOUTS = [(0, 0, 0, 0, 0, 0), (4, 8, 12, 4, 8, 4), (1, 3, 5, 0, 0, 0), (0, 0, 0, 1, 0, 0),
           (0, 0, 0, 0, 3, 0), (0, 0, 0, 0, 0, 2), (5, 7, 9, 3, 1, 1)]


@pytest.mark.parametrize("entry", ENTRIES)
@pytest.mark.parametrize("layout", LAYOUTS)
def test_padded_and_unaligned_operands(lib, entry, layout):
    pa, pb, pc, oa, ob, oc = layout
    M, N, K = 131, 257, 77
    rng = np.random.default_rng(71)
    A = rng.integers(-4, 5, (M, K)).astype(np.float32)
    B = rng.integers(-4, 5, (K, N)).astype(np.float32)
    C = _run(lib, entry, A, B, lda=K + pa, ldb=N + pb, ldc=N + pc, a_off=oa, b_off=ob, c_off=oc)
    parity.assert_bit_exact(C, oracle.gemm(A, B), f"{entry} {layout}")


@pytest.mark.parametrize("entry", ["gemm_f32", "gemm_f32_tc3"])
def test_ragged_workload(lib, entry):
    w = inputs.WORKLOADS["ragged4000x3001x2047"]
    A, B = inputs.workload_operands(w)
    C = _run(lib, entry, A, B, check_canaries=False)
    parity.assert_close(C, oracle.gemm(A, B), w.K, f"{entry} ragged")


def test_ragged_naive(lib):
    rng = np.random.default_rng(72)
    A = rng.random((300, 1001), dtype=np.float32) * 2 - 1
    B = rng.random((1001, 257), dtype=np.float32) * 2 - 1
    parity.assert_close(_run(lib, "gemm_f32_naive", A, B), oracle.gemm(A, B), 1001, "naive")


@pytest.mark.parametrize("entry", ["gemm_f32_ex", "gemm_f32_tc3_ex"])
@pytest.mark.parametrize("trans", [(1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("shape", [(300, 257, 129), (1024, 1024, 256), (301, 1003, 517)])
def test_transposed_layouts(lib, entry, trans, shape):
    # (301, 1003, 517): A stored K x M and B stored K x N with rows off 16-byte
    # boundaries, restaged (re-pitched) before the product; B stored N x K is
    # restaged (transposed) in every shape.
    M, N, K = shape
    rng = np.random.default_rng(73)
    A = rng.integers(-4, 5, (M, K)).astype(np.float32)
    B = rng.integers(-4, 5, (K, N)).astype(np.float32)
    As = np.ascontiguousarray(A.T) if trans[0] else A
    Bs = np.ascontiguousarray(B.T) if trans[1] else B
    C = _run(lib, entry, As, Bs, trans=trans)
    parity.assert_bit_exact(C, oracle.gemm(A, B), f"{entry} {trans} {shape}")


@pytest.mark.parametrize("entry", ["gemm_f32", "gemm_f32_tc3"])
@pytest.mark.parametrize("shape", [(1024, 1024, 1024), (37, 1000, 2000), (2600, 2700, 1001)])
def test_split_k_schedules(lib, entry, shape):
    M, N, K = shape
    rng = np.random.default_rng(74)
    A = rng.integers(-4, 5, (M, K)).astype(np.float32)
    B = rng.integers(-4, 5, (K, N)).astype(np.float32)
    C = _run(lib, entry, A, B, check_canaries=False)
    parity.assert_bit_exact(C, oracle.gemm(A, B), f"{entry} {shape}")
