"""gemm_f32_tc3_noalloc: the tensor-core product without any device allocation.

Callers that cannot allocate device memory where they call the library (a
memory manager that owns the device budget, a latency-critical path that
cannot take cudaMalloc's implicit synchronisation, a context where the CUDA
allocation API may not be used) call this entry point instead of gemm_f32_tc3:
it keeps the split operands in a fixed 64 MiB scratch array inside the library.

Every result is checked against the CPU oracle (normwise 1e-5, elementwise
1e-4 sqrt(K); bit for bit on integer inputs) and must equal, bit for bit,
gemm_f32_tc3 given a caller-allocated workspace on the same inputs (both run
the same kernels; only the workspace's address differs).  The calls come two
in a row with different shapes, so the second runs on the scratch the first
left behind.  The size limit is checked at its edge: the largest accepted
product (its split operands fill the scratch exactly) and the next larger K,
refused with real device buffers.  The file is named so that pytest collects
it last; it depends on no state left by other tests.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import parity  # noqa: E402
from tiled_matrix_multiply_gb300 import _abi, build  # noqa: E402

pytestmark = pytest.mark.gpu

SCRATCH = 64 << 20      # TMM_TC3_NOALLOC_SCRATCH_BYTES


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return _abi.load()


def _with_workspace(lib, A, B, stream):
    M, K = A.shape
    N = B.shape[1]
    need = int(lib.gemm_f32_tc3_workspace_size(M, N, K))
    ws = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
    wptr = (ws.data_ptr() + 255) // 256 * 256
    C = torch.full((M, N), float("nan"), device="cuda")
    rc = lib.gemm_f32_tc3(M, N, K, A.data_ptr(), K, B.data_ptr(), N, C.data_ptr(), N, wptr, need,
                          stream)
    assert rc == _abi.TMM_OK, _abi.last_error()
    torch.cuda.synchronize()
    return C.cpu().numpy()


def _no_alloc(lib, A, B, stream):
    M, K = A.shape
    N = B.shape[1]
    C = torch.full((M, N), float("nan"), device="cuda")
    rc = lib.gemm_f32_tc3_noalloc(M, N, K, A.data_ptr(), K, B.data_ptr(), N, C.data_ptr(), N,
                                  stream)
    assert rc == _abi.TMM_OK, _abi.last_error()
    torch.cuda.synchronize()
    assert lib.tmm_check_device(stream) == _abi.TMM_OK, _abi.last_error()
    return C.cpu().numpy()


def _check(lib, A_h, B_h, exact, what):
    stream = torch.cuda.current_stream().cuda_stream
    A = torch.from_numpy(A_h).cuda()
    B = torch.from_numpy(B_h).cuda()
    got = _no_alloc(lib, A, B, stream)
    ref = oracle.gemm(A_h, B_h)
    if exact:
        parity.assert_bit_exact(got, ref, what)
    else:
        parity.assert_close(got, ref, A_h.shape[1], what)
    want = _with_workspace(lib, A, B, stream)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), \
        f"{what}: differs from gemm_f32_tc3 with a caller workspace"


def test_no_alloc_matches_oracle_and_workspace_entry_on_two_calls(lib):
    rng = np.random.default_rng(60)
    for (M, N, K) in [(1024, 1024, 1024), (700, 900, 1500)]:
        A = rng.standard_normal((M, K), dtype=np.float32)
        B = rng.standard_normal((K, N), dtype=np.float32)
        _check(lib, A, B, False, f"no-alloc {M}x{N}x{K}")


def test_no_alloc_integer_tile_edges_bit_exact(lib):
    # Shapes one past the 128 x 256 tile edges and the 32-wide K padding.
    rng = np.random.default_rng(61)
    for (M, N, K) in [(129, 257, 33), (257, 513, 1025), (1, 300, 31)]:
        A = rng.integers(-4, 5, (M, K)).astype(np.float32)
        B = rng.integers(-4, 5, (K, N)).astype(np.float32)
        _check(lib, A, B, True, f"no-alloc integer {M}x{N}x{K}")


def test_no_alloc_largest_accepted_product(lib):
    # 2048^3: A_hi, A_lo, B^T_hi and B^T_lo fill the 64 MiB scratch exactly.
    M = N = K = 2048
    assert lib.gemm_f32_tc3_workspace_size(M, N, K) == SCRATCH
    rng = np.random.default_rng(62)
    A = rng.random((M, K), dtype=np.float32) * 2 - 1
    B = rng.random((K, N), dtype=np.float32) * 2 - 1
    _check(lib, A, B, False, "no-alloc 2048^3 (scratch full)")


def test_no_alloc_refuses_the_next_larger_product(lib):
    # One more K (padded to 2080) needs more than the scratch: refused, and C
    # (real buffers of the stated shapes) is left as it was.
    M, N, K = 2048, 2048, 2049
    assert lib.gemm_f32_tc3_workspace_size(M, N, K) > SCRATCH
    A = torch.ones(M, K, device="cuda")
    B = torch.ones(K, N, device="cuda")
    C = torch.full((M, N), 7.0, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.gemm_f32_tc3_noalloc(M, N, K, A.data_ptr(), K, B.data_ptr(), N, C.data_ptr(), N,
                                  stream)
    assert rc == _abi.TMM_ERR_INVALID_ARG
    assert "scratch" in _abi.last_error()
    torch.cuda.synchronize()
    assert bool(torch.all(C == 7.0))
    assert lib.tmm_check_device(stream) == _abi.TMM_OK
