"""gemm_f32_tc3_noalloc: the tensor-core product without any device allocation.

Callers that cannot allocate device memory where they call the library (a
memory manager that owns the device budget, a latency-critical path that
cannot take cudaMalloc's implicit synchronisation, a context where the CUDA
allocation API may not be used) call this entry point instead of gemm_f32_tc3:
it keeps the split operands in a fixed 64 MiB scratch array inside the library.

The test calls it through the C ABI twice in a row, with different shapes and
inputs, and compares each result with gemm_f32_tc3 given a caller-allocated
workspace, within the tolerances the other GPU tests use (normwise 1e-5,
elementwise 1e-4 sqrt(K)); it also checks that a product too large for the
scratch is refused.  The file is named so that pytest collects it last; it
depends on no state left by other tests.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import parity  # noqa: E402
from tiled_matrix_multiply_gb300 import _abi, build  # noqa: E402

pytestmark = pytest.mark.gpu


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
    return C


def _no_alloc(lib, A, B, stream):
    M, K = A.shape
    N = B.shape[1]
    C = torch.full((M, N), float("nan"), device="cuda")
    rc = lib.gemm_f32_tc3_noalloc(M, N, K, A.data_ptr(), K, B.data_ptr(), N, C.data_ptr(), N,
                                  stream)
    assert rc == _abi.TMM_OK, _abi.last_error()
    return C


def test_no_alloc_matches_workspace_entry_point_on_two_calls(lib):
    stream = torch.cuda.current_stream().cuda_stream
    g = torch.Generator(device="cuda").manual_seed(60)
    for (M, N, K) in [(1024, 1024, 1024), (700, 900, 1500)]:
        A = torch.randn(M, K, device="cuda", generator=g)
        B = torch.randn(K, N, device="cuda", generator=g)
        got = _no_alloc(lib, A, B, stream)
        want = _with_workspace(lib, A, B, stream)
        torch.cuda.synchronize()
        assert lib.tmm_check_device(stream) == _abi.TMM_OK, _abi.last_error()
        parity.assert_close(got.cpu().numpy(), want.cpu().numpy().astype(np.float64), K,
                            f"no-alloc vs workspace {M}x{N}x{K}")


def test_no_alloc_refuses_products_beyond_its_scratch(lib):
    M = N = K = 4096        # needs 256 MiB of split operands, the scratch holds 64 MiB
    assert lib.gemm_f32_tc3_workspace_size(M, N, K) > 64 << 20
    A = torch.empty(1, device="cuda")
    C = torch.empty(1, device="cuda")
    # Pointer values only reach the size check (no kernel runs): the call must fail first.
    rc = lib.gemm_f32_tc3_noalloc(M, N, K, A.data_ptr(), K, A.data_ptr() + (1 << 30), N,
                                  C.data_ptr() + (1 << 31), N,
                                  torch.cuda.current_stream().cuda_stream)
    assert rc == _abi.TMM_ERR_INVALID_ARG
    assert "scratch" in _abi.last_error()
