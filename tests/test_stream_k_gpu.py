"""GPU tests of the persistent stream-K schedule of gemm_f32 and of its bounded waits.

Shapes are chosen so that the tile count (64 x 256 tiles) leaves a partial
last wave on a 152-SM GB300 with two resident blocks per SM, which sends
gemm_f32 down the persistent stream-K path: split tiles are summed by two
blocks that meet through a flag.  The small shapes have fewer tiles than
resident blocks: every tile is split over several consecutive blocks, each
adding the next block's running sum (a chain of up to five), or -- with few
tiles, or C without 16-byte rows -- every block takes an equal share and the
blocks sharing a tile reduce it together from their partial sums (up to one
contributor per resident block).  The timeout
tests make one block skip its flag (a testing hook of the library) with a
2 ms limit: the waiting block must give up, the library must report
TMM_ERR_DEVICE_TIMEOUT through tmm_check_device, and the next call must be
correct again.  No kernel faults or hangs: every wait is bounded and the
kernel always runs to completion.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import parity  # noqa: E402
from tiled_matrix_multiply_gb300 import _abi, build  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    _abi.load()


def _run(*a, **k):
    from gpu_util import run_entry
    return run_entry(*a, **k)


# (M, N, K): all tiles split (400 tiles); data-parallel waves plus split tiles
# (1122 tiles); ragged K; ragged M and N with odd leading dimensions.  Then
# fewer tiles than resident blocks, chained: 64 tiles in four unequal parts
# each; 64 tiles of 187 slices; 200 tiles (shares of two thirds of a tile).
# Reduced together: one tile over 64 blocks; single rows and columns; 4
# tiles of 125 slices; 4 tiles of 16 slices; 16 tiles of 256 slices (19
# contributors each); C rows of 1023 floats (no 16-byte stores); one tile of
# 4096 slices over all 304 resident blocks.
SK_SHAPES = [(2560, 2560, 1000), (4224, 4224, 256), (2600, 2700, 1001), (3001, 2999, 777),
             (1024, 1024, 1024), (1000, 1000, 2990), (64, 256, 4096), (1, 1, 1024),
             (37, 1000, 2000), (256, 256, 256), (1280, 2560, 1024), (512, 512, 4096),
             (1024, 1023, 1024), (64, 256, 65536)]


@pytest.mark.parametrize("shape", SK_SHAPES)
def test_stream_k_shapes_float(shape):
    M, N, K = shape
    rng = np.random.default_rng(40)
    A = rng.random((M, K), dtype=np.float32) * 2 - 1
    B = rng.random((K, N), dtype=np.float32) * 2 - 1
    C = _run("gemm_f32", A, B, check_canaries=False)
    ref = oracle.gemm(A, B)
    if M * N < 16:   # a single output: its own error bound, not a normwise ratio
        parity.assert_close_few_outputs(C, A, B, f"stream-K {shape}")
        assert np.max(np.abs(C - ref)) <= parity.elementwise_tol(K)
    else:
        parity.assert_close(C, ref, K, f"stream-K {shape}")
    assert _abi.load().tmm_check_device(torch.cuda.current_stream().cuda_stream) == _abi.TMM_OK


@pytest.mark.parametrize("shape", SK_SHAPES)
def test_stream_k_shapes_integer_exact_and_deterministic(shape):
    M, N, K = shape
    rng = np.random.default_rng(41)
    A = rng.integers(-4, 5, (M, K)).astype(np.float32)
    B = rng.integers(-4, 5, (K, N)).astype(np.float32)
    C1 = _run("gemm_f32", A, B, check_canaries=False)
    parity.assert_bit_exact(C1, oracle.gemm(A, B), f"stream-K {shape}")
    Af = rng.standard_normal((M, K), dtype=np.float32)
    Bf = rng.standard_normal((K, N), dtype=np.float32)
    D1 = _run("gemm_f32", Af, Bf, check_canaries=False)
    D2 = _run("gemm_f32", Af, Bf, check_canaries=False)
    assert np.array_equal(D1.view(np.uint32), D2.view(np.uint32))


@pytest.mark.parametrize("shape", [(2560, 2560, 256), (1024, 1024, 1024), (512, 512, 4096)])
def test_stream_k_wait_timeout_is_reported_and_recovers(shape):
    # 2560^2 x 256: block 1 holds the tail of a two-block tile.  1024^3: block 1
    # holds the second of four shares of tile 0, so block 0 waits for it.
    # 512^2 x 4096 (reduced together): block 1 never raises the flags of its
    # partial sums, so every block sharing its tiles waits for them.
    lib = _abi.load()
    stream = torch.cuda.current_stream().cuda_stream
    M, N, K = shape
    rng = np.random.default_rng(42)
    A = rng.integers(-4, 5, (M, K)).astype(np.float32)
    B = rng.integers(-4, 5, (K, N)).astype(np.float32)
    assert lib.tmm_check_device(stream) == _abi.TMM_OK      # clean slate
    try:
        assert lib.tmm_testing_set_wait_hooks(1, 2_000_000) == _abi.TMM_OK
        _run("gemm_f32", A, B, check_canaries=False, check_status=False)
        rc = lib.tmm_check_device(stream)
        assert rc == _abi.TMM_ERR_DEVICE_TIMEOUT, rc
        assert "ran out of time" in _abi.last_error()
    finally:
        lib.tmm_testing_set_wait_hooks(-1, 0)
    # The status was cleared by the check and the context is usable.
    assert lib.tmm_check_device(stream) == _abi.TMM_OK
    C = _run("gemm_f32", A, B, check_canaries=False)
    parity.assert_bit_exact(C, oracle.gemm(A, B), "after timeout")
    assert lib.tmm_check_device(stream) == _abi.TMM_OK


@pytest.mark.parametrize("transa", [0, 1])
def test_tma_wait_timeout_is_reported_and_recovers(transa):
    # 1216 x 4096 tiles exactly into 304 blocks of 64 x 256 (two per SM): one
    # plain wave, no split tiles, so only the TMA wait of block 1 -- armed for
    # 16 bytes its copy never brings -- can run out of time.  transa = 1 stages
    # both operands by TMA (A stored K x M), transa = 0 only B.
    lib = _abi.load()
    stream = torch.cuda.current_stream().cuda_stream
    M, N, K = 1216, 4096, 512
    rng = np.random.default_rng(43)
    A = rng.integers(-4, 5, (M, K)).astype(np.float32)
    B = rng.integers(-4, 5, (K, N)).astype(np.float32)
    dA = torch.from_numpy(np.ascontiguousarray(A.T) if transa else A).cuda()
    dB = torch.from_numpy(B).cuda()
    lda = M if transa else K

    def call():
        C = torch.full((M, N), float("nan"), device="cuda")
        rc = lib.gemm_f32_ex(transa, 0, M, N, K, dA.data_ptr(), lda, dB.data_ptr(), N,
                             C.data_ptr(), N, stream)
        assert rc == _abi.TMM_OK, _abi.last_error()
        return C

    assert lib.tmm_check_device(stream) == _abi.TMM_OK      # clean slate
    try:
        assert lib.tmm_testing_set_wait_hooks(1, 2_000_000) == _abi.TMM_OK
        call()
        rc = lib.tmm_check_device(stream)
        assert rc == _abi.TMM_ERR_DEVICE_TIMEOUT, rc
    finally:
        lib.tmm_testing_set_wait_hooks(-1, 0)
    assert lib.tmm_check_device(stream) == _abi.TMM_OK
    C = call()
    torch.cuda.synchronize()
    parity.assert_bit_exact(C.cpu().numpy(), oracle.gemm(A, B), f"after TMA timeout, transa={transa}")
    assert lib.tmm_check_device(stream) == _abi.TMM_OK
