"""GPU parity of gemm_f32_tc3 (tcgen05 tensor cores, split-TF32 operands) against the oracle.

Same bars as the FFMA path: normwise error <= 1e-5 and elementwise error
<= 1e-4 sqrt(K) against the FP64-accumulated oracle for float inputs, bit-exact
results for integer-valued inputs (small integers are exact TF32 values and all
partial sums stay below 2^24).  Also covers the workspace contract.
"""
import itertools

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import parity  # noqa: E402
from tiled_matrix_multiply_gb300 import _abi, build, inputs  # noqa: E402

pytestmark = pytest.mark.gpu
ENTRY = "gemm_f32_tc3"


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    _abi.load()


def _run(*a, **k):
    from gpu_util import run_entry
    return run_entry(ENTRY, *a, **k)


@pytest.mark.parametrize("name", ["square256", "square256_int", "square1024",
                                  "ragged4000x3001x2047", "square4096"])
def test_workload_full_compare(name):
    w = inputs.WORKLOADS[name]
    A, B = inputs.workload_operands(w)
    C = _run(A, B, check_canaries=(w.M * w.N <= 1 << 22))
    ref = oracle.gemm(A, B)
    if w.dist == "int4":
        parity.assert_bit_exact(C, ref, name)
    else:
        parity.assert_close(C, ref, w.K, name)


@pytest.mark.parametrize("name", ["square1024", "ragged4000x3001x2047", "square4096"])
def test_workload_integer_variant_bit_exact(name):
    w = inputs.WORKLOADS[name]
    A, B = inputs.make_operands(w.M, w.N, w.K, "int4", w.seed)
    C = _run(A, B, check_canaries=False)
    parity.assert_bit_exact(C, oracle.gemm(A, B), name + " int4")


@pytest.mark.parametrize("name", ["rect8192x8192x1024", "rect16384x1024x4096",
                                  "rect1024x16384x4096", "square8192"])
def test_large_workload_sampled_and_freivalds(name):
    w = inputs.WORKLOADS[name]
    A, B = inputs.workload_operands(w)
    C = _run(A, B, check_canaries=False)
    rng = np.random.default_rng(50)
    ii = np.concatenate([rng.integers(0, w.M, 4096), [0, w.M - 1, 0, w.M - 1]])
    jj = np.concatenate([rng.integers(0, w.N, 4096), [0, 0, w.N - 1, w.N - 1]])
    ref = oracle.gemm_entries(A, B, ii, jj)
    got = C[ii, jj]
    assert np.max(np.abs(got - ref)) <= parity.elementwise_tol(w.K)
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= parity.NORMWISE_TOL
    x = rng.standard_normal(w.N)
    lhs = C.astype(np.float64) @ x
    rhs = A.astype(np.float64) @ (B.astype(np.float64) @ x)
    assert np.linalg.norm(lhs - rhs) / np.linalg.norm(rhs) <= parity.NORMWISE_TOL


def test_large_integer_exact_freivalds():
    w = inputs.WORKLOADS["square8192"]
    A, B = inputs.make_operands(w.M, w.N, w.K, "int4", w.seed)
    C = _run(A, B, check_canaries=False)
    rng = np.random.default_rng(51)
    ii = rng.integers(0, w.M, 2048)
    jj = rng.integers(0, w.N, 2048)
    parity.assert_bit_exact(C[ii, jj], oracle.gemm_entries(A, B, ii, jj), "square8192 int4")
    for _ in range(2):
        x = rng.integers(-1, 2, w.N).astype(np.float64)
        assert np.array_equal(C.astype(np.float64) @ x,
                              A.astype(np.float64) @ (B.astype(np.float64) @ x))


def test_tile_edge_shapes_integer_exact():
    rng = np.random.default_rng(52)
    for M, N, K in itertools.product([1, 127, 128, 129, 255], [1, 255, 256, 257, 300],
                                     [1, 15, 16, 17, 33, 127, 128, 129, 300]):
        A = rng.integers(-4, 5, (M, K)).astype(np.float32)
        B = rng.integers(-4, 5, (K, N)).astype(np.float32)
        parity.assert_bit_exact(_run(A, B), oracle.gemm(A, B), f"{M}x{N}x{K}")


def test_tiny_shapes_brute_force():
    rng = np.random.default_rng(53)
    for M, N, K in itertools.product(range(1, 7), repeat=3):
        A = rng.integers(-4, 5, (M, K)).astype(np.float32)
        B = rng.integers(-4, 5, (K, N)).astype(np.float32)
        parity.assert_bit_exact(_run(A, B), oracle.gemm(A, B), f"{M}x{N}x{K}")


@pytest.mark.parametrize("shape", [(129, 257, 1000), (300, 700, 129), (1, 1000, 4097)])
def test_float_odd_shapes(shape):
    M, N, K = shape
    rng = np.random.default_rng(54)
    A = rng.random((M, K), dtype=np.float32) * 2 - 1
    B = rng.random((K, N), dtype=np.float32) * 2 - 1
    parity.assert_close(_run(A, B), oracle.gemm(A, B), K, f"{shape}")


# Fewer tiles than half the slots: every tile is cut into K-parts of at least
# two 256-value chunks, each part adding the running sum of the parts before it.  Block
# pairs: 6 tiles in 4 parts; 16 tiles in 2 parts, the last chunk 32 values long.
# One-block kernel: 4 tiles of K = 2000 in 4 parts; one tile of K = 8192 in 4 parts.
PART_SHAPES = [(512, 768, 3000), (1024, 1024, 1050), (100, 1000, 2000), (64, 256, 8192)]


@pytest.mark.parametrize("shape", PART_SHAPES)
def test_k_parts_float_integer_and_deterministic(shape):
    M, N, K = shape
    rng = np.random.default_rng(59)
    A = rng.random((M, K), dtype=np.float32) * 2 - 1
    B = rng.random((K, N), dtype=np.float32) * 2 - 1
    C1 = _run(A, B)
    parity.assert_close(C1, oracle.gemm(A, B), K, f"parts {shape}")
    assert np.array_equal(C1.view(np.uint32), _run(A, B).view(np.uint32))
    Ai = rng.integers(-4, 5, (M, K)).astype(np.float32)
    Bi = rng.integers(-4, 5, (K, N)).astype(np.float32)
    parity.assert_bit_exact(_run(Ai, Bi), oracle.gemm(Ai, Bi), f"parts {shape} integer")


@pytest.mark.parametrize("layout", [(4, 8, 12, 4, 8, 4), (1, 3, 5, 0, 0, 0), (5, 7, 9, 3, 1, 1)])
def test_layouts(layout):
    pa, pb, pc, oa, ob, oc = layout
    M, N, K = 200, 300, 150
    rng = np.random.default_rng(55)
    A = rng.standard_normal((M, K), dtype=np.float32)
    B = rng.standard_normal((K, N), dtype=np.float32)
    C = _run(A, B, lda=K + pa, ldb=N + pb, ldc=N + pc, a_off=oa, b_off=ob, c_off=oc)
    parity.assert_close(C, oracle.gemm(A, B), K, f"layout {layout}")


def test_k_zero_and_repeat_determinism():
    from gpu_util import DevMatrix
    M, N = 33, 70
    dC = DevMatrix(None, M, N, N + 2, offset=3)
    lib = _abi.load()
    rc = lib.gemm_f32_tc3(M, N, 0, 0, 1, 0, N, dC.ptr, dC.ld, 0, 0,
                          torch.cuda.current_stream().cuda_stream)
    assert rc == _abi.TMM_OK
    torch.cuda.synchronize()
    assert np.all(dC.window() == 0) and dC.outside_window_untouched()
    rng = np.random.default_rng(56)
    A = rng.standard_normal((500, 700), dtype=np.float32)
    B = rng.standard_normal((700, 600), dtype=np.float32)
    C1, C2 = _run(A, B), _run(A, B)
    assert np.array_equal(C1.view(np.uint32), C2.view(np.uint32))


def test_workspace_contract():
    lib = _abi.load()
    s = torch.cuda.current_stream().cuda_stream
    M, N, K = 64, 64, 64
    A = torch.randn(M, K, device="cuda")
    B = torch.randn(K, N, device="cuda")
    C = torch.zeros(M, N, device="cuda")
    need = lib.gemm_f32_tc3_workspace_size(M, N, K)
    assert need == 4 * 64 * (2 * M + 2 * N)
    assert lib.gemm_f32_tc3_workspace_size(0, N, K) == 0
    ws = torch.empty(need + 512, dtype=torch.uint8, device="cuda")
    base = (ws.data_ptr() + 255) // 256 * 256
    args = (M, N, K, A.data_ptr(), K, B.data_ptr(), N, C.data_ptr(), N)
    assert lib.gemm_f32_tc3(*args, 0, need, s) == _abi.TMM_ERR_INVALID_ARG
    assert lib.gemm_f32_tc3(*args, base, need - 1, s) == _abi.TMM_ERR_INVALID_ARG
    assert lib.gemm_f32_tc3(*args, base + 16, need, s) == _abi.TMM_ERR_INVALID_ARG
    # Workspace overlapping C.
    assert lib.gemm_f32_tc3(M, N, K, A.data_ptr(), K, B.data_ptr(), N, base, N, base, need,
                            s) == _abi.TMM_ERR_ALIAS
    torch.cuda.synchronize()
    assert torch.count_nonzero(C) == 0          # nothing ran
    assert lib.gemm_f32_tc3(*args, base, need, s) == _abi.TMM_OK
    torch.cuda.synchronize()
    ref = oracle.gemm(A.cpu().numpy(), B.cpu().numpy())
    parity.assert_close(C.cpu().numpy(), ref, K, "after contract checks")


def test_python_binding_side_stream():
    import tiled_matrix_multiply_gb300 as tmm
    rng = np.random.default_rng(57)
    A = rng.standard_normal((300, 200), dtype=np.float32)
    B = rng.standard_normal((200, 400), dtype=np.float32)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        C = tmm.gemm_f32_tc3(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda())
        tmm.check_device(s)
    parity.assert_close(C.cpu().numpy(), oracle.gemm(A, B), 200, "binding")


@pytest.mark.parametrize("M,N,K,drop", [(128, 51200, 512, 0), (2560, 2560, 512, 0),
                                        (2560, 2560, 1024, 2), (512, 768, 3000, 1),
                                        (100, 1000, 2000, 1)])
def test_stream_k_wait_timeout_is_reported_and_recovers(M, N, K, drop):
    # The first three shapes leave a partial last wave, so the tail tiles are
    # split along K: 128 rows run on the one-block kernel (200 tiles of
    # 128 x 256, 152 per wave); 2560 x 2560 on the block-pair kernel (100 tiles
    # of 256 x 256, 76 pairs per wave).  The last two have few tiles, each cut
    # into four K-parts (pairs; one-block kernel).  Split unit `drop` never
    # raises its flags: the first part of a tile (0, 2) or a middle part (1 of
    # four), so the next part waits in vain.
    lib = _abi.load()
    stream = torch.cuda.current_stream().cuda_stream
    rng = np.random.default_rng(58)
    A = rng.integers(-4, 5, (M, K)).astype(np.float32)
    B = rng.integers(-4, 5, (K, N)).astype(np.float32)
    assert lib.tmm_check_device(stream) == _abi.TMM_OK
    try:
        assert lib.tmm_testing_set_wait_hooks(drop, 2_000_000) == _abi.TMM_OK
        _run(A, B, check_canaries=False, check_status=False)
        rc = lib.tmm_check_device(stream)
        assert rc == _abi.TMM_ERR_DEVICE_TIMEOUT, rc
        assert "gemm_f32_tc3" in _abi.last_error()
    finally:
        lib.tmm_testing_set_wait_hooks(-1, 0)
    assert lib.tmm_check_device(stream) == _abi.TMM_OK
    parity.assert_bit_exact(_run(A, B, check_canaries=False), oracle.gemm(A, B), "after timeout")
