"""GPU parity: every entry point of the C ABI against the CPU oracle.

Float inputs must meet the normwise (1e-5) and elementwise (1e-4 sqrt(K))
bars of ``parity.py`` against the oracle's FP64-accumulated product;
integer-valued inputs must equal the oracle rounded to FP32 bit for bit.
Full-size workloads the oracle can form in seconds are compared entry by
entry; the 8192-class workloads are compared on sampled entries (the oracle
computes each one separately) plus Freivalds' identity on the whole result,
exact for integer inputs.
"""
import itertools

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import parity  # noqa: E402
from tiled_matrix_multiply_gb300 import _abi, build, inputs  # noqa: E402

pytestmark = pytest.mark.gpu

ENTRIES = _abi.GEMM_ENTRY_POINTS


@pytest.fixture(scope="session", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    _abi.load()


def _run(*a, **k):
    from gpu_util import run_entry
    return run_entry(*a, **k)


_oracle_cache = {}


def _oracle_full(name, A, B):
    if name not in _oracle_cache:
        _oracle_cache[name] = oracle.gemm(A, B)
    return _oracle_cache[name]


# -- the workloads at their full sizes ------------------------------------------------

FULL_ORACLE = ["square256", "square256_int", "square1024", "ragged4000x3001x2047", "square4096"]


@pytest.mark.parametrize("entry", ENTRIES)
@pytest.mark.parametrize("name", FULL_ORACLE)
def test_workload_full_compare(entry, name):
    w = inputs.WORKLOADS[name]
    A, B = inputs.workload_operands(w)
    C = _run(entry, A, B, check_canaries=(w.M * w.N <= 1 << 22))
    ref = _oracle_full(name, A, B)
    if w.dist == "int4":
        parity.assert_bit_exact(C, ref, f"{entry} {name}")
    else:
        parity.assert_close(C, ref, w.K, f"{entry} {name}")


@pytest.mark.parametrize("entry", ENTRIES)
@pytest.mark.parametrize("name", ["square1024", "ragged4000x3001x2047", "square4096"])
def test_workload_integer_variant_bit_exact(entry, name):
    w = inputs.WORKLOADS[name]
    A, B = inputs.make_operands(w.M, w.N, w.K, "int4", w.seed)
    C = _run(entry, A, B, check_canaries=False)
    parity.assert_bit_exact(C, _oracle_full(name + "/int4", A, B), f"{entry} {name} int4")


LARGE = ["rect8192x8192x1024", "rect16384x1024x4096", "rect1024x16384x4096", "square8192"]


def _sample_indices(M, N, count, seed):
    rng = np.random.default_rng(seed)
    ii = rng.integers(0, M, count)
    jj = rng.integers(0, N, count)
    # Always include the four corners and the last row/column tails.
    ii = np.concatenate([ii, [0, 0, M - 1, M - 1], np.full(64, M - 1), np.arange(64) % M])
    jj = np.concatenate([jj, [0, N - 1, 0, N - 1], np.arange(64) % N, np.full(64, N - 1)])
    return ii, jj


def _freivalds(A, B, C, x):
    lhs = C.astype(np.float64) @ x
    rhs = A.astype(np.float64) @ (B.astype(np.float64) @ x)
    return lhs, rhs


@pytest.mark.parametrize("entry", ENTRIES)
@pytest.mark.parametrize("name", LARGE)
def test_large_workload_sampled_and_freivalds(entry, name):
    w = inputs.WORKLOADS[name]
    A, B = inputs.workload_operands(w)
    C = _run(entry, A, B, check_canaries=False)
    ii, jj = _sample_indices(w.M, w.N, 4096, 7)
    ref = oracle.gemm_entries(A, B, ii, jj)
    got = C[ii, jj]
    assert np.max(np.abs(got - ref)) <= parity.elementwise_tol(w.K)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel <= parity.NORMWISE_TOL
    x = np.random.default_rng(8).standard_normal(w.N)
    lhs, rhs = _freivalds(A, B, C, x)
    assert np.linalg.norm(lhs - rhs) / np.linalg.norm(rhs) <= parity.NORMWISE_TOL


@pytest.mark.parametrize("entry", ENTRIES)
@pytest.mark.parametrize("name", LARGE)
def test_large_workload_integer_variant_exact(entry, name):
    w = inputs.WORKLOADS[name]
    A, B = inputs.make_operands(w.M, w.N, w.K, "int4", w.seed)
    C = _run(entry, A, B, check_canaries=False)
    ii, jj = _sample_indices(w.M, w.N, 4096, 9)
    ref = oracle.gemm_entries(A, B, ii, jj)
    parity.assert_bit_exact(C[ii, jj], ref, f"{entry} {name}")
    # With integer C and x in {-1, 0, 1} both sides of Freivalds' identity are
    # exact in FP64, so any wrong entry shows with probability >= 1/2 per vector.
    rng = np.random.default_rng(10)
    for _ in range(2):
        x = rng.integers(-1, 2, w.N).astype(np.float64)
        lhs, rhs = _freivalds(A, B, C, x)
        assert np.array_equal(lhs, rhs)


# -- shapes around tile edges, tiny shapes, layouts -----------------------------------

EDGE_M = [1, 2, 127, 128, 129, 255, 257]
EDGE_N = [1, 3, 4, 127, 128, 129, 131]
EDGE_K = [1, 3, 7, 8, 9, 16, 17, 33]


@pytest.mark.parametrize("entry", ENTRIES)
def test_tile_edge_shapes_integer_exact(entry):
    rng = np.random.default_rng(30)
    for M, N, K in itertools.product(EDGE_M, EDGE_N, EDGE_K):
        A = rng.integers(-4, 5, (M, K)).astype(np.float32)
        B = rng.integers(-4, 5, (K, N)).astype(np.float32)
        C = _run(entry, A, B)
        parity.assert_bit_exact(C, oracle.gemm(A, B), f"{entry} {M}x{N}x{K}")


@pytest.mark.parametrize("entry", ENTRIES)
def test_tile_edge_shapes_float(entry):
    rng = np.random.default_rng(31)
    for M, N, K in [(129, 131, 1000), (255, 127, 517), (257, 257, 129), (1, 1000, 999),
                    (1000, 1, 999), (130, 260, 4099)]:
        A = rng.random((M, K), dtype=np.float32) * 2 - 1
        B = rng.random((K, N), dtype=np.float32) * 2 - 1
        C = _run(entry, A, B)
        parity.assert_close(C, oracle.gemm(A, B), K, f"{entry} {M}x{N}x{K}")


@pytest.mark.parametrize("entry", ENTRIES)
def test_tiny_shapes_brute_force(entry):
    rng = np.random.default_rng(32)
    for M, N, K in itertools.product(range(1, 10), repeat=3):
        A = rng.integers(-4, 5, (M, K)).astype(np.float32)
        B = rng.integers(-4, 5, (K, N)).astype(np.float32)
        C = _run(entry, A, B)
        parity.assert_bit_exact(C, oracle.gemm(A, B), f"{entry} {M}x{N}x{K}")


LAYOUTS = {
    # name: (lda_pad, ldb_pad, ldc_pad, a_off, b_off, c_off)
    "compact_aligned": (0, 0, 0, 0, 0, 0),
    "padded_aligned": (4, 8, 12, 4, 8, 4),
    "padded_odd": (1, 3, 5, 0, 0, 0),
    "a_unaligned": (0, 0, 0, 1, 0, 0),
    "b_unaligned": (0, 0, 0, 0, 3, 0),
    "c_unaligned": (0, 0, 0, 0, 0, 2),
    "all_unaligned_padded": (5, 7, 9, 3, 1, 1),
}


@pytest.mark.parametrize("entry", ENTRIES)
@pytest.mark.parametrize("layout", sorted(LAYOUTS))
@pytest.mark.parametrize("shape", [(200, 136, 64), (131, 257, 77)])
def test_layouts(entry, layout, shape):
    M, N, K = shape
    pa, pb, pc, oa, ob, oc = LAYOUTS[layout]
    rng = np.random.default_rng(33)
    A = rng.standard_normal((M, K), dtype=np.float32)
    B = rng.standard_normal((K, N), dtype=np.float32)
    C = _run(entry, A, B, lda=K + pa, ldb=N + pb, ldc=N + pc, a_off=oa, b_off=ob, c_off=oc)
    parity.assert_close(C, oracle.gemm(A, B), K, f"{entry} {layout}")
    Ai = rng.integers(-4, 5, (M, K)).astype(np.float32)
    Bi = rng.integers(-4, 5, (K, N)).astype(np.float32)
    Ci = _run(entry, Ai, Bi, lda=K + pa, ldb=N + pb, ldc=N + pc, a_off=oa, b_off=ob, c_off=oc)
    parity.assert_bit_exact(Ci, oracle.gemm(Ai, Bi), f"{entry} {layout} int")


@pytest.mark.parametrize("entry", ENTRIES)
def test_k_zero_writes_zeros_inside_window_only(entry):
    from gpu_util import DevMatrix
    M, N = 37, 45
    dA = DevMatrix(np.zeros((M, 0), np.float32), M, 0, 1)
    dB = DevMatrix(np.zeros((0, N), np.float32), 0, N, N)
    dC = DevMatrix(None, M, N, N + 3, offset=5)
    rc = _abi.call(entry, M, N, 0, dA.ptr, dA.ld, dB.ptr, dB.ld, dC.ptr, dC.ld,
                   torch.cuda.current_stream().cuda_stream)
    assert rc == _abi.TMM_OK
    torch.cuda.synchronize()
    assert np.all(dC.window() == 0)
    assert dC.outside_window_untouched()


@pytest.mark.parametrize("entry", ENTRIES)
def test_overlapping_output_is_rejected_and_nothing_runs(entry):
    M = N = K = 64
    buf = torch.zeros(M * K * 2, device="cuda")
    A = buf[: M * K]
    C = buf[M * K // 2: M * K // 2 + M * N]     # overlaps the second half of A
    B = torch.ones(K * N, device="cuda")
    before = buf.clone()
    rc = _abi.call(entry, M, N, K, A.data_ptr(), K, B.data_ptr(), N, C.data_ptr(), N,
                   torch.cuda.current_stream().cuda_stream)
    assert rc == _abi.TMM_ERR_ALIAS
    torch.cuda.synchronize()
    assert torch.equal(buf, before)


@pytest.mark.parametrize("entry", ENTRIES)
def test_side_stream_and_python_binding(entry):
    import tiled_matrix_multiply_gb300 as tmm
    rng = np.random.default_rng(34)
    A = rng.standard_normal((300, 200), dtype=np.float32)
    B = rng.standard_normal((200, 400), dtype=np.float32)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dA = torch.from_numpy(A).cuda()
        dB = torch.from_numpy(B).cuda()
        fn = tmm.gemm_f32 if entry == "gemm_f32" else tmm.gemm_f32_naive
        C = fn(dA, dB)
    s.synchronize()
    parity.assert_close(C.cpu().numpy(), oracle.gemm(A, B), 200, entry)


def test_repeat_calls_are_bit_identical():
    rng = np.random.default_rng(35)
    A = rng.standard_normal((513, 700), dtype=np.float32)
    B = rng.standard_normal((700, 390), dtype=np.float32)
    C1 = _run("gemm_f32", A, B)
    C2 = _run("gemm_f32", A, B)
    assert np.array_equal(C1.view(np.uint32), C2.view(np.uint32))


# Shapes large enough for the 64 x 512 tiles of aligned A x B (their tiles fill two
# waves of SMs), with tails in M, N and K: N a multiple of 4, and N odd with a
# padded, aligned leading dimension (B staged by TMA either way).
@pytest.mark.parametrize("M,N,K,ldb", [(4000, 2996, 1001, 2996), (4000, 3001, 1001, 3004),
                                        (2500, 4100, 517, 4100)])
def test_wide_tile_path_tails(M, N, K, ldb):
    rng = np.random.default_rng(36)
    A = rng.random((M, K), dtype=np.float32) * 2 - 1
    B = rng.random((K, N), dtype=np.float32) * 2 - 1
    C = _run("gemm_f32", A, B, ldb=ldb, check_canaries=False)
    parity.assert_close(C, oracle.gemm(A, B), K, f"wide {M}x{N}x{K}")
    Ai = rng.integers(-4, 5, (M, K)).astype(np.float32)
    Bi = rng.integers(-4, 5, (K, N)).astype(np.float32)
    Ci = _run("gemm_f32", Ai, Bi, ldb=ldb, ldc=N + 3)
    parity.assert_bit_exact(Ci, oracle.gemm(Ai, Bi), f"wide int {M}x{N}x{K}")
