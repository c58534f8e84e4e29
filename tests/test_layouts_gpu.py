"""GPU parity of the transposed layouts: C = op(A) x op(B) through gemm_f32_ex
and gemm_f32_tc3_ex, against the oracle applied to op(A), op(B).

op(A) = A^T reads A stored K x M -- the layout of "CMU DLSys Lecture 12"
section 4, C_ij = sum_k A_ki B_kj; op(B) = B^T reads B stored N x K.  The
oracle's arithmetic is unchanged: the tests form op(A), op(B) on the host by a
transpose (data movement only) and compare entry by entry, with the usual bars
(normwise 1e-5, elementwise 1e-4 sqrt(K), bit-exact for integer inputs).
"""
import itertools

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import parity  # noqa: E402
from gpu_util import DevMatrix  # noqa: E402
from tiled_matrix_multiply_gb300 import _abi, build, inputs  # noqa: E402

pytestmark = pytest.mark.gpu

ENTRIES = ["gemm_f32_ex", "gemm_f32_tc3_ex"]
TRANS = list(itertools.product([0, 1], repeat=2))


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    _abi.load()


def run_layout(entry, ta, tb, opA, opB, pad=(0, 0, 0), off=(0, 0, 0), canaries=True):
    """C = opA x opB with A stored as opA (ta = 0) or opA^T (ta = 1), likewise B."""
    M, K = opA.shape
    N = opB.shape[1]
    As = np.ascontiguousarray(opA.T) if ta else opA
    Bs = np.ascontiguousarray(opB.T) if tb else opB
    dA = DevMatrix(As, As.shape[0], As.shape[1], As.shape[1] + pad[0], off[0])
    dB = DevMatrix(Bs, Bs.shape[0], Bs.shape[1], Bs.shape[1] + pad[1], off[1])
    dC = DevMatrix(None, M, N, N + pad[2], off[2])
    lib = _abi.load()
    s = torch.cuda.current_stream().cuda_stream
    if entry == "gemm_f32_tc3_ex":
        need = int(lib.gemm_f32_tc3_workspace_size(M, N, K))
        ws = torch.empty(max(need, 1) + 256, dtype=torch.uint8, device="cuda")
        wptr = (ws.data_ptr() + 255) // 256 * 256
        rc = lib.gemm_f32_tc3_ex(ta, tb, M, N, K, dA.ptr, dA.ld, dB.ptr, dB.ld, dC.ptr, dC.ld,
                                 wptr, need, s)
    else:
        rc = lib.gemm_f32_ex(ta, tb, M, N, K, dA.ptr, dA.ld, dB.ptr, dB.ld, dC.ptr, dC.ld, s)
    assert rc == _abi.TMM_OK, _abi.last_error()
    torch.cuda.synchronize()
    assert lib.tmm_check_device(s) == _abi.TMM_OK
    if canaries:
        assert dC.outside_window_untouched()
    return dC.window()


@pytest.mark.parametrize("entry", ENTRIES)
@pytest.mark.parametrize("ta,tb", TRANS)
@pytest.mark.parametrize("shape", [(256, 384, 200), (129, 257, 77), (300, 521, 1000),
                                   (1, 300, 33), (250, 1, 129)])
def test_layouts_float(entry, ta, tb, shape):
    M, N, K = shape
    rng = np.random.default_rng(70)
    A = rng.random((M, K), dtype=np.float32) * 2 - 1
    B = rng.random((K, N), dtype=np.float32) * 2 - 1
    C = run_layout(entry, ta, tb, A, B)
    parity.assert_close(C, oracle.gemm(A, B), K, f"{entry} ta={ta} tb={tb} {shape}")


@pytest.mark.parametrize("entry", ENTRIES)
@pytest.mark.parametrize("ta,tb", TRANS)
def test_layouts_integer_exact_tile_edges(entry, ta, tb):
    rng = np.random.default_rng(71)
    for M, N, K in itertools.product([1, 63, 64, 65, 129], [1, 255, 256, 257], [1, 15, 17, 48]):
        A = rng.integers(-4, 5, (M, K)).astype(np.float32)
        B = rng.integers(-4, 5, (K, N)).astype(np.float32)
        C = run_layout(entry, ta, tb, A, B)
        parity.assert_bit_exact(C, oracle.gemm(A, B), f"{entry} ta={ta} tb={tb} {M}x{N}x{K}")


@pytest.mark.parametrize("entry", ENTRIES)
@pytest.mark.parametrize("ta,tb", TRANS)
@pytest.mark.parametrize("pad,off", [((4, 8, 12), (4, 8, 4)), ((1, 3, 5), (3, 1, 1))])
def test_layouts_padded_and_unaligned(entry, ta, tb, pad, off):
    rng = np.random.default_rng(72)
    M, N, K = 200, 300, 150
    A = rng.standard_normal((M, K), dtype=np.float32)
    B = rng.standard_normal((K, N), dtype=np.float32)
    C = run_layout(entry, ta, tb, A, B, pad, off)
    parity.assert_close(C, oracle.gemm(A, B), K, f"{entry} ta={ta} tb={tb} pad={pad} off={off}")


@pytest.mark.parametrize("ta,tb", TRANS)
@pytest.mark.parametrize("shape", [(130, 515, 45), (700, 1030, 333)])
def test_simt_rows_at_every_alignment(ta, tb, shape):
    # Rows of A (stored K x M) and B (stored K x N) that start at each 4-byte
    # position inside a 16-byte line: every base offset mod 4 against every
    # leading dimension mod 4, over several tiles in each direction and a
    # ragged K.  Integer inputs, so the products are exact; the canary NaNs
    # around each matrix reach C if any element outside the matrix is read
    # into a sum.
    M, N, K = shape
    rng = np.random.default_rng(73)
    A = rng.integers(-8, 9, (M, K)).astype(np.float32)
    B = rng.integers(-8, 9, (K, N)).astype(np.float32)
    want = oracle.gemm(A, B)
    for off, pad in itertools.product(range(4), range(4)):
        o = (off, (off + 2) % 4, 0)
        d = (pad, (pad + 1) % 4, 0)
        C = run_layout("gemm_f32_ex", ta, tb, A, B, d, o)
        parity.assert_bit_exact(C, want, f"ta={ta} tb={tb} {shape} off={o} pad={d}")


@pytest.mark.parametrize("entry", ENTRIES)
@pytest.mark.parametrize("ta,tb", [(1, 0), (0, 1), (1, 1)])
def test_headline_size_transposed(entry, ta, tb):
    # The 4096^3 workload read through each transposed layout (A^T B is the
    # DLSys layout); full comparison with the oracle.
    w = inputs.WORKLOADS["square4096"]
    A, B = inputs.workload_operands(w)
    C = run_layout(entry, ta, tb, A, B, canaries=False)
    parity.assert_close(C, oracle.gemm(A, B), w.K, f"{entry} ta={ta} tb={tb} 4096^3")


def test_python_binding_accepts_transposed_views():
    import tiled_matrix_multiply_gb300 as tmm
    rng = np.random.default_rng(73)
    At = torch.from_numpy(rng.standard_normal((500, 300), dtype=np.float32)).cuda()  # K x M
    Bt = torch.from_numpy(rng.standard_normal((400, 500), dtype=np.float32)).cuda()  # N x K
    ref = oracle.gemm(np.ascontiguousarray(At.cpu().numpy().T),
                      np.ascontiguousarray(Bt.cpu().numpy().T))
    for fn in (tmm.gemm_f32, tmm.gemm_f32_tc3):
        C = fn(At.t(), Bt.t())
        torch.cuda.synchronize()
        parity.assert_close(C.cpu().numpy(), ref, 500, fn.__name__)
