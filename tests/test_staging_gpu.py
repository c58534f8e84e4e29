"""Operands restaged for the FFMA path's TMA copies (gemm_f32, gemm_f32_ex).

B stored N x K, B with rows off 16-byte boundaries, and A stored K x M with
rows off 16-byte boundaries are first copied into a K x N (K x M) scratch copy
with 16-byte rows, and the product then runs exactly as on an operand stored
that way by the caller.  The copy is a pure data movement, so:

* every restaged call equals, bit for bit, the same product with the operand
  handed over already in the aligned K-major layout (a copy made on the
  host), and agrees with the oracle within the usual bars;
* the scratch is stream-ordered and reused: repeated calls do not grow the
  device memory in use, and calls on two streams at once (each with its own
  scratch) give the single-stream results bit for bit.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import parity  # noqa: E402
from gpu_util import DevMatrix  # noqa: E402
from tiled_matrix_multiply_gb300 import _abi, build  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return _abi.load()


def _product(lib, ta, tb, As, lda, Bs, ldb, M, N, K, a_off=0, b_off=0, stream=None):
    """gemm_f32_ex on host arrays As (stored) and Bs (stored) padded to lda/ldb."""
    dA = DevMatrix(As, As.shape[0], As.shape[1], lda, a_off)
    dB = DevMatrix(Bs, Bs.shape[0], Bs.shape[1], ldb, b_off)
    dC = DevMatrix(None, M, N, N, 0)
    s = (stream or torch.cuda.current_stream()).cuda_stream
    rc = lib.gemm_f32_ex(ta, tb, M, N, K, dA.ptr, dA.ld, dB.ptr, dB.ld, dC.ptr, dC.ld, s)
    assert rc == _abi.TMM_OK, _abi.last_error()
    torch.cuda.synchronize()
    assert lib.tmm_check_device(s) == _abi.TMM_OK, _abi.last_error()
    assert dC.outside_window_untouched()
    return dC.window()


def _bits(x):
    return np.ascontiguousarray(x).view(np.uint32)


@pytest.mark.parametrize("shape", [(300, 257, 129), (1000, 3001, 517), (129, 4, 1000)])
def test_transposed_b_equals_b_given_k_major(lib, shape):
    M, N, K = shape
    rng = np.random.default_rng(80)
    A = rng.standard_normal((M, K), dtype=np.float32)
    B = rng.standard_normal((K, N), dtype=np.float32)
    Bt = np.ascontiguousarray(B.T)
    got = _product(lib, 0, 1, A, K, Bt, K, M, N, K)                 # B restaged (transposed)
    ref_ld = (N + 3) // 4 * 4
    want = _product(lib, 0, 0, A, K, B, ref_ld, M, N, K)            # B stored K x N, aligned
    assert np.array_equal(_bits(got), _bits(want)), f"{shape}: restaged B^T differs"
    parity.assert_close(got, oracle.gemm(A, B), K, f"A B^T {shape}")


@pytest.mark.parametrize("ldb_pad,b_off", [(0, 0), (1, 0), (0, 1), (3, 2)])
def test_unaligned_b_rows_equal_aligned_copy(lib, ldb_pad, b_off):
    M, N, K = 700, 1001, 333          # N = 1001: rows 4004 bytes apart
    rng = np.random.default_rng(81)
    A = rng.standard_normal((M, K), dtype=np.float32)
    B = rng.standard_normal((K, N), dtype=np.float32)
    got = _product(lib, 0, 0, A, K, B, N + ldb_pad, M, N, K, b_off=b_off)
    want = _product(lib, 0, 0, A, K, B, 1004, M, N, K)
    assert np.array_equal(_bits(got), _bits(want)), f"ldb={N + ldb_pad} off={b_off}"
    parity.assert_close(got, oracle.gemm(A, B), K, "unaligned B")


@pytest.mark.parametrize("tb", [0, 1])
def test_unaligned_a_stored_k_major_equals_aligned_copy(lib, tb):
    M, N, K = 501, 640, 250           # A stored K x M, M = 501: rows 2004 bytes apart
    rng = np.random.default_rng(82)
    A = rng.standard_normal((M, K), dtype=np.float32)
    B = rng.standard_normal((K, N), dtype=np.float32)
    At = np.ascontiguousarray(A.T)
    Bs, ldb = (np.ascontiguousarray(B.T), K) if tb else (B, N)
    got = _product(lib, 1, tb, At, M, Bs, ldb, M, N, K)
    want = _product(lib, 1, 0, At, 504, B, N, M, N, K)
    assert np.array_equal(_bits(got), _bits(want)), f"tb={tb}"
    parity.assert_close(got, oracle.gemm(A, B), K, f"A^T op(B) tb={tb}")


def test_restaging_scratch_is_reused(lib):
    M, N, K = 1024, 2048, 2048        # B^T restaged: 16 MiB of scratch per call
    dev = torch.device("cuda")
    A = torch.randn(M, K, device=dev)
    Bt = torch.randn(N, K, device=dev)
    C = torch.empty(M, N, device=dev)
    s = torch.cuda.current_stream().cuda_stream

    def call():
        rc = lib.gemm_f32_ex(0, 1, M, N, K, A.data_ptr(), K, Bt.data_ptr(), K, C.data_ptr(), N, s)
        assert rc == _abi.TMM_OK, _abi.last_error()

    call()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(40):
        call()
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert free0 - free1 < (16 << 20), f"device memory in use grew by {free0 - free1} bytes"
    assert lib.tmm_check_device(s) == _abi.TMM_OK


def test_two_streams_restaging_at_once(lib):
    M, N, K = 512, 1001, 777          # both restaged: B^T transposed, and B with unaligned rows
    rng = np.random.default_rng(83)
    dev = torch.device("cuda")
    A = torch.from_numpy(rng.standard_normal((M, K), dtype=np.float32)).to(dev)
    Bt = torch.from_numpy(rng.standard_normal((N, K), dtype=np.float32)).to(dev)
    B = Bt.t().contiguous()           # K x N, ldb = 1001
    want_t = torch.empty(M, N, device=dev)
    want_n = torch.empty(M, N, device=dev)
    s0 = torch.cuda.current_stream().cuda_stream
    assert lib.gemm_f32_ex(0, 1, M, N, K, A.data_ptr(), K, Bt.data_ptr(), K, want_t.data_ptr(),
                           N, s0) == _abi.TMM_OK
    assert lib.gemm_f32_ex(0, 0, M, N, K, A.data_ptr(), K, B.data_ptr(), N, want_n.data_ptr(),
                           N, s0) == _abi.TMM_OK
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [[torch.empty(M, N, device=dev) for _ in range(6)] for _ in streams]
    for i in range(6):
        for j, st in enumerate(streams):
            if j == 0:
                rc = lib.gemm_f32_ex(0, 1, M, N, K, A.data_ptr(), K, Bt.data_ptr(), K,
                                     outs[j][i].data_ptr(), N, st.cuda_stream)
            else:
                rc = lib.gemm_f32_ex(0, 0, M, N, K, A.data_ptr(), K, B.data_ptr(), N,
                                     outs[j][i].data_ptr(), N, st.cuda_stream)
            assert rc == _abi.TMM_OK, _abi.last_error()
    torch.cuda.synchronize()
    assert lib.tmm_check_device(s0) == _abi.TMM_OK
    for i in range(6):
        assert torch.equal(outs[0][i].view(torch.int32), want_t.view(torch.int32))
        assert torch.equal(outs[1][i].view(torch.int32), want_n.view(torch.int32))
    # The two layouts read the same matrix: the same products, bit for bit.
    assert torch.equal(want_t.view(torch.int32), want_n.view(torch.int32))
