"""GPU parity of window_sum_f32 ("CMU DLSys Lecture 12" section 3) against the oracle.

The kernel sums each window from 0 in ascending d in FP32, the page's order, so
it must equal the oracle's float ascending sums bit for bit; it must also stay
within W float roundings of the FP64 definition.  Covers the page's worked
example, tile edges, widths 1..129, unaligned input, a large input, and that
nothing is written past the n outputs.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from gpu_util import CANARY_BITS  # noqa: E402
from tiled_matrix_multiply_gb300 import _abi, build  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    _abi.load()


def gpu_window(x_host, W, x_off=0, y_off=0):
    n = x_host.shape[0] - W + 1
    xb = torch.zeros(x_off + x_host.shape[0] + 8, dtype=torch.float32, device="cuda")
    xb[x_off:x_off + x_host.shape[0]] = torch.from_numpy(x_host).cuda()
    yb = torch.from_numpy(np.full(y_off + n + 64, CANARY_BITS, np.uint32).view(np.float32)).cuda()
    rc = _abi.load().window_sum_f32(n, W, xb.data_ptr() + 4 * x_off, yb.data_ptr() + 4 * y_off,
                                    torch.cuda.current_stream().cuda_stream)
    assert rc == _abi.TMM_OK, _abi.last_error()
    torch.cuda.synchronize()
    out = yb.cpu().numpy()
    assert np.all(out[:y_off].view(np.uint32) == CANARY_BITS), "wrote before the outputs"
    assert np.all(out[y_off + n:].view(np.uint32) == CANARY_BITS), "wrote past the n outputs"
    return out[y_off:y_off + n]


def check(x, W, x_off=0, y_off=0):
    y = gpu_window(x, W, x_off, y_off)
    want32 = oracle.window_sum_f32_ascending(x, W)
    assert np.array_equal(y.view(np.uint32), want32.view(np.uint32)), (W, x.shape)
    ref = oracle.window_sum(x, W)
    absx = oracle.window_sum(np.abs(x), W)
    assert np.all(np.abs(y - ref) <= W * 2.0 ** -24 * absx + 1e-45)


def test_page_worked_example():
    x = np.arange(1, 9, dtype=np.float32)
    assert np.array_equal(gpu_window(x, 5), [15, 20, 25, 30])


@pytest.mark.parametrize("W", [1, 2, 3, 4, 5, 6, 7, 9, 11, 13, 15, 17, 18, 33, 129])
@pytest.mark.parametrize("n", [1, 5, 4095, 4096, 4097, 12289, 100003])
def test_random_float_bit_exact(W, n):
    rng = np.random.default_rng(90 + W)
    check(rng.standard_normal(n + W - 1, dtype=np.float32), W)


@pytest.mark.parametrize("x_off", [1, 2, 3])
def test_unaligned_input(x_off):
    rng = np.random.default_rng(91)
    check(rng.standard_normal(50001, dtype=np.float32), 5, x_off)


@pytest.mark.parametrize("W", [2, 5, 17])
@pytest.mark.parametrize("x_off,y_off", [(0, 1), (0, 2), (1, 3), (2, 0), (3, 1)])
def test_unaligned_output_and_input(W, x_off, y_off):
    # y off a 16-byte boundary takes the one-output-per-thread form; n = 4097 + 2
    # leaves a ragged group of four at the end.
    rng = np.random.default_rng(92 + W)
    check(rng.standard_normal(4099 + W - 1, dtype=np.float32), W, x_off, y_off)


def test_integer_inputs_exact_against_definition():
    rng = np.random.default_rng(92)
    x = rng.integers(-1000, 1001, 1 << 20).astype(np.float32)
    y = gpu_window(x, 5)
    assert np.array_equal(y.astype(np.float64), oracle.window_sum(x, 5))


def test_large_input():
    rng = np.random.default_rng(93)
    check(rng.random((1 << 26) + 4, dtype=np.float32) * 2 - 1, 5)


def test_rejects_bad_arguments():
    lib = _abi.load()
    x = torch.zeros(100, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert lib.window_sum_f32(10, 0, x.data_ptr(), x.data_ptr() + 400, s) == _abi.TMM_ERR_INVALID_ARG
    assert lib.window_sum_f32(10, 130, x.data_ptr(), x.data_ptr() + 400, s) == _abi.TMM_ERR_INVALID_ARG
    assert lib.window_sum_f32(50, 5, x.data_ptr(), x.data_ptr() + 40, s) == _abi.TMM_ERR_ALIAS
    assert lib.window_sum_f32(0, 5, 0, 0, s) == _abi.TMM_OK


def test_bulk_copy_wait_timeout_is_reported_and_recovers():
    # Block 0 is armed for 16 bytes more than its first tile copy brings, so its
    # bounded wait runs out (2 ms); the status is reported once and the next call
    # is correct again.
    lib = _abi.load()
    s = torch.cuda.current_stream().cuda_stream
    x = np.arange(1 << 20, dtype=np.float32) % 7
    assert lib.tmm_check_device(s) == _abi.TMM_OK
    try:
        assert lib.tmm_testing_set_wait_hooks(0, 2_000_000) == _abi.TMM_OK
        xb = torch.from_numpy(x).cuda()
        yb = torch.empty(x.shape[0] - 4, device="cuda")
        assert lib.window_sum_f32(x.shape[0] - 4, 5, xb.data_ptr(), yb.data_ptr(), s) == _abi.TMM_OK
        assert lib.tmm_check_device(s) == _abi.TMM_ERR_DEVICE_TIMEOUT
        assert "window_sum_f32" in _abi.last_error()
    finally:
        lib.tmm_testing_set_wait_hooks(-1, 0)
    assert lib.tmm_check_device(s) == _abi.TMM_OK
    check(x, 5)
