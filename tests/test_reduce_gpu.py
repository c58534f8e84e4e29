"""GPU parity of sum_f32 and softmax_rows_f32 ("Tiling Strategies", section 5)
against the FP64 oracle, through the C ABI.

Tolerances follow from the arithmetic the header states:
  * sum: every term passes through at most D = ceil(n / 2^25) + 54 FP32
    additions, so |s - S| <= D 2^-24 sum|x| (times 1.01 for higher-order
    terms); integer inputs whose partial sums stay below 2^24 are exact, so
    they must match bit for bit.
  * softmax: with t_j = x_j - m, fl(t_j) costs |t_j| 2^-24 relative in e^t,
    expf at most 2 ulp (4 * 2^-24), the FP32 sum of the row at most
    ceil(cols / 32) + 16 roundings on top of its terms' own errors (weighted
    by their shares Y_k), 1/s and the product one each, so to first order
    |y_j - Y_j| <= (|t_j| + 4 + sum_k Y_k (|t_k| + 4) + ceil(cols/32) + 18) 2^-24 Y_j
                   + 2^-146
    (the last term for results in the subnormal range).  Rows of more than
    65536 columns keep running sums: each rise of a thread's maximum costs one expf
    and one product (at most cols / (4 * 512 * G) of them per thread, G >= 3
    blocks per row), well inside the ceil(cols/32) additions allowed.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from gpu_util import CANARY_BITS  # noqa: E402
from tiled_matrix_multiply_gb300 import _abi, build  # noqa: E402

pytestmark = pytest.mark.gpu

CANARY = np.array([CANARY_BITS], np.uint32).view(np.float32)[0]


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    _abi.load()


def _stream():
    return torch.cuda.current_stream().cuda_stream


# ---------------------------------------------------------------- sum

def gpu_sum(x_host, offset=0):
    lib = _abi.load()
    n = x_host.shape[0]
    buf = torch.zeros(offset + n + 4, dtype=torch.float32, device="cuda")
    if n:
        buf[offset:offset + n] = torch.from_numpy(x_host).cuda()
    need = int(lib.sum_f32_workspace_size(n))
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    out = torch.full((2,), float(CANARY), dtype=torch.float32, device="cuda")
    rc = lib.sum_f32(n, buf.data_ptr() + 4 * offset, out.data_ptr(), ws.data_ptr(), need,
                     _stream())
    assert rc == _abi.TMM_OK, _abi.last_error()
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert got[1].view(np.uint32) == CANARY_BITS, "wrote past the result"
    return got[0]


def sum_bound(x):
    n = x.shape[0]
    depth = math.ceil(n / 2 ** 25) + 54
    return 1.01 * depth * 2.0 ** -24 * float(np.abs(x.astype(np.float64)).sum())


@pytest.mark.parametrize("offset", [0, 1, 2, 3])
@pytest.mark.parametrize("n", [1, 3, 4, 5, 7, 1000, 32775, 1_000_003])
def test_sum_integers_bit_exact(n, offset):
    rng = np.random.default_rng(100 + n % 97 + offset)
    x = rng.integers(-4, 5, n).astype(np.float32)
    want = oracle.array_sum(x)
    assert abs(want) < 2 ** 24
    assert gpu_sum(x, offset) == np.float32(want)


def test_sum_empty_writes_zero():
    assert gpu_sum(np.zeros(0, np.float32)) == 0.0


@pytest.mark.parametrize("n", [17, 65536, 1_048_577, (1 << 24) + 5])
def test_sum_random_within_bound(n):
    rng = np.random.default_rng(110)
    x = rng.standard_normal(n, dtype=np.float32)
    got = gpu_sum(x, offset=n % 4)
    assert abs(float(got) - oracle.array_sum(x)) <= sum_bound(x)


def test_sum_is_deterministic():
    rng = np.random.default_rng(111)
    x = rng.standard_normal((1 << 22) + 9, dtype=np.float32)
    a, b = gpu_sum(x, 1), gpu_sum(x, 1)
    assert a.view(np.uint32) == b.view(np.uint32)


def test_sum_large_uniform():
    rng = np.random.default_rng(112)
    x = rng.random((1 << 27) + 3, dtype=np.float32)
    got = gpu_sum(x)
    assert abs(float(got) - oracle.array_sum(x)) <= sum_bound(x)


# ---------------------------------------------------------------- softmax

def softmax_tolerance(x, want):
    t = np.abs(x.astype(np.float64) - x.max(axis=1, keepdims=True).astype(np.float64))
    t = np.where(np.isfinite(t), t, 0.0)      # -inf entries: e = 0 exactly on both sides
    cols = x.shape[1]
    # relative error of s: each term's own error weighted by its share Y_k, plus the additions
    sum_units = (want * (t + 4)).sum(axis=1, keepdims=True) + math.ceil(cols / 32) + 16
    units = t + 4 + sum_units + 2
    return 1.01 * units * 2.0 ** -24 * want + 2.0 ** -146


def gpu_softmax(x_host, ldx=None, ldy=None, x_off=0, in_place=False):
    """Run softmax_rows_f32 on x_host (rows, cols) placed with the given strides and offset;
    returns y (rows, cols) and checks that nothing outside y's rows was written."""
    rows, cols = x_host.shape
    ldx = ldx or max(cols, 1)
    ldy = ldx if in_place else (ldy or max(cols, 1))
    xb = torch.from_numpy(np.full(x_off + rows * ldx + 8, CANARY, np.float32)).cuda()
    view = xb[x_off:x_off + rows * ldx].view(rows, ldx)
    view[:, :cols] = torch.from_numpy(x_host).cuda()
    if in_place:
        yb, y_off = xb, x_off
    else:
        yb, y_off = torch.from_numpy(np.full(rows * ldy + 8, CANARY, np.float32)).cuda(), 0
    rc = _abi.load().softmax_rows_f32(rows, cols, xb.data_ptr() + 4 * x_off, ldx,
                                      yb.data_ptr() + 4 * y_off, ldy, _stream())
    assert rc == _abi.TMM_OK, _abi.last_error()
    torch.cuda.synchronize()
    out = yb.cpu().numpy()
    ymat = out[y_off:y_off + rows * ldy].reshape(rows, ldy)
    pad = ymat[:, cols:]
    if not in_place:
        assert np.all(pad.view(np.uint32) == CANARY_BITS), "wrote into the row padding"
        assert np.all(out[rows * ldy:].view(np.uint32) == CANARY_BITS), "wrote past y"
    return ymat[:, :cols].copy()


def check_softmax(x, **kw):
    y = gpu_softmax(x, **kw)
    want = oracle.softmax_rows(x)
    err = np.abs(y.astype(np.float64) - want)
    tol = softmax_tolerance(x, want)
    bad = np.argwhere(~(err <= tol))
    assert bad.size == 0, (x.shape, kw, bad[:3], y[tuple(bad[0])], want[tuple(bad[0])])
    return y, want


def logits(rows, cols, seed, scale=4.0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((rows, cols)) * scale).astype(np.float32)


COLS = [1, 2, 31, 32, 33, 64, 100, 128, 255, 256, 511, 512, 1000, 1024, 1025, 2047, 2048, 2049,
        4096, 8191, 8192, 8193, 16384, 16385, 24577, 32768, 49152, 49153, 65536, 65537, 65540,
        81920, 100003, 131072, 131073, 262144, 786432, 800000]


def rows_for(cols):
    return max(1, min(300, (2 << 20) // cols))


@pytest.mark.parametrize("cols", COLS)
def test_softmax_contiguous(cols):
    check_softmax(logits(rows_for(cols), cols, 120 + cols % 1000))


@pytest.mark.parametrize("cols", [3, 17, 33, 1000, 1025, 4096, 8193, 49152, 65536, 262147,
                                  400003, 1048576])
def test_softmax_strided_and_unaligned(cols):
    x = logits(min(37, rows_for(cols)), cols, 121)
    check_softmax(x, ldx=cols + 3, ldy=cols + 5)      # row starts off 16-byte boundaries
    check_softmax(x, ldx=cols + 4, x_off=1)           # x misaligned by one float
    check_softmax(x, ldx=cols + 8, ldy=cols + 12)     # padded, aligned rows


@pytest.mark.parametrize("cols", [100, 1024, 4096, 30000, 70000, 600000])
def test_softmax_in_place(cols):
    x = logits(min(21, rows_for(cols)), cols, 122)
    y = gpu_softmax(x, ldx=cols + 4, in_place=True)
    want = oracle.softmax_rows(x)
    assert np.all(np.abs(y - want) <= softmax_tolerance(x, want))


@pytest.mark.parametrize("cols", [7, 700, 7000, 70000, 500000])
def test_softmax_special_rows(cols):
    x = logits(6, cols, 123)
    x[0, :] = 2.5                       # constant row: 1 / cols everywhere
    x[1, cols // 2] = 1000.0            # one dominant entry
    x[2, ::3] = -np.inf                 # masked entries give exactly 0
    x[3, :] *= 30.0                     # wide range: many results underflow
    x[4, :] = -80.0 - np.abs(x[4, :])   # every entry very negative
    x[5, :] = np.float32(3e38) * np.sign(x[5, :]) * 0.5
    y, want = check_softmax(x)
    assert np.all(y[2, ::3] == 0.0)
    assert np.all(np.abs(y[0] - 1.0 / cols) <= (math.ceil(cols / 32) + 40) * 2.0 ** -24 / cols)


@pytest.mark.parametrize("cols", [4096, 200000, 1000000])
def test_softmax_monotone_rows(cols):
    # Ascending rows raise the running maximum at every step (the most rescales
    # of a running sum); descending rows never do.
    base = np.linspace(-30.0, 30.0, cols, dtype=np.float32)
    x = np.stack([base, base[::-1].copy(), np.sort(logits(1, cols, 126)[0])])
    check_softmax(x)


@pytest.mark.parametrize("cols,pad", [(4194304, 0), (4000037, 1)])
def test_softmax_very_long_rows(cols, pad):
    # 128 (123) blocks of the cooperative grid per row, at most 3 rows in
    # flight at once; pad = 1 takes the scalar (unaligned) form.
    x = logits(2, cols, 128)
    check_softmax(x, ldx=cols + pad, ldy=cols + pad)


def test_softmax_rows_sum_to_one_at_full_size():
    # The benchmark's shape, 65536 rows of 4096 logits, in the launch the benchmark times:
    # every row sums to 1 within the tolerance; sampled rows match the oracle.
    rows, cols = 65536, 4096
    g = torch.Generator(device="cuda").manual_seed(124)
    x = torch.randn(rows, cols, device="cuda", generator=g) * 4
    y = torch.empty_like(x)
    rc = _abi.load().softmax_rows_f32(rows, cols, x.data_ptr(), cols, y.data_ptr(), cols,
                                      _stream())
    assert rc == _abi.TMM_OK, _abi.last_error()
    sums = y.double().sum(dim=1)
    assert float((sums - 1).abs().max()) <= (2 * math.ceil(cols / 32) + 60) * 2.0 ** -24
    pick = np.random.default_rng(125).choice(rows, 48, replace=False)
    xs = x[torch.from_numpy(pick).cuda()].cpu().numpy()
    ys = y[torch.from_numpy(pick).cuda()].cpu().numpy()
    want = oracle.softmax_rows(xs)
    assert np.all(np.abs(ys - want) <= softmax_tolerance(xs, want))


def test_softmax_empty_shapes_are_noops():
    lib = _abi.load()
    y = torch.full((4,), float(CANARY), device="cuda")
    assert lib.softmax_rows_f32(0, 5, 0, 5, 0, 5, _stream()) == _abi.TMM_OK
    assert lib.softmax_rows_f32(3, 0, y.data_ptr(), 1, y.data_ptr() + 4, 1, _stream()) == _abi.TMM_OK
    torch.cuda.synchronize()
    assert np.all(y.cpu().numpy().view(np.uint32) == CANARY_BITS)


def test_python_wrappers():
    import tiled_matrix_multiply_gb300 as tmm
    x = torch.arange(1, 9, dtype=torch.float32, device="cuda")
    assert float(tmm.sum_f32(x)) == 36.0
    m = torch.tensor([[0.0, 0.0], [1.0, 1.0]], device="cuda")
    assert torch.equal(tmm.softmax_rows_f32(m), torch.full((2, 2), 0.5, device="cuda"))
    tmm.softmax_rows_f32(m, m)
    assert torch.equal(m, torch.full((2, 2), 0.5, device="cuda"))


@pytest.mark.parametrize("rows,cols", [(64, 98304), (64, 300000), (4, 4194304)])
def test_softmax_grid_wait_timeout_is_reported_and_recovers(rows, cols):
    # Rows of more than 65536 columns are shared by several blocks that meet
    # through a counter in global memory (3 blocks per row; 10; 128).  Block 1
    # never counts itself in, so the other blocks of its row run into the
    # (2 ms) limit.
    lib = _abi.load()
    stream = _stream()
    x = logits(rows, cols, 127)
    assert lib.tmm_check_device(stream) == _abi.TMM_OK
    try:
        assert lib.tmm_testing_set_wait_hooks(1, 2_000_000) == _abi.TMM_OK
        xd = torch.from_numpy(x).cuda()
        yd = torch.empty_like(xd)
        assert lib.softmax_rows_f32(rows, cols, xd.data_ptr(), cols, yd.data_ptr(), cols,
                                    stream) == _abi.TMM_OK
        rc = lib.tmm_check_device(stream)
        assert rc == _abi.TMM_ERR_DEVICE_TIMEOUT, rc
        assert "softmax_rows_f32" in _abi.last_error()
    finally:
        lib.tmm_testing_set_wait_hooks(-1, 0)
    assert lib.tmm_check_device(stream) == _abi.TMM_OK
    check_softmax(x)
    assert lib.tmm_check_device(stream) == _abi.TMM_OK


def test_softmax_long_rows_on_concurrent_streams():
    # Calls in flight at once on different streams take different regions of
    # the library's exchange memory; every result must still be right.
    lib = _abi.load()
    shapes = [(16, 131072), (8, 300000), (3, 1048576), (32, 98304)]
    xs = [logits(r, c, 129 + i) for i, (r, c) in enumerate(shapes)]
    streams = [torch.cuda.Stream() for _ in shapes]
    xd = [torch.from_numpy(x).cuda() for x in xs]
    yd = [torch.empty_like(d) for d in xd]
    torch.cuda.synchronize()
    for _ in range(3):
        for (r, c), x, y, st in zip(shapes, xd, yd, streams):
            assert lib.softmax_rows_f32(r, c, x.data_ptr(), c, y.data_ptr(), c,
                                        st.cuda_stream) == _abi.TMM_OK
    torch.cuda.synchronize()
    assert lib.tmm_check_device(_stream()) == _abi.TMM_OK
    for x, y in zip(xs, yd):
        want = oracle.softmax_rows(x)
        assert np.all(np.abs(y.cpu().numpy() - want) <= softmax_tolerance(x, want))
