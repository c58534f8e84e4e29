"""CPU oracle for C = A x B (FP32 operands, FP64 accumulation).

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this package.  The library
under ``tiled_matrix_multiply_gb300`` never imports it and shares no code with
it: the arithmetic lives in ``gemm_oracle.c`` (plain C, compiled with gcc),
this module only builds that file and marshals numpy arrays to it.

Definition followed ("Tiling Hierarchy on GPUs", section "Inner Product"):
``C[i][j] = sum_k A[i][k] * B[k][j]`` with every term widened to double and
summed in ascending k.  ``gemm`` returns that double matrix; ``gemm_f32``
rounds it once to float (round to nearest even), the value an exact FP32
result must equal bit for bit.

``window_sum`` follows "CMU DLSys Lecture 12" section 3 (``window_oracle.c``)
and is pinned by ``tests/test_window_oracle.py``; ``array_sum`` and
``softmax_rows`` follow "Tiling Strategies" section 5 (``reduce_oracle.c``)
and are pinned by ``tests/test_reduce_oracle.py``.

Every gemm function here is pinned by ``tests/test_oracle.py`` against closed forms
(identity, permutation, all-ones, integer rank-1 products), the worked
outer-product example of "CMU DLSys Lecture 12: GPU Acceleration" section 4
(``tests/golden``), exact rational brute force on tiny shapes and an
independent FP64 library product.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "gemm_oracle.c")
SOURCES = [SOURCE, os.path.join(_HERE, "window_oracle.c"),
           os.path.join(_HERE, "reduce_oracle.c")]
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libtmm_oracle.so")

_lock = threading.Lock()
_default = None


def compile_source(src, out: str) -> str:
    """gcc C sources of the oracle's form (one path or a list) into a shared library."""
    srcs = [src] if isinstance(src, str) else list(src)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-Wall", "-Wextra", "-o", tmp, *srcs, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle's C sources (gcc, OpenMP) unless an up-to-date build exists."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    fresh = (os.path.exists(_LIB_PATH)
             and all(os.path.getmtime(_LIB_PATH) >= os.path.getmtime(f) for f in SOURCES))
    if fresh and not force:
        return _LIB_PATH
    return compile_source(SOURCES, _LIB_PATH)


def _row_major_view(x: np.ndarray, name: str):
    """Return (rows, cols, ld) for a float32 row-major (possibly padded) matrix."""
    if x.dtype != np.float32:
        raise TypeError(f"{name} must be float32, got {x.dtype}")
    if x.ndim != 2:
        raise ValueError(f"{name} must be 2-D")
    rows, cols = x.shape
    item = x.itemsize
    if x.size == 0:
        return rows, cols, max(cols, 1)
    if cols > 1 and x.strides[1] != item:
        raise ValueError(f"{name} must have unit column stride")
    ld = x.strides[0] // item if rows > 1 else max(cols, 1)
    if x.strides[0] % item or ld < cols:
        raise ValueError(f"{name} has an unsupported row stride")
    return rows, cols, ld


class OracleLib:
    """Marshalling around one compiled copy of the oracle source."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i64, ptr = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_gemm_f64.argtypes = [i64, i64, i64, ptr, i64, ptr, i64, ptr, i64,
                                        ctypes.c_int]
        lib.oracle_gemm_f64.restype = ctypes.c_int
        lib.oracle_gemm_entries_f64.argtypes = [i64, i64, i64, ptr, i64, ptr, i64,
                                                ptr, ptr, i64, ptr, ctypes.c_int]
        lib.oracle_gemm_entries_f64.restype = ctypes.c_int
        lib.oracle_default_threads.argtypes = []
        lib.oracle_default_threads.restype = ctypes.c_int
        if hasattr(lib, "oracle_window_sum_f64"):
            lib.oracle_window_sum_f64.argtypes = [i64, ctypes.c_int, ptr, ptr]
            lib.oracle_window_sum_f64.restype = ctypes.c_int
            lib.oracle_window_sum_f32_ascending.argtypes = [i64, ctypes.c_int, ptr, ptr]
            lib.oracle_window_sum_f32_ascending.restype = ctypes.c_int
        if hasattr(lib, "oracle_sum_f64"):
            lib.oracle_sum_f64.argtypes = [i64, ptr, ptr]
            lib.oracle_sum_f64.restype = ctypes.c_int
            lib.oracle_softmax_rows_f64.argtypes = [i64, i64, ptr, i64, ptr, i64]
            lib.oracle_softmax_rows_f64.restype = ctypes.c_int
        self._lib = lib
        self.path = path

    def default_threads(self) -> int:
        return int(self._lib.oracle_default_threads())

    def gemm(self, A: np.ndarray, B: np.ndarray, threads: int | None = None) -> np.ndarray:
        M, K, lda = _row_major_view(A, "A")
        K2, N, ldb = _row_major_view(B, "B")
        if K != K2:
            raise ValueError(f"inner dimensions differ: {K} vs {K2}")
        C = np.empty((M, N), dtype=np.float64)
        nthr = threads if threads is not None else self.default_threads()
        rc = self._lib.oracle_gemm_f64(M, N, K, A.ctypes.data, lda, B.ctypes.data, ldb,
                                       C.ctypes.data, max(N, 1), int(nthr))
        if rc != 0:
            raise ValueError("oracle_gemm_f64 rejected its arguments")
        return C

    def gemm_entries(self, A: np.ndarray, B: np.ndarray, ii, jj,
                     threads: int | None = None) -> np.ndarray:
        M, K, lda = _row_major_view(A, "A")
        K2, N, ldb = _row_major_view(B, "B")
        if K != K2:
            raise ValueError(f"inner dimensions differ: {K} vs {K2}")
        ii = np.ascontiguousarray(ii, dtype=np.int64)
        jj = np.ascontiguousarray(jj, dtype=np.int64)
        if ii.shape != jj.shape or ii.ndim != 1:
            raise ValueError("ii and jj must be 1-D and of equal length")
        out = np.empty(ii.shape[0], dtype=np.float64)
        nthr = threads if threads is not None else self.default_threads()
        rc = self._lib.oracle_gemm_entries_f64(M, N, K, A.ctypes.data, lda,
                                               B.ctypes.data, ldb, ii.ctypes.data,
                                               jj.ctypes.data, ii.shape[0],
                                               out.ctypes.data, int(nthr))
        if rc != 0:
            raise ValueError("oracle_gemm_entries_f64 rejected its arguments")
        return out


    def window_sum(self, x: np.ndarray, W: int, fp32_ascending: bool = False) -> np.ndarray:
        """y_i = sum_{d<W} x_{i+d} for the n = len(x) - W + 1 valid windows."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        if x.ndim != 1:
            raise ValueError("x must be 1-D")
        n = x.shape[0] - W + 1
        if n < 0:
            raise ValueError("x shorter than one window")
        if fp32_ascending:
            y = np.empty(n, dtype=np.float32)
            rc = self._lib.oracle_window_sum_f32_ascending(n, W, x.ctypes.data, y.ctypes.data)
        else:
            y = np.empty(n, dtype=np.float64)
            rc = self._lib.oracle_window_sum_f64(n, W, x.ctypes.data, y.ctypes.data)
        if rc != 0:
            raise ValueError("window sum rejected its arguments")
        return y


    def array_sum(self, x: np.ndarray) -> float:
        """sum_i x_i of a float32 vector, FP64 in ascending i."""
        x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
        out = ctypes.c_double(0.0)
        rc = self._lib.oracle_sum_f64(x.shape[0], x.ctypes.data, ctypes.byref(out))
        if rc != 0:
            raise ValueError("oracle_sum_f64 rejected its arguments")
        return out.value

    def softmax_rows(self, x: np.ndarray) -> np.ndarray:
        """Row softmax of a float32 (rows, cols) matrix (row stride allowed), as float64."""
        rows, cols, ldx = _row_major_view(x, "x")
        y = np.empty((rows, cols), dtype=np.float64)
        rc = self._lib.oracle_softmax_rows_f64(rows, cols, x.ctypes.data, ldx,
                                               y.ctypes.data, max(cols, 1))
        if rc != 0:
            raise ValueError("oracle_softmax_rows_f64 rejected its arguments")
        return y


def _oracle() -> OracleLib:
    global _default
    with _lock:
        if _default is None:
            _default = OracleLib(build())
        return _default


def default_threads() -> int:
    """Host threads the oracle uses when none are given (all cores OpenMP sees)."""
    return _oracle().default_threads()


def gemm(A: np.ndarray, B: np.ndarray, threads: int | None = None) -> np.ndarray:
    """C = A x B as float64 (FP64 accumulation in ascending k), shape (M, N)."""
    return _oracle().gemm(A, B, threads)


def gemm_f32(A: np.ndarray, B: np.ndarray, threads: int | None = None) -> np.ndarray:
    """The FP64-accumulated product rounded once to float32 (round to nearest even)."""
    return gemm(A, B, threads).astype(np.float32)


def gemm_entries(A: np.ndarray, B: np.ndarray, ii, jj,
                 threads: int | None = None) -> np.ndarray:
    """C[ii[t], jj[t]] for each t, each a separate FP64 dot product in ascending k."""
    return _oracle().gemm_entries(A, B, ii, jj, threads)


def window_sum(x: np.ndarray, W: int = 5) -> np.ndarray:
    """Sliding-window sums y_i = sum_{d<W} x_{i+d} in FP64 (the definition)."""
    return _oracle().window_sum(x, W)


def window_sum_f32_ascending(x: np.ndarray, W: int = 5) -> np.ndarray:
    """The same sums accumulated in float from 0 in ascending d, as the page's fragment does."""
    return _oracle().window_sum(x, W, fp32_ascending=True)


def array_sum(x: np.ndarray) -> float:
    """sum_i x_i over a float32 array, every term in double, ascending i."""
    return _oracle().array_sum(x)


def softmax_rows(x: np.ndarray) -> np.ndarray:
    """Row-wise softmax of a float32 matrix in FP64: max pass, then normalise pass."""
    return _oracle().softmax_rows(x)
