"""ctypes view of libtmm_gemm.so (include/tmm_gemm.h): names, argument types, status codes.

Argument marshalling only; the library does all of the work.  Loading fails
loudly (RuntimeError) when the library has not been built: there is no other
implementation to fall back on.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

TMM_OK = 0
TMM_ERR_INVALID_ARG = -1
TMM_ERR_ALIAS = -2
TMM_ERR_UNSUPPORTED_DEVICE = -3
TMM_ERR_CUDA = -4
TMM_ERR_DEVICE_TIMEOUT = -5
TMM_ERR_BOUNDS = -6          # the bounds-checked debug build only
# The boundary contract's names for the same codes (GEMM_ERR_* in the header).
GEMM_OK = TMM_OK
GEMM_ERR_INVALID_ARG = TMM_ERR_INVALID_ARG
GEMM_ERR_ALIAS = TMM_ERR_ALIAS
GEMM_ERR_UNSUPPORTED_DEVICE = TMM_ERR_UNSUPPORTED_DEVICE
GEMM_ERR_CUDA = TMM_ERR_CUDA
GEMM_ERR_DEVICE_TIMEOUT = TMM_ERR_DEVICE_TIMEOUT
GEMM_ERR_BOUNDS = TMM_ERR_BOUNDS

STATUS_NAMES = {
    TMM_OK: "TMM_OK",
    TMM_ERR_INVALID_ARG: "TMM_ERR_INVALID_ARG",
    TMM_ERR_ALIAS: "TMM_ERR_ALIAS",
    TMM_ERR_UNSUPPORTED_DEVICE: "TMM_ERR_UNSUPPORTED_DEVICE",
    TMM_ERR_CUDA: "TMM_ERR_CUDA",
    TMM_ERR_DEVICE_TIMEOUT: "TMM_ERR_DEVICE_TIMEOUT",
    TMM_ERR_BOUNDS: "TMM_ERR_BOUNDS",
}

# Entry points with the common product signature
# (M, N, K, A, lda, B, ldb, C, ldc, stream) -> int.
GEMM_ENTRY_POINTS = ("gemm_f32", "gemm_f32_naive")
# Every symbol include/tmm_gemm.h declares.
EXPORTED = GEMM_ENTRY_POINTS + ("gemm_f32_ex", "gemm_f32_tc3", "gemm_f32_tc3_ex",
                                 "gemm_f32_tc3_workspace_size", "gemm_f32_tc3_noalloc",
                                 "window_sum_f32", "sum_f32", "sum_f32_workspace_size",
                                 "softmax_rows_f32",
                                 "tmm_check_device", "tmm_testing_set_wait_hooks",
                                 "tmm_testing_simt_plan", "tmm_testing_tc3_plan",
                                 "tmm_last_error_string", "tmm_version",
                                 "gemm_last_error_string", "gemm_check_status")

_lock = threading.Lock()
_lib = None


class TmmError(RuntimeError):
    """A library call returned a non-zero status."""

    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn} failed with {STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def library_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libtmm_gemm.so and declare its signatures (once per process)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or library_path()
        if not os.path.exists(p):
            raise RuntimeError(
                f"{p} is missing: build it with tiled_matrix_multiply_gb300.build.build() "
                "(needs nvcc); there is no fallback implementation")
        lib = ctypes.CDLL(p)
        i64, ptr = ctypes.c_int64, ctypes.c_void_p
        for name in GEMM_ENTRY_POINTS:
            fn = getattr(lib, name)
            fn.argtypes = [i64, i64, i64, ptr, i64, ptr, i64, ptr, i64, ptr]
            fn.restype = ctypes.c_int
        lib.gemm_f32_tc3.argtypes = [i64, i64, i64, ptr, i64, ptr, i64, ptr, i64, ptr,
                                     ctypes.c_size_t, ptr]
        lib.gemm_f32_tc3.restype = ctypes.c_int
        ci = ctypes.c_int
        lib.gemm_f32_ex.argtypes = [ci, ci, i64, i64, i64, ptr, i64, ptr, i64, ptr, i64, ptr]
        lib.gemm_f32_ex.restype = ctypes.c_int
        lib.gemm_f32_tc3_ex.argtypes = [ci, ci, i64, i64, i64, ptr, i64, ptr, i64, ptr, i64,
                                        ptr, ctypes.c_size_t, ptr]
        lib.gemm_f32_tc3_ex.restype = ctypes.c_int
        lib.gemm_f32_tc3_noalloc.argtypes = [i64, i64, i64, ptr, i64, ptr, i64, ptr, i64, ptr]
        lib.gemm_f32_tc3_noalloc.restype = ctypes.c_int
        lib.gemm_f32_tc3_workspace_size.argtypes = [i64, i64, i64]
        lib.gemm_f32_tc3_workspace_size.restype = ctypes.c_size_t
        lib.window_sum_f32.argtypes = [i64, ctypes.c_int, ptr, ptr, ptr]
        lib.window_sum_f32.restype = ctypes.c_int
        lib.sum_f32.argtypes = [i64, ptr, ptr, ptr, ctypes.c_size_t, ptr]
        lib.sum_f32.restype = ctypes.c_int
        lib.sum_f32_workspace_size.argtypes = [i64]
        lib.sum_f32_workspace_size.restype = ctypes.c_size_t
        lib.softmax_rows_f32.argtypes = [i64, i64, ptr, i64, ptr, i64, ptr]
        lib.softmax_rows_f32.restype = ctypes.c_int
        lib.tmm_check_device.argtypes = [ptr]
        lib.tmm_check_device.restype = ctypes.c_int
        lib.tmm_testing_set_wait_hooks.argtypes = [ctypes.c_int, i64]
        lib.tmm_testing_set_wait_hooks.restype = ctypes.c_int
        lib.tmm_testing_simt_plan.argtypes = [i64, i64, i64, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, i64, ctypes.c_void_p]
        lib.tmm_testing_simt_plan.restype = ctypes.c_int
        lib.tmm_testing_tc3_plan.argtypes = [i64, i64, i64, ctypes.c_int, i64, ctypes.c_void_p]
        lib.tmm_testing_tc3_plan.restype = ctypes.c_int
        lib.tmm_last_error_string.argtypes = []
        lib.tmm_last_error_string.restype = ctypes.c_char_p
        lib.tmm_version.argtypes = []
        lib.tmm_version.restype = ctypes.c_int
        lib.gemm_last_error_string.argtypes = []
        lib.gemm_last_error_string.restype = ctypes.c_char_p
        lib.gemm_check_status.argtypes = [ptr]
        lib.gemm_check_status.restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


def last_error() -> str:
    return load().tmm_last_error_string().decode(errors="replace")


def call(name: str, *args) -> int:
    """Call an entry point with raw integers (pointers as ints); returns its status."""
    return int(getattr(load(), name)(*args))


def check(name: str, *args) -> None:
    """Call an entry point and raise TmmError on a non-zero status."""
    rc = call(name, *args)
    if rc != TMM_OK:
        raise TmmError(name, rc, last_error())
