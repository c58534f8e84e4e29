"""FP32 matrix product C = A x B on one GB300 (sm_103a), hand-written CUDA kernels.

The work is done by ``libtmm_gemm.so`` (C ABI in ``include/tmm_gemm.h``);
this package marshals torch CUDA tensors to it.  PyTorch provides device
memory and streams only.

    import torch, tiled_matrix_multiply_gb300 as tmm
    C = tmm.gemm_f32(A, B)            # A: (M, K), B: (K, N) float32 CUDA tensors

``gemm_f32`` is the tiled FFMA path; ``gemm_f32_naive`` is the
one-output-per-thread contrast kernel; ``gemm_f32_tc3`` runs the product on the
tensor cores with split-TF32 operands (it needs a workspace, allocated here
through torch unless one is passed).  ``window_sum_f32``, ``sum_f32`` and
``softmax_rows_f32`` are the other tiled workloads of the same pages (sliding
window sums, the array reduction, the two-pass row softmax).  All are
asynchronous on the current torch stream of the operands' device.
"""
from __future__ import annotations

from ._abi import (TMM_ERR_ALIAS, TMM_ERR_CUDA, TMM_ERR_INVALID_ARG,  # noqa: F401
                   TMM_ERR_UNSUPPORTED_DEVICE, TMM_OK, TmmError)

__all__ = ["gemm_f32", "gemm_f32_naive", "gemm_f32_tc3", "tc3_workspace_bytes",
           "window_sum_f32", "sum_f32", "softmax_rows_f32", "check_device", "raw_call",
           "TmmError"]


def _matrix(x, name, allow_transposed=False):
    """(rows, cols, ld, trans) of a float32 CUDA matrix.

    trans = 0: row-major (unit column stride, ld = row stride); trans = 1: a
    transposed view of a row-major matrix (unit row stride, ld = column stride),
    accepted only where the entry point can read the operand transposed.
    """
    import torch
    if not isinstance(x, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if x.dtype != torch.float32:
        raise TypeError(f"{name} must be float32, got {x.dtype}")
    if x.dim() != 2:
        raise ValueError(f"{name} must be 2-D, got shape {tuple(x.shape)}")
    if not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    rows, cols = x.shape
    if cols <= 1 or x.stride(1) == 1:
        ld = x.stride(0) if rows > 1 else max(cols, 1)
        if x.numel() and ld < cols:
            raise ValueError(f"{name} has a row stride shorter than its rows")
        return rows, cols, max(ld, cols, 1), 0
    if allow_transposed and (rows <= 1 or x.stride(0) == 1) and x.stride(1) >= rows:
        return rows, cols, max(x.stride(1), rows, 1), 1
    raise ValueError(f"{name} must be row-major (unit column stride)"
                     + (" or a transposed row-major view" if allow_transposed else ""))


def _product(entry: str, A, B, C=None, stream=None):
    import torch
    from . import _abi
    transposable = entry == "gemm_f32"
    M, K, lda, ta = _matrix(A, "A", transposable)
    K2, N, ldb, tb = _matrix(B, "B", transposable)
    if K != K2:
        raise ValueError(f"inner dimensions differ: A is {tuple(A.shape)}, B is {tuple(B.shape)}")
    if A.device != B.device:
        raise ValueError("A and B are on different devices")
    if C is None:
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    elif C.shape != (M, N) or C.device != A.device:
        raise ValueError(f"C must be ({M}, {N}) on {A.device}")
    _, _, ldc, _ = _matrix(C, "C")
    with torch.cuda.device(A.device):
        s = stream if stream is not None else torch.cuda.current_stream(A.device)
        if ta or tb:
            rc = _abi.load().gemm_f32_ex(ta, tb, M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb,
                                         C.data_ptr(), ldc, s.cuda_stream)
            if rc != _abi.TMM_OK:
                raise _abi.TmmError("gemm_f32_ex", rc, _abi.last_error())
        else:
            _abi.check(entry, M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, C.data_ptr(), ldc,
                       s.cuda_stream)
    return C


def gemm_f32(A, B, C=None, stream=None):
    """C = A x B on the tiled FFMA path (C allocated when not given).

    A and B may also be transposed views of row-major matrices (``X.t()``):
    they are read transposed in place, without a copy.
    """
    return _product("gemm_f32", A, B, C, stream)


def gemm_f32_naive(A, B, C=None, stream=None):
    """C = A x B, one output per thread, operands from global memory."""
    return _product("gemm_f32_naive", A, B, C, stream)


def tc3_workspace_bytes(M: int, N: int, K: int) -> int:
    """Bytes of workspace gemm_f32_tc3 needs for an M x N x K product."""
    from . import _abi
    return int(_abi.load().gemm_f32_tc3_workspace_size(M, N, K))


def gemm_f32_tc3(A, B, C=None, workspace=None, stream=None):
    """C = A x B on the tensor cores (3 x TF32 split products, FP32 accumulation).

    A and B may be transposed views of row-major matrices, as for gemm_f32.
    ``workspace``: a CUDA tensor of at least ``tc3_workspace_bytes(M, N, K)``
    bytes whose storage starts 256-byte aligned (torch allocations do); one is
    allocated when not given.
    """
    import torch
    from . import _abi
    M, K, lda, ta = _matrix(A, "A", True)
    K2, N, ldb, tb = _matrix(B, "B", True)
    if K != K2:
        raise ValueError(f"inner dimensions differ: A is {tuple(A.shape)}, B is {tuple(B.shape)}")
    if A.device != B.device:
        raise ValueError("A and B are on different devices")
    if C is None:
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    elif C.shape != (M, N) or C.device != A.device:
        raise ValueError(f"C must be ({M}, {N}) on {A.device}")
    _, _, ldc, _ = _matrix(C, "C")
    need = tc3_workspace_bytes(M, N, K)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=A.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    with torch.cuda.device(A.device):
        s = stream if stream is not None else torch.cuda.current_stream(A.device)
        rc = _abi.load().gemm_f32_tc3_ex(ta, tb, M, N, K, A.data_ptr(), lda, B.data_ptr(),
                                         ldb, C.data_ptr(), ldc, workspace.data_ptr(), ws_bytes,
                                         s.cuda_stream)
        if rc != _abi.TMM_OK:
            raise _abi.TmmError("gemm_f32_tc3", rc, _abi.last_error())
    return C


def window_sum_f32(x, W=5, y=None, stream=None):
    """y[i] = sum_{d<W} x[i + d] for the len(x) - W + 1 valid windows (float32 CUDA tensors)."""
    import torch
    from . import _abi
    if not isinstance(x, torch.Tensor) or x.dtype != torch.float32 or not x.is_cuda:
        raise TypeError("x must be a float32 CUDA tensor")
    if x.dim() != 1 or (x.numel() > 1 and x.stride(0) != 1):
        raise ValueError("x must be a contiguous 1-D tensor")
    n = x.numel() - W + 1
    if n < 0:
        raise ValueError("x is shorter than one window")
    if y is None:
        y = torch.empty(n, dtype=torch.float32, device=x.device)
    elif y.shape != (n,) or (n > 1 and y.stride(0) != 1):
        raise ValueError(f"y must be a contiguous tensor of {n} floats")
    with torch.cuda.device(x.device):
        s = stream if stream is not None else torch.cuda.current_stream(x.device)
        rc = _abi.load().window_sum_f32(n, W, x.data_ptr(), y.data_ptr(), s.cuda_stream)
        if rc != _abi.TMM_OK:
            raise _abi.TmmError("window_sum_f32", rc, _abi.last_error())
    return y


def sum_f32(x, out=None, stream=None):
    """sum of every element of a contiguous float32 CUDA tensor, as a 0-d tensor (FP32)."""
    import torch
    from . import _abi
    if not isinstance(x, torch.Tensor) or x.dtype != torch.float32 or not x.is_cuda:
        raise TypeError("x must be a float32 CUDA tensor")
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")
    if out is None:
        out = torch.empty((), dtype=torch.float32, device=x.device)
    lib = _abi.load()
    need = int(lib.sum_f32_workspace_size(x.numel()))
    ws = torch.empty(need, dtype=torch.uint8, device=x.device)
    with torch.cuda.device(x.device):
        s = stream if stream is not None else torch.cuda.current_stream(x.device)
        rc = lib.sum_f32(x.numel(), x.data_ptr(), out.data_ptr(), ws.data_ptr(), need,
                         s.cuda_stream)
        if rc != _abi.TMM_OK:
            raise _abi.TmmError("sum_f32", rc, _abi.last_error())
    return out


def softmax_rows_f32(x, y=None, stream=None):
    """Softmax of every row of a float32 CUDA matrix (rows, cols); y may be x (in place)."""
    import torch
    from . import _abi
    rows, cols, ldx, trans = _matrix(x, "x")
    if y is None:
        y = torch.empty((rows, cols), dtype=torch.float32, device=x.device)
    ry, cy, ldy, _ = _matrix(y, "y")
    if (ry, cy) != (rows, cols):
        raise ValueError(f"y must be {rows} x {cols}")
    with torch.cuda.device(x.device):
        s = stream if stream is not None else torch.cuda.current_stream(x.device)
        rc = _abi.load().softmax_rows_f32(rows, cols, x.data_ptr(), ldx, y.data_ptr(), ldy,
                                          s.cuda_stream)
        if rc != _abi.TMM_OK:
            raise _abi.TmmError("softmax_rows_f32", rc, _abi.last_error())
    return y


def check_device(stream=None) -> None:
    """Synchronise the stream and raise TmmError if a bounded wait in a kernel ran out."""
    import torch
    from . import _abi
    s = stream if stream is not None else torch.cuda.current_stream()
    rc = _abi.load().tmm_check_device(s.cuda_stream)
    if rc != _abi.TMM_OK:
        raise _abi.TmmError("tmm_check_device", rc, _abi.last_error())


def raw_call(entry: str, M, N, K, A_ptr, lda, B_ptr, ldb, C_ptr, ldc, stream_ptr=0) -> int:
    """Call a C-ABI entry point with plain integers; returns the status code."""
    from . import _abi
    return _abi.call(entry, M, N, K, A_ptr, lda, B_ptr, ldb, C_ptr, ldc, stream_ptr)
