"""Device-buffer helpers for the GPU parity tests (torch used for memory only).

Operands are placed in flat device buffers at a chosen element offset and
leading dimension, with every element outside the matrix window set to a
canary NaN bit pattern; after a call the canaries of C are checked untouched,
so a kernel that writes outside its M x N window (or into the ldc gaps) fails.
"""
from __future__ import annotations

import numpy as np
import torch

from tiled_matrix_multiply_gb300 import _abi

CANARY_BITS = np.uint32(0x7FC0DEAD)   # a quiet NaN with a recognisable payload
GUARD = 64                              # canary elements after each window


class DevMatrix:
    """A rows x cols float32 matrix inside a canary-filled flat device buffer.

    Layout: ``offset`` canary elements, then ``rows`` rows of ``ld`` elements
    (the first ``cols`` of each are the matrix), then ``GUARD`` canaries.
    """

    def __init__(self, host: np.ndarray | None, rows: int, cols: int, ld: int | None = None,
                 offset: int = 0, device="cuda"):
        self.rows, self.cols = rows, cols
        self.ld = max(ld if ld is not None else cols, 1)
        self.offset = offset
        n = offset + rows * self.ld + GUARD
        flat = np.full(n, CANARY_BITS, dtype=np.uint32).view(np.float32)
        if host is not None and rows and cols:
            self._rows_view(flat)[:, :cols] = host
        self.buf = torch.from_numpy(flat).to(device)
        self.ptr = self.buf.data_ptr() + 4 * offset

    def _rows_view(self, flat):
        return flat[self.offset:self.offset + self.rows * self.ld].reshape(self.rows, self.ld)

    def window(self) -> np.ndarray:
        flat = self.buf.cpu().numpy()
        return self._rows_view(flat)[:, :self.cols].copy()

    def outside_window_untouched(self) -> bool:
        flat = self.buf.cpu().numpy().view(np.uint32)
        ok = np.all(flat[:self.offset] == CANARY_BITS)
        ok &= np.all(flat[self.offset + self.rows * self.ld:] == CANARY_BITS)
        ok &= np.all(self._rows_view(flat)[:, self.cols:] == CANARY_BITS)
        return bool(ok)


def run_entry(entry: str, A: np.ndarray, B: np.ndarray, *, lda=None, ldb=None, ldc=None,
              a_off=0, b_off=0, c_off=0, stream=None, check_canaries=True,
              check_status=True, lib=None, trans=(0, 0)) -> np.ndarray:
    """C = op(A) x op(B) through the C ABI on device buffers laid out as requested.

    A and B are the stored matrices: with trans = (1, *) A is stored K x M, with
    (*, 1) B is stored N x K (the layouts of gemm_f32_ex / gemm_f32_tc3_ex).
    `lib` selects another build of the library (default: the normal one)."""
    ta, tb = trans
    M, K = (A.shape[1], A.shape[0]) if ta else A.shape
    N, K2 = (B.shape[0], B.shape[1]) if tb else (B.shape[1], B.shape[0])
    assert K == K2
    lib = lib if lib is not None else _abi.load()
    dA = DevMatrix(A, A.shape[0], A.shape[1], lda, a_off)
    dB = DevMatrix(B, B.shape[0], B.shape[1], ldb, b_off)
    dC = DevMatrix(None, M, N, ldc, c_off)
    s = stream if stream is not None else torch.cuda.current_stream()
    if entry in ("gemm_f32_tc3", "gemm_f32_tc3_ex"):
        need = int(lib.gemm_f32_tc3_workspace_size(M, N, K))
        ws = torch.empty(max(need, 1) + 256, dtype=torch.uint8, device=dC.buf.device)
        wptr = (ws.data_ptr() + 255) // 256 * 256
        if entry == "gemm_f32_tc3":
            assert trans == (0, 0)
            rc = lib.gemm_f32_tc3(M, N, K, dA.ptr, dA.ld, dB.ptr, dB.ld, dC.ptr, dC.ld, wptr,
                                  need, s.cuda_stream)
        else:
            rc = lib.gemm_f32_tc3_ex(ta, tb, M, N, K, dA.ptr, dA.ld, dB.ptr, dB.ld, dC.ptr,
                                     dC.ld, wptr, need, s.cuda_stream)
    elif entry == "gemm_f32_ex":
        rc = lib.gemm_f32_ex(ta, tb, M, N, K, dA.ptr, dA.ld, dB.ptr, dB.ld, dC.ptr, dC.ld,
                             s.cuda_stream)
    else:
        assert trans == (0, 0)
        rc = int(getattr(lib, entry)(M, N, K, dA.ptr, dA.ld, dB.ptr, dB.ld, dC.ptr, dC.ld,
                                     s.cuda_stream))
    msg = lib.tmm_last_error_string().decode(errors="replace")
    assert rc == _abi.TMM_OK, f"{entry} returned {rc}: {msg}"
    torch.cuda.synchronize()
    if check_status:
        st = lib.tmm_check_device(s.cuda_stream)
        assert st == _abi.TMM_OK, (st, lib.tmm_last_error_string().decode(errors="replace"))
    if check_canaries:
        assert dC.outside_window_untouched(), f"{entry} wrote outside C's M x N window"
    return dC.window()
