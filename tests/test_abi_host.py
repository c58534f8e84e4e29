"""The C-ABI library on the host: it builds, loads, exports what the header
declares, and rejects bad arguments before touching the GPU (CPU only; no
compute call is made)."""
import ctypes
import os
import re

import pytest

from tiled_matrix_multiply_gb300 import _abi, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _abi.load()


def declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if not f.endswith(".h"):
            continue
        text = open(os.path.join(inc, f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(",
                             text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_product_entry_points():
    names = declared_functions()
    for n in ("gemm_f32", "gemm_f32_naive", "tmm_last_error_string", "tmm_version"):
        assert n in names
    assert set(names) == set(_abi.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_version(lib):
    assert lib.tmm_version() >= 100


FAKE = 0x7F0000001000  # never dereferenced: every case below fails validation first


@pytest.mark.parametrize("entry", _abi.GEMM_ENTRY_POINTS)
@pytest.mark.parametrize("args,status", [
    ((-1, 4, 4, FAKE, 4, FAKE, 4, FAKE + (1 << 20), 4), _abi.TMM_ERR_INVALID_ARG),  # M < 0
    ((4, -1, 4, FAKE, 4, FAKE, 4, FAKE, 4), _abi.TMM_ERR_INVALID_ARG),             # N < 0
    ((4, 4, -2, FAKE, 4, FAKE, 4, FAKE, 4), _abi.TMM_ERR_INVALID_ARG),             # K < 0
    ((4, 4, 8, FAKE, 7, FAKE, 4, FAKE, 4), _abi.TMM_ERR_INVALID_ARG),              # lda < K
    ((4, 5, 8, FAKE, 8, FAKE, 4, FAKE, 5), _abi.TMM_ERR_INVALID_ARG),              # ldb < N
    ((4, 5, 8, FAKE, 8, FAKE, 5, FAKE, 4), _abi.TMM_ERR_INVALID_ARG),              # ldc < N
    ((4, 4, 4, 0, 4, FAKE, 4, FAKE, 4), _abi.TMM_ERR_INVALID_ARG),                 # A NULL
    ((4, 4, 4, FAKE, 4, 0, 4, FAKE, 4), _abi.TMM_ERR_INVALID_ARG),                 # B NULL
    ((4, 4, 4, FAKE, 4, FAKE, 4, 0, 4), _abi.TMM_ERR_INVALID_ARG),                 # C NULL
    ((4, 4, 4, FAKE + 2, 4, FAKE, 4, FAKE + (1 << 20), 4), _abi.TMM_ERR_INVALID_ARG),  # misaligned
    ((1 << 31, 4, 4, FAKE, 4, FAKE, 4, FAKE + (1 << 20), 4),
     _abi.TMM_ERR_INVALID_ARG),                                                     # M >= 2^31
    ((1 << 20, 1 << 30, 4, FAKE, 4, FAKE, 1 << 30, FAKE, (1 << 62)),
     _abi.TMM_ERR_INVALID_ARG),                                                     # overflow
    ((8, 8, 8, FAKE, 8, FAKE + (1 << 20), 8, FAKE + 64, 8), _abi.TMM_ERR_ALIAS),   # C inside A
    ((8, 8, 8, FAKE, 8, FAKE + (1 << 20), 8, FAKE + (1 << 20) + 32, 8),
     _abi.TMM_ERR_ALIAS),                                                           # C inside B
])
def test_invalid_arguments_are_rejected_without_a_launch(lib, entry, args, status):
    rc = getattr(lib, entry)(*args, None)
    assert rc == status
    assert lib.tmm_last_error_string().decode()


@pytest.mark.parametrize("entry", _abi.GEMM_ENTRY_POINTS)
def test_empty_output_is_a_no_op(lib, entry):
    # M == 0 or N == 0: nothing to compute, success without any CUDA call.
    assert getattr(lib, entry)(0, 4, 4, 0, 4, 0, 4, 0, 4, None) == _abi.TMM_OK
    assert getattr(lib, entry)(4, 0, 4, 0, 4, 0, 1, 0, 1, None) == _abi.TMM_OK


def test_python_binding_rejects_host_tensors():
    torch = pytest.importorskip("torch")
    import tiled_matrix_multiply_gb300 as tmm
    A = torch.zeros(4, 4)
    with pytest.raises(ValueError):
        tmm.gemm_f32(A, A)
    with pytest.raises(TypeError):
        tmm.gemm_f32(A.double(), A.double())


@pytest.mark.parametrize("entry", ["gemm_f32_ex", "gemm_f32_tc3_ex"])
@pytest.mark.parametrize("trans,args", [
    ((2, 0), (4, 4, 4, FAKE, 4, FAKE + (1 << 20), 4, FAKE + (2 << 20), 4)),   # bad transa
    ((0, -1), (4, 4, 4, FAKE, 4, FAKE + (1 << 20), 4, FAKE + (2 << 20), 4)),  # bad transb
    ((1, 0), (8, 4, 6, FAKE, 6, FAKE + (1 << 20), 4, FAKE + (2 << 20), 4)),   # A^T: lda < M
    ((0, 1), (8, 4, 6, FAKE, 6, FAKE + (1 << 20), 4, FAKE + (2 << 20), 4)),   # B^T: ldb < K
])
def test_ex_entry_points_reject_bad_layouts(lib, entry, trans, args):
    extra = (0, 0) if entry == "gemm_f32_tc3_ex" else ()
    rc = getattr(lib, entry)(*trans, *args, *extra, None)
    assert rc == _abi.TMM_ERR_INVALID_ARG


def test_sum_workspace_size(lib):
    assert lib.sum_f32_workspace_size(0) == lib.sum_f32_workspace_size(1 << 30) == 65536


@pytest.mark.parametrize("args,status", [
    ((-1, FAKE, FAKE + (1 << 30), FAKE + (1 << 31), 65536), _abi.TMM_ERR_INVALID_ARG),  # n < 0
    (((1 << 40) + 1, FAKE, FAKE + (1 << 30), FAKE + (1 << 31), 65536),
     _abi.TMM_ERR_INVALID_ARG),                                                    # n > 2^40
    ((8, FAKE, 0, FAKE + (1 << 31), 65536), _abi.TMM_ERR_INVALID_ARG),              # out NULL
    ((8, 0, FAKE + (1 << 30), FAKE + (1 << 31), 65536), _abi.TMM_ERR_INVALID_ARG),  # x NULL
    ((8, FAKE, FAKE + (1 << 30), 0, 65536), _abi.TMM_ERR_INVALID_ARG),              # no workspace
    ((8, FAKE, FAKE + (1 << 30), FAKE + (1 << 31), 65535), _abi.TMM_ERR_INVALID_ARG),  # too small
    ((8, FAKE, FAKE + (1 << 30), FAKE + (1 << 31) + 4, 65536),
     _abi.TMM_ERR_INVALID_ARG),                                                    # ws misaligned
    ((8, FAKE + 2, FAKE + (1 << 30), FAKE + (1 << 31), 65536),
     _abi.TMM_ERR_INVALID_ARG),                                                    # x misaligned
    ((65536, FAKE, FAKE + (1 << 30), FAKE + 64, 65536), _abi.TMM_ERR_ALIAS),         # ws inside x
])
def test_sum_rejects_bad_arguments_without_a_launch(lib, args, status):
    assert lib.sum_f32(*args, None) == status
    assert lib.tmm_last_error_string().decode()


@pytest.mark.parametrize("args,status", [
    ((-1, 4, FAKE, 4, FAKE + (1 << 30), 4), _abi.TMM_ERR_INVALID_ARG),           # rows < 0
    ((4, -4, FAKE, 4, FAKE + (1 << 30), 4), _abi.TMM_ERR_INVALID_ARG),           # cols < 0
    ((1, 1 << 31, FAKE, 1 << 31, FAKE + (1 << 40), 1 << 31),
     _abi.TMM_ERR_INVALID_ARG),                                                  # cols >= 2^31
    ((4, 8, FAKE, 7, FAKE + (1 << 30), 8), _abi.TMM_ERR_INVALID_ARG),            # ldx < cols
    ((4, 8, FAKE, 8, FAKE + (1 << 30), 7), _abi.TMM_ERR_INVALID_ARG),            # ldy < cols
    ((4, 8, 0, 8, FAKE + (1 << 30), 8), _abi.TMM_ERR_INVALID_ARG),               # x NULL
    ((4, 8, FAKE, 8, 0, 8), _abi.TMM_ERR_INVALID_ARG),                           # y NULL
    ((4, 8, FAKE + 1, 8, FAKE + (1 << 30), 8), _abi.TMM_ERR_INVALID_ARG),        # misaligned
    ((1 << 40, 8, FAKE, 1 << 60, FAKE + (1 << 30), 8), _abi.TMM_ERR_INVALID_ARG),  # overflow
    ((4, 8, FAKE, 8, FAKE + 4, 8), _abi.TMM_ERR_ALIAS),                          # shifted by one
    ((4, 8, FAKE, 8, FAKE, 16), _abi.TMM_ERR_ALIAS),                             # same base, ld differs
])
def test_softmax_rejects_bad_arguments_without_a_launch(lib, args, status):
    assert lib.softmax_rows_f32(*args, None) == status
    assert lib.tmm_last_error_string().decode()


def test_softmax_empty_shapes_need_no_device(lib):
    assert lib.softmax_rows_f32(0, 8, FAKE, 8, FAKE + 64, 8, None) == _abi.TMM_OK
    assert lib.softmax_rows_f32(8, 0, FAKE, 1, FAKE, 1, None) == _abi.TMM_OK


def _header_macros():
    text = open(os.path.join(ROOT, "include", "tmm_gemm.h")).read()
    return dict(re.findall(r"^#define\s+(\w+)\s+(.+?)\s*$", text, flags=re.M))


def _macro_value(macros, name):
    v = macros[name]
    while v in macros:          # an alias of another macro
        v = macros[v]
    return int(v.strip("()"))


def test_boundary_contract_names_alias_the_library_names(lib):
    # Status codes: GEMM_ERR_* in the header equal the TMM_ERR_* codes, and the
    # binding carries both names.
    macros = _header_macros()
    for suffix in ("INVALID_ARG", "ALIAS", "UNSUPPORTED_DEVICE", "CUDA", "DEVICE_TIMEOUT", "BOUNDS"):
        g, t = _macro_value(macros, "GEMM_ERR_" + suffix), _macro_value(macros, "TMM_ERR_" + suffix)
        assert g == t == getattr(_abi, "GEMM_ERR_" + suffix) == getattr(_abi, "TMM_ERR_" + suffix)
    assert _macro_value(macros, "GEMM_OK") == _abi.TMM_OK == 0
    # The error string: both names read the calling thread's last failure.
    assert lib.gemm_f32(-1, 4, 4, FAKE, 4, FAKE, 4, FAKE + (1 << 20), 4, None) \
        == _abi.GEMM_ERR_INVALID_ARG
    msg = lib.gemm_last_error_string().decode()
    assert msg and msg == lib.tmm_last_error_string().decode()
    assert "negative size" in msg


SCRATCH = 64 << 20      # TMM_TC3_NOALLOC_SCRATCH_BYTES


def test_noalloc_scratch_constant_matches_header():
    macros = _header_macros()
    assert macros["TMM_TC3_NOALLOC_SCRATCH_BYTES"] == "((size_t)64 << 20)"


def test_tc3_workspace_size_formula_and_overflow(lib):
    # 4 Kp (2M + 2N) in 256-byte sections, Kp = K rounded up to 32.
    assert lib.gemm_f32_tc3_workspace_size(2048, 2048, 2048) == SCRATCH
    assert lib.gemm_f32_tc3_workspace_size(3, 5, 1) == 2 * 512 + 2 * 768   # 384 -> 512, 640 -> 768
    assert lib.gemm_f32_tc3_workspace_size(0, 5, 7) == 0
    assert lib.gemm_f32_tc3_workspace_size(5, 5, 1 << 31) == 0       # K out of range
    # The largest sizes: 4 * 2^31 * (4 (2^31 - 1)) bytes does not fit in size_t.
    big = (1 << 31) - 1
    assert lib.gemm_f32_tc3_workspace_size(big, big, big) == 2 ** 64 - 1


def test_noalloc_scratch_limit_boundary(lib):
    # 2048^3 needs exactly the scratch; every K that rounds to the next 32 needs more.
    assert lib.gemm_f32_tc3_workspace_size(2048, 2048, 2048) <= SCRATCH
    for K in (2049, 2080):
        assert lib.gemm_f32_tc3_workspace_size(2048, 2048, K) > SCRATCH
    assert lib.gemm_f32_tc3_workspace_size(2048, 2049, 2048) > SCRATCH
    assert lib.gemm_f32_tc3_workspace_size(3072, 1024, 2048) == SCRATCH


def _no_cuda_device():
    try:
        import torch
        return not torch.cuda.is_available()
    except ImportError:
        return True


@pytest.mark.skipif(not _no_cuda_device(),
                    reason="placeholder pointers are only passed where no GPU exists")
@pytest.mark.parametrize("shape", [(2048, 2048, 2049), (4096, 4096, 4096), (2048, 2049, 2048)])
def test_noalloc_refuses_oversized_products_before_any_cuda_call(lib, shape):
    # Refused on the size alone: on a machine without a GPU any CUDA call would
    # fail with TMM_ERR_CUDA instead, so this status shows that none was made.
    M, N, K = shape
    rc = lib.gemm_f32_tc3_noalloc(M, N, K, FAKE, K, FAKE + (1 << 36), N, FAKE + (1 << 37), N,
                                  None)
    assert rc == _abi.TMM_ERR_INVALID_ARG
    assert "scratch" in lib.tmm_last_error_string().decode()


@pytest.mark.skipif(not _no_cuda_device(),
                    reason="placeholder pointers are only passed where no GPU exists")
def test_tc3_refuses_unrepresentable_workspace(lib):
    big = (1 << 31) - 1
    rc = lib.gemm_f32_tc3(big, big, big, FAKE, big, FAKE + (1 << 62), big, FAKE + (1 << 63), big,
                          FAKE, 2 ** 64 - 1, None)
    # Either the extent check or the workspace-size check refuses it, before any CUDA call.
    assert rc == _abi.TMM_ERR_INVALID_ARG
