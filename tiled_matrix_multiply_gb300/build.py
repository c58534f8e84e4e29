"""Compile the CUDA library (libtmm_gemm.so) in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel to an object under ``_build/``
and the objects are linked into ``tiled_matrix_multiply_gb300/lib/``.  A build
is skipped when the library is newer than every source and header.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_DIR = os.path.join(PKG, "lib")
LIB_PATH = os.path.join(LIB_DIR, "libtmm_gemm.so")
# The bounds-checked debug build (every global address and shared-memory offset
# of the product kernels range-checked, see csrc/bounds_check.cuh): its own
# objects and library, beside the normal ones.
CHECKED_FLAGS = ["-DTMM_BOUNDS_CHECK"]
CHECKED_BUILD_DIR = os.path.join(PKG, "_build_checked")
CHECKED_LIB_PATH = os.path.join(LIB_DIR, "libtmm_gemm_checked.so")

SOURCES = ["gemm_abi.cpp", "gemm_naive.cu", "gemm_simt.cu", "gemm_tc3.cu",
           "gemm_tc3_noalloc.cu", "window_sum.cu", "reduce_softmax.cu", "tensor_map.cpp",
           "operand_stage.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-Wall", "-I", INCLUDE, "-I", CSRC] + ARCH


def nvcc() -> str:
    exe = shutil.which("nvcc")
    if exe is None:
        cand = "/usr/local/cuda/bin/nvcc"
        if os.path.exists(cand):
            return cand
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtmm_gemm.so")
    return exe


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    files.append(os.path.abspath(__file__))
    return files


def source_digest(names: list[str] | None = None) -> str:
    """SHA-256 over CUDA/C++ sources (default: all sources and headers).

    ``names`` restricts it to the given files of ``csrc/`` -- the files one
    kernel is built from -- so a recorded measurement of that kernel stays
    valid while other kernels change.
    """
    import hashlib
    h = hashlib.sha256()
    if names:
        files = sorted(os.path.join(CSRC, n) for n in names)
    else:
        files = sorted(f for f in _inputs() if not f.endswith(".py"))
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def is_fresh(lib_path: str = LIB_PATH) -> bool:
    if not os.path.exists(lib_path):
        return False
    t = os.path.getmtime(lib_path)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _compile(src: str, extra: list[str], build_dir: str) -> str:
    obj = os.path.join(build_dir, os.path.basename(src) + ".o")
    cmd = [nvcc(), *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{res.stderr}")
    return obj


def _build(lib_path: str, build_dir: str, extra: list[str]) -> str:
    os.makedirs(build_dir, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    with ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, build_dir), srcs))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc(), "-shared", *ARCH, "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{res.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


def build(force: bool = False, extra_flags: list[str] | None = None) -> str:
    """Build libtmm_gemm.so unless an up-to-date copy exists; return its path."""
    if not force and not extra_flags and is_fresh():
        return LIB_PATH
    return _build(LIB_PATH, BUILD_DIR, list(extra_flags or []))


def build_checked(force: bool = False) -> str:
    """Build the bounds-checked libtmm_gemm_checked.so (a debug build for the tests) unless
    an up-to-date copy exists; return its path."""
    if not force and is_fresh(CHECKED_LIB_PATH):
        return CHECKED_LIB_PATH
    return _build(CHECKED_LIB_PATH, CHECKED_BUILD_DIR, CHECKED_FLAGS)
