"""The range predicate of the bounds-checked debug build, on the CPU.

csrc/bounds_check.cuh decides whether `count` consecutive elements at an
element offset lie inside a rows x cols window of row stride ld (never in the
ld - cols gap after a row).  The header is compiled here with the host C++
compiler and the predicate is compared, offset by offset, with a brute-force
enumeration of the window's elements.
"""
import itertools
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "tiled_matrix_multiply_gb300", "csrc")

SHAPES = [(1, 1, 1), (3, 4, 6), (2, 5, 5), (4, 3, 8), (1, 7, 9), (5, 1, 4)]
COUNTS = [1, 2, 4]

PROGRAM = r'''
#include <cstdio>
#include "bounds_check.cuh"
int main() {
  const long shapes[][3] = {%s};
  const int counts[] = {%s};
  for (const auto &s : shapes)
    for (int c : counts)
      for (long off = -3; off < s[0] * s[2] + 6; ++off)
        std::printf("%%ld %%ld %%ld %%d %%ld %%d\n", s[0], s[1], s[2], c, off,
                    tmm::in_window(off, s[0], s[1], s[2], c) ? 1 : 0);
  // Degenerate windows and a leading dimension shorter than the row.
  std::printf("deg %%d %%d %%d\n", tmm::in_window(0, 0, 4, 4, 1), tmm::in_window(0, 4, 0, 4, 1),
              tmm::in_window(0, 2, 5, 4, 1));
  return 0;
}
'''


def brute(rows, cols, ld, count, off):
    inside = {r * ld + c for r, c in itertools.product(range(rows), range(cols))}
    return all(off + j in inside and (off + j) // ld == off // ld for j in range(count))


@pytest.fixture(scope="module")
def output(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    d = tmp_path_factory.mktemp("bounds")
    src = d / "t.cpp"
    src.write_text(PROGRAM % (", ".join("{%d, %d, %d}" % s for s in SHAPES),
                              ", ".join(map(str, COUNTS))))
    exe = d / "t"
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    return subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout


def test_in_window_matches_enumeration(output):
    checked = 0
    for line in output.splitlines():
        if line.startswith("deg"):
            continue
        rows, cols, ld, count, off, got = map(int, line.split())
        assert bool(got) == brute(rows, cols, ld, count, off), line
        checked += 1
    assert checked == sum((r * ld + 9) * len(COUNTS) for r, _, ld in SHAPES)


def test_in_window_degenerate_windows_are_refused(output):
    deg = [line for line in output.splitlines() if line.startswith("deg")]
    assert deg == ["deg 0 0 0"]
