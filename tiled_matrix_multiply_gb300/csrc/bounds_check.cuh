// bounds_check.cuh -- range checks of the library's debug build.
//
// Built with -DTMM_BOUNDS_CHECK, the product kernels check every global
// address they read or write against the extent of its matrix -- its stored
// rows and columns, never the gap a leading dimension leaves after a row --
// and every shared-memory offset against its slab.  An access that fails its
// check is skipped (a load yields 0) and bit 2 (kStatusBounds) of the kernel's
// status word is set; tmm_check_device reports it as TMM_ERR_BOUNDS.  Nothing
// traps.  In the normal build TMM_IN_BOUNDS(cond, status) is the constant true
// and its arguments are never evaluated, so the kernels compile exactly as
// without the checks.
//
// The checks stand in for a memory checker where none can run: they catch an
// index past a buffer's end or into a row gap even where the value read there
// would not change a result.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define TMM_HD __host__ __device__
#else
#define TMM_HD
#endif

namespace tmm {

constexpr unsigned int kStatusBounds = 4u;

// Whether the `count` consecutive elements starting at element offset `off`
// from a matrix's base all lie inside its rows x cols window (row stride ld):
// the row is below `rows`, and the columns col .. col + count - 1 are below
// `cols` (so none falls in the ld - cols gap after the row).
TMM_HD inline bool in_window(int64_t off, int64_t rows, int64_t cols, int64_t ld, int count) {
  if (off < 0 || rows <= 0 || cols <= 0 || ld < cols || count < 1) return false;
  const int64_t r = off / ld, c = off - r * ld;
  return r < rows && c + count <= cols;
}

#if defined(__CUDACC__)
__device__ __forceinline__ bool in_matrix(const float *p, const float *base, int64_t rows,
                                          int64_t cols, int64_t ld, int count = 1) {
  return in_window(p - base, rows, cols, ld, count);
}
// `count` floats from byte offset `byte_off` inside a region of `region_floats` floats.
__device__ __forceinline__ bool in_region(int64_t byte_off, int64_t region_floats,
                                          int count = 1) {
  return byte_off >= 0 && (byte_off & 3) == 0 && byte_off / 4 + count <= region_floats;
}
__device__ __forceinline__ bool bounds_ok(bool cond, unsigned int *status) {
  if (!cond) atomicOr(status, kStatusBounds);
  return cond;
}
#endif

}  // namespace tmm

#ifdef TMM_BOUNDS_CHECK
#define TMM_IN_BOUNDS(cond, status) (::tmm::bounds_ok((cond), (status)))
#else
#define TMM_IN_BOUNDS(cond, status) (true)
#endif
