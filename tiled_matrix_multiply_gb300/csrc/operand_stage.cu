// operand_stage.cu -- operands of the tiled product restaged for its TMA copies.
//
// The tiled kernel reads each K-slice of B as one TMA box of b[k][n] (and of A
// as a[k][m] when A is stored K x M).  A TMA copy needs the rows of its matrix
// to start on 16-byte boundaries (base 16-byte aligned, row pitch a multiple
// of 4 floats) and the copied rows to run along n (or m).  An operand stored
// otherwise -- B stored N x K (the A B^T layouts), or rows whose pitch is not
// a multiple of 4 floats (N = 3001, say) -- is first copied into that layout
// in a scratch buffer: element by element when only the pitch changes, by a
// shared-memory transpose when the stored rows run along k.  Either copy
// reads and writes the operand once (8 bytes per element of HBM traffic),
// about 1 % of the product's time at 4096^3, and lets the product run its
// copy-free B path instead of one 4-byte copy per element and K-slice.
//
// The scratch comes from a stream-ordered memory pool the library owns (one
// per device): allocated on the call's stream before the copy, freed on it
// after the product, so concurrent calls on different streams never share a
// buffer.  The pool keeps up to kPoolKeepBytes of freed memory for later
// calls (a 4096 x 4096 operand is 64 MiB), so steady use makes no driver
// allocation; memory beyond that goes back to the device when the stream is
// synchronised.
#include <cstdint>
#include <mutex>

#include "bounds_check.cuh"
#include "tmm_internal.h"

namespace tmm {

// Bit 2 (kStatusBounds) of the bounds-checked build, as for the product kernels.
__device__ unsigned int g_stage_status;

namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 8;

// dst[r][c] = src[r][c] for r < rows, c < cols; dst rows are ld_dst apart.
// Consecutive threads take consecutive columns of a row (4-byte accesses, a
// warp covers 128 contiguous bytes on either side); each thread takes
// kCopyUnroll rows of its column per step, all loads in flight together.
__global__ void __launch_bounds__(kCopyThreads)
stage_rows_kernel(const float *__restrict__ src, int64_t ld_src, int64_t rows, int64_t cols,
                  float *__restrict__ dst, int64_t ld_dst) {
  const int64_t col_blocks = (cols + kCopyThreads - 1) / kCopyThreads;
  const int64_t row_groups = (rows + kCopyUnroll - 1) / kCopyUnroll;
  for (int64_t item = blockIdx.x; item < col_blocks * row_groups; item += gridDim.x) {
    const int64_t rg = item / col_blocks;
    const int64_t c = (item - rg * col_blocks) * kCopyThreads + threadIdx.x;
    if (c >= cols) continue;
    float v[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t r = rg * kCopyUnroll + u;
      const float *s = src + r * ld_src + c;
      v[u] = (r < rows && TMM_IN_BOUNDS(in_matrix(s, src, rows, cols, ld_src), &g_stage_status))
                 ? __ldg(s) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t r = rg * kCopyUnroll + u;
      float *d = dst + r * ld_dst + c;
      if (r < rows && TMM_IN_BOUNDS(in_matrix(d, dst, rows, cols, ld_dst), &g_stage_status))
        *d = v[u];
    }
  }
}

// dst[c][r] = src[r][c] for r < rows, c < cols (dst has cols rows, ld_dst
// apart).  32 x 32 tiles through shared memory: a warp reads 32 consecutive
// columns of a source row and writes 32 consecutive columns of a
// destination row; the tile's row pitch of 33 words keeps the column reads
// of shared memory on 32 distinct banks.
constexpr int kTile = 32, kTileRowsPerPass = kCopyThreads / kTile;

__global__ void __launch_bounds__(kCopyThreads)
stage_transpose_kernel(const float *__restrict__ src, int64_t ld_src, int64_t rows,
                       int64_t cols, float *__restrict__ dst, int64_t ld_dst) {
  __shared__ float tile[kTile][kTile + 1];
  const int tx = threadIdx.x % kTile, ty = threadIdx.x / kTile;
  const int64_t tiles_c = (cols + kTile - 1) / kTile;
  const int64_t tiles = ((rows + kTile - 1) / kTile) * tiles_c;
  for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
    const int64_t r0 = (t / tiles_c) * kTile, c0 = (t % tiles_c) * kTile;
#pragma unroll
    for (int i = ty; i < kTile; i += kTileRowsPerPass) {
      const int64_t r = r0 + i, c = c0 + tx;
      const float *s = src + r * ld_src + c;
      tile[i][tx] = (r < rows && c < cols &&
                     TMM_IN_BOUNDS(in_matrix(s, src, rows, cols, ld_src), &g_stage_status))
                        ? __ldg(s) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int i = ty; i < kTile; i += kTileRowsPerPass) {
      const int64_t c = c0 + i, r = r0 + tx;   // destination row c, column r
      float *d = dst + c * ld_dst + r;
      if (c < cols && r < rows &&
          TMM_IN_BOUNDS(in_matrix(d, dst, cols, rows, ld_dst), &g_stage_status))
        *d = tile[tx][i];
    }
    __syncthreads();   // the tile is refilled by the next item
  }
}

int64_t copy_grid(int64_t items, const DeviceInfo &dev) {
  const int64_t cap = int64_t(dev.sm_count) * 8;   // 8 blocks of 256 threads per SM
  return items < cap ? (items > 0 ? items : 1) : cap;
}

// The launch's own status (not an error left pending by earlier calls).
template <class Kernel, class... Args>
cudaError_t launch_copy(Kernel kernel, int64_t items, const DeviceInfo &dev, cudaStream_t stream,
                        Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(copy_grid(items, dev)), 1, 1);
  cfg.blockDim = dim3(kCopyThreads, 1, 1);
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

constexpr int kMaxDevices = 64;
constexpr uint64_t kPoolKeepBytes = uint64_t(256) << 20;
std::mutex g_pool_mutex;
cudaMemPool_t g_pool[kMaxDevices] = {};

cudaError_t device_pool(int dev, cudaMemPool_t *pool) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_pool_mutex);
  if (!g_pool[dev]) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t p = nullptr;
    cudaError_t e = cudaMemPoolCreate(&p, &props);
    if (e != cudaSuccess) return e;
    uint64_t keep = kPoolKeepBytes;
    e = cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep);
    if (e != cudaSuccess) {
      cudaMemPoolDestroy(p);
      return e;
    }
    g_pool[dev] = p;
  }
  *pool = g_pool[dev];
  return cudaSuccess;
}

}  // namespace

cudaError_t stage_rows(const float *src, int64_t ld_src, int64_t rows, int64_t cols, float *dst,
                       int64_t ld_dst, const DeviceInfo &dev, cudaStream_t stream) {
  const int64_t items = (cols + kCopyThreads - 1) / kCopyThreads *
                        ((rows + kCopyUnroll - 1) / kCopyUnroll);
  return launch_copy(stage_rows_kernel, items, dev, stream, src, ld_src, rows, cols, dst, ld_dst);
}

cudaError_t stage_transpose(const float *src, int64_t ld_src, int64_t rows, int64_t cols,
                            float *dst, int64_t ld_dst, const DeviceInfo &dev,
                            cudaStream_t stream) {
  const int64_t items = ((rows + kTile - 1) / kTile) * ((cols + kTile - 1) / kTile);
  return launch_copy(stage_transpose_kernel, items, dev, stream, src, ld_src, rows, cols, dst,
                     ld_dst);
}

cudaError_t scratch_alloc(void **ptr, size_t bytes, const DeviceInfo &dev, cudaStream_t stream) {
  *ptr = nullptr;
  cudaMemPool_t pool;
  cudaError_t e = device_pool(dev.id, &pool);
  if (e == cudaSuccess) e = cudaMallocFromPoolAsync(ptr, bytes, pool, stream);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();   // a failed allocation is reported here, not to later calls
    *ptr = nullptr;
  }
  return e;
}

cudaError_t scratch_free(void *ptr, cudaStream_t stream) {
  return ptr ? cudaFreeAsync(ptr, stream) : cudaSuccess;
}

cudaError_t stage_device_status(unsigned int *status, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(status, g_stage_status, sizeof(unsigned int));
  if (e != cudaSuccess || !clear) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_stage_status, &zero, sizeof(unsigned int));
}

}  // namespace tmm
