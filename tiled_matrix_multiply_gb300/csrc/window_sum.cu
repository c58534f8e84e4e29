// window_sum.cu -- valid sliding-window sums with cooperative shared-memory staging.
//
// "CMU DLSys Lecture 12: GPU Acceleration", section 3: for n outputs and an
// input of n + W - 1 elements, y_i = sum_{d=0}^{W-1} x_{i+d}.  Neighbouring
// outputs share W - 1 of their inputs, so a block stages its tile of T inputs
// plus the W - 1 halo values once in shared memory, synchronises, and lets
// every thread read its windows there: T + W - 1 global loads instead of
// T W, the ratio T W / (T + W - 1) the page derives.  Every thread reaches
// the barriers; only the output stores are guarded (the page's rule).
//
// GB300 layout: the work is bound by HBM bandwidth (8 bytes moved per
// output), so the kernel is shaped for bandwidth, not arithmetic:
//   * tiles of T = 256 x 16 = 4096 outputs; a grid of a few blocks per SM
//     strides over them.  Each block stages its tiles with cp.async (16-byte
//     copies when x is 16-byte aligned) two buffers deep: the next tile's
//     copies are in flight while this one is summed (the halo is re-read by
//     the next tile, an L2 hit);
//   * thread t owns outputs t, t + 256, ..., so a warp's shared-memory reads
//     and global stores are consecutive words (no bank conflicts, full
//     128-byte store lines);
//   * each sum starts from 0 and adds x_{i+d} in ascending d in FP32, the
//     page's order, so results equal that sequence of roundings exactly.
#include <atomic>
#include <cstdint>

#include "tmm_internal.h"

namespace tmm {
namespace {

constexpr int kWinThreads = 256;
constexpr int kWinItems = 16;
constexpr int kWinTile = kWinThreads * kWinItems;   // outputs per tile
constexpr int kWinMaxHalo = kMaxWindow - 1;
constexpr int kWinBuf = kWinTile + kWinMaxHalo + 4;  // floats per staging buffer (16-byte multiple)
constexpr int kWinSmemBytes = 2 * kWinBuf * int(sizeof(float));

__device__ __forceinline__ void win_cp16(float *dst, const float *src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(src) : "memory");
}

__device__ __forceinline__ void win_cp4(float *dst, const float *src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(d), "l"(src) : "memory");
}

__device__ __forceinline__ void win_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }

template <int N>
__device__ __forceinline__ void win_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

template <int kW>   // kW > 0: compile-time width; 0: runtime width
__global__ void __launch_bounds__(kWinThreads)
window_sum_kernel(int64_t n, int W_rt, const float *__restrict__ x, float *__restrict__ y,
                  int vec) {
  extern __shared__ __align__(16) float stage[];   // two buffers of kWinBuf floats
  const int W = kW > 0 ? kW : W_rt;
  const int64_t len = n + W - 1;                  // valid input elements
  const int64_t tiles = (n + kWinTile - 1) / kWinTile;
  const int need = kWinTile + W - 1;              // staged elements of a tile
  const int t = threadIdx.x;
  // Copy tile tl's inputs (the tile and its halo; nothing past the input's end:
  // those slots only feed outputs >= n, which are not stored).
  auto copy_tile = [&](float *buf, int64_t tl) {
    const int64_t base = tl * kWinTile;
    const int64_t rem = len - base;
    const int avail = rem < need ? int(rem) : need;
    if (vec) {
      const int nv = avail >> 2;
      for (int q = t; q < nv; q += kWinThreads) win_cp16(buf + 4 * q, x + base + 4 * q);
      for (int j = 4 * nv + t; j < avail; j += kWinThreads) win_cp4(buf + j, x + base + j);
    } else {
      for (int j = t; j < avail; j += kWinThreads) win_cp4(buf + j, x + base + j);
    }
  };
  int64_t tl = blockIdx.x;
  if (tl < tiles) copy_tile(stage, tl);
  win_commit();
  for (int it = 0; tl < tiles; tl += gridDim.x, ++it) {
    const float *tile = stage + (it & 1) * kWinBuf;
    const int64_t next = tl + gridDim.x;
    // The other buffer was last read before the barrier that ended the previous tile.
    if (next < tiles) copy_tile(stage + ((it + 1) & 1) * kWinBuf, next);
    win_commit();
    win_wait<1>();       // this thread's copies of tile tl have landed ...
    __syncthreads();     // ... and every thread's
    const int64_t base = tl * kWinTile;
#pragma unroll 4
    for (int j = 0; j < kWinItems; ++j) {
      const int o = j * kWinThreads + t;
      float s = 0.0f;
      if (kW > 0) {
#pragma unroll
        for (int d = 0; d < kW; ++d) s += tile[o + d];
      } else {
        for (int d = 0; d < W; ++d) s += tile[o + d];
      }
      if (base + o < n) __stcs(y + base + o, s);
    }
    __syncthreads();     // every thread is done with this buffer before it is refilled
  }
  win_wait<0>();
}

template <int kW>
cudaError_t launch_width(int64_t n, int W, const float *x, float *y, int vec,
                         const DeviceInfo &dev, cudaStream_t stream) {
  static std::atomic<uint64_t> configured{0};
  auto kernel = window_sum_kernel<kW>;
  const uint64_t bit = uint64_t(1) << (dev.id & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kWinSmemBytes);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_release);
  }
  int nb = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, kWinThreads,
                                                                kWinSmemBytes);
  if (e != cudaSuccess) return e;
  const int64_t tiles = (n + kWinTile - 1) / kWinTile;
  const int64_t grid = std::min<int64_t>(tiles, int64_t(dev.sm_count) * (nb > 0 ? nb : 1));
  kernel<<<unsigned(grid), kWinThreads, kWinSmemBytes, stream>>>(n, W, x, y, vec);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_window_sum(int64_t n, int W, const float *x, float *y,
                              const DeviceInfo &dev, cudaStream_t stream) {
  const int vec = (reinterpret_cast<uintptr_t>(x) & 15u) == 0 ? 1 : 0;
  // Widths up to 17 with the window unrolled at compile time; wider ones loop.
  switch (W) {
    case 2: return launch_width<2>(n, W, x, y, vec, dev, stream);
    case 3: return launch_width<3>(n, W, x, y, vec, dev, stream);
    case 4: return launch_width<4>(n, W, x, y, vec, dev, stream);
    case 5: return launch_width<5>(n, W, x, y, vec, dev, stream);
    case 7: return launch_width<7>(n, W, x, y, vec, dev, stream);
    case 9: return launch_width<9>(n, W, x, y, vec, dev, stream);
    case 11: return launch_width<11>(n, W, x, y, vec, dev, stream);
    case 13: return launch_width<13>(n, W, x, y, vec, dev, stream);
    case 15: return launch_width<15>(n, W, x, y, vec, dev, stream);
    case 17: return launch_width<17>(n, W, x, y, vec, dev, stream);
    default: return launch_width<0>(n, W, x, y, vec, dev, stream);
  }
}

}  // namespace tmm
