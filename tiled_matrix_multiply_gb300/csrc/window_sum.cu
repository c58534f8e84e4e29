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
//     strides over them, each block staging its tile with 16-byte streaming
//     loads (the halo is re-read by the next tile, an L2 hit);
//   * thread t owns outputs t, t + 256, ..., so a warp's shared-memory reads
//     and global stores are consecutive words (no bank conflicts, full
//     128-byte store lines);
//   * each sum starts from 0 and adds x_{i+d} in ascending d in FP32, the
//     page's order, so results equal that sequence of roundings exactly.
#include <cstdint>

#include "tmm_internal.h"

namespace tmm {
namespace {

constexpr int kWinThreads = 256;
constexpr int kWinItems = 16;
constexpr int kWinTile = kWinThreads * kWinItems;   // outputs per tile
constexpr int kWinMaxHalo = kMaxWindow - 1;

template <int kW>   // kW > 0: compile-time width; 0: runtime width
__global__ void __launch_bounds__(kWinThreads)
window_sum_kernel(int64_t n, int W_rt, const float *__restrict__ x, float *__restrict__ y,
                  int vec) {
  __shared__ __align__(16) float tile[kWinTile + kWinMaxHalo + 4];
  const int W = kW > 0 ? kW : W_rt;
  const int64_t len = n + W - 1;                  // valid input elements
  const int64_t tiles = (n + kWinTile - 1) / kWinTile;
  const int t = threadIdx.x;
  for (int64_t tl = blockIdx.x; tl < tiles; tl += gridDim.x) {
    const int64_t base = tl * kWinTile;
    const int need = kWinTile + W - 1;            // staged elements of this tile
    // Cooperative load: 16-byte vectors where the whole vector is inside the
    // input, single elements otherwise (zero beyond the end, never used).
    if (vec) {
      for (int q = 4 * t; q < need; q += 4 * kWinThreads) {
        const int64_t g = base + q;
        if (g + 4 <= len) {
          const float4 v = __ldcs(reinterpret_cast<const float4 *>(x + g));
          *reinterpret_cast<float4 *>(&tile[q]) = v;
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) tile[q + j] = g + j < len ? x[g + j] : 0.0f;
        }
      }
    } else {
      for (int q = t; q < need; q += kWinThreads) {
        const int64_t g = base + q;
        tile[q] = g < len ? x[g] : 0.0f;
      }
    }
    __syncthreads();
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
    __syncthreads();   // the next tile overwrites the staging buffer
  }
}

}  // namespace

cudaError_t launch_window_sum(int64_t n, int W, const float *x, float *y,
                              const DeviceInfo &dev, cudaStream_t stream) {
  const int64_t tiles = (n + kWinTile - 1) / kWinTile;
  const int64_t grid = std::min<int64_t>(tiles, int64_t(dev.sm_count) * 8);
  const int vec = (reinterpret_cast<uintptr_t>(x) & 15u) == 0 ? 1 : 0;
  if (W == 5)
    window_sum_kernel<5><<<unsigned(grid), kWinThreads, 0, stream>>>(n, W, x, y, vec);
  else if (W == 3)
    window_sum_kernel<3><<<unsigned(grid), kWinThreads, 0, stream>>>(n, W, x, y, vec);
  else
    window_sum_kernel<0><<<unsigned(grid), kWinThreads, 0, stream>>>(n, W, x, y, vec);
  return cudaGetLastError();
}

}  // namespace tmm
