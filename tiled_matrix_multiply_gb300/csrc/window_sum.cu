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
//     strides over them.  Each block stages its tiles two buffers deep, the
//     next tile's copy in flight while this one is summed (the halo is re-read
//     by the next tile, an L2 hit): one bulk copy (the TMA unit's
//     cp.async.bulk, counted on an mbarrier) per tile when x is 16-byte
//     aligned, 4-byte cp.async copies by every thread otherwise;
//   * with a compile-time width and y 16-byte aligned, thread t owns groups of
//     four consecutive outputs (4 g .. 4 g + 3, g = t, t + 256, ...), reads
//     their inputs as ceil((W + 3) / 4) 16-byte vectors and stores the four
//     sums with one 16-byte store: a warp's reads and stores are consecutive
//     vectors (no bank conflicts, whole 128-byte lines), with a fifth of the
//     shared-memory reads of one output per thread at W = 5; otherwise thread
//     t owns outputs t, t + 256, ... (consecutive words per warp);
//   * each sum starts from 0 and adds x_{i+d} in ascending d in FP32, the
//     page's order, so results equal that sequence of roundings exactly.
#include <atomic>
#include <cstdint>

#include "tmm_internal.h"

namespace tmm {

// Device status word (bit 0: a bounded wait for a bulk copy ran out of time).
__device__ unsigned int g_win_status;

namespace {

constexpr int kWinThreads = 256;
constexpr int kWinItems = 16;
constexpr int kWinTile = kWinThreads * kWinItems;   // outputs per tile
static_assert(kWinItems % 4 == 0, "whole groups of four outputs per thread");
constexpr int kWinMaxHalo = kMaxWindow - 1;
constexpr int kWinBuf = kWinTile + kWinMaxHalo + 4;  // floats per staging buffer (16-byte multiple)
constexpr int kWinSmemBytes = 2 * kWinBuf * int(sizeof(float));

__device__ __forceinline__ void win_cp4(float *dst, const float *src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(d), "l"(src) : "memory");
}

__device__ __forceinline__ void win_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }

__device__ __forceinline__ void win_bar_init(uint32_t bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
}
// One bulk copy of `bytes` (a multiple of 16) from global to shared memory,
// counted on `bar`, which this thread arms for exactly those bytes.
// `expect` is the byte count the barrier is armed for (bytes, except under the
// testing hook that makes one block wait for bytes that never come).
__device__ __forceinline__ void win_bulk(float *dst, const float *src, uint32_t bytes,
                                         uint32_t expect, uint32_t bar) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(expect)
               : "memory");
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(d),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ bool win_bar_try(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
// Bounded wait for phase `parity`; false after limit_ns.
__device__ __forceinline__ bool win_bar_wait(uint32_t bar, uint32_t parity, int64_t limit_ns) {
  if (win_bar_try(bar, parity)) return true;
  uint64_t t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (;;) {
    if (win_bar_try(bar, parity)) return true;
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (int64_t(t - t0) > limit_ns) return false;
  }
}

template <int N>
__device__ __forceinline__ void win_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

template <int kW>   // kW > 0: compile-time width; 0: runtime width
__global__ void __launch_bounds__(kWinThreads)
window_sum_kernel(int64_t n, int W_rt, const float *__restrict__ x, float *__restrict__ y,
                  int vec, int yvec, int64_t wait_limit_ns, int drop_block,
                  unsigned long long *tilectr) {
  extern __shared__ __align__(16) float stage[];   // two buffers of kWinBuf floats
  __shared__ __align__(8) uint64_t bars[2];         // bulk copies into buffer b (vec)
  __shared__ long long s_next;
  const int W = kW > 0 ? kW : W_rt;
  const int64_t len = n + W - 1;                  // valid input elements
  const int64_t tiles = (n + kWinTile - 1) / kWinTile;
  const int need = kWinTile + W - 1;              // staged elements of a tile
  const int t = threadIdx.x;
  // Copy tile tl's inputs (the tile and its halo; nothing past the input's end:
  // those slots only feed outputs >= n, which are not stored).
  // With x 16-byte aligned (vec), one thread moves the whole 16-byte-aligned
  // part with a single bulk copy counted on the buffer's barrier, and the at
  // most three elements after it are plain loads (seen by the other threads
  // after the barrier that precedes the tile's use).  Otherwise every thread
  // issues 4-byte asynchronous copies.
  const uint32_t bar0 = static_cast<uint32_t>(__cvta_generic_to_shared(&bars[0]));
  if (vec && t == 0) {
    win_bar_init(bar0);
    win_bar_init(bar0 + 8);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (vec) __syncthreads();
  auto copy_tile = [&](int b, int64_t tl) {
    float *buf = stage + b * kWinBuf;
    const int64_t base = tl * kWinTile;
    const int64_t rem = len - base;
    const int avail = rem < need ? int(rem) : need;
    if (vec) {
      const int body = avail & ~3;
      if (t == 0) {
        const uint32_t bar = bar0 + 8u * uint32_t(b);
        const uint32_t bytes = uint32_t(body) * 4u;
        // Testing hook: block drop_block waits for 16 bytes more than its first copy brings.
        const uint32_t extra = (int(blockIdx.x) == drop_block && tl == blockIdx.x) ? 16u : 0u;
        if (body > 0) win_bulk(buf, x + base, bytes, bytes + extra, bar);
        else asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
      }
      if (t < avail - body) buf[body + t] = x[base + body + t];
    } else {
      for (int j = t; j < avail; j += kWinThreads) win_cp4(buf + j, x + base + j);
    }
  };
  bool timed_out = false;
  int stop_it = -1;            // the iteration a timeout ended (vec)
  bool next_issued = false;
  // Tiles: a block's first is its index; with a tile counter each later one is
  // taken from it while the block works on the one before, so blocks the warp
  // schedulers favour take more tiles and all finish together.
  const bool dyn = tilectr != nullptr;
  int64_t tl = blockIdx.x;
  int64_t next = tl + gridDim.x;   // the tile after tl
  if (dyn) {
    if (t == 0) s_next = (long long)(gridDim.x + atomicAdd(&tilectr[0], 1ull));
    __syncthreads();
    next = s_next;
  }
  if (tl < tiles) copy_tile(0, tl);
  win_commit();
  for (int it = 0; tl < tiles; ++it) {
    const float *tile = stage + (it & 1) * kWinBuf;
    // The tile after next: taken now, its number needed only after this tile.
    unsigned long long tok = 0;
    if (dyn && t == 0) tok = atomicAdd(&tilectr[0], 1ull);
    // The other buffer was last read before the barrier that ended the previous tile.
    next_issued = next < tiles;
    if (next_issued) copy_tile((it + 1) & 1, next);
    win_commit();
    if (vec) {
      if (!win_bar_wait(bar0 + 8u * uint32_t(it & 1), uint32_t(it >> 1) & 1u, wait_limit_ns))
        timed_out = true;
    } else {
      win_wait<1>();     // this thread's copies of tile tl have landed ...
    }
    if (__syncthreads_or(timed_out)) {   // ... and every thread's
      stop_it = it;
      break;
    }
    if (dyn && t == 0) s_next = (long long)(gridDim.x + tok);   // read after the last barrier
    const int64_t base = tl * kWinTile;
    if (kW > 0 && yvec) {
      // Thread t owns the groups of four outputs 4 g .. 4 g + 3, g = t, t + 256,
      // ...: their inputs are ceil((kW + 3) / 4) consecutive 16-byte vectors of
      // the tile (consecutive lanes, consecutive vectors: no bank conflicts),
      // and one 16-byte store writes the four sums.
      constexpr int kVecs = (kW + 3 + 3) / 4;
#pragma unroll
      for (int j = 0; j < kWinItems / 4; ++j) {
        const int g = j * kWinThreads + t;
        float v[4 * kVecs];
#pragma unroll
        for (int k = 0; k < kVecs; ++k) {
          const float4 a = reinterpret_cast<const float4 *>(tile)[g + k];
          v[4 * k] = a.x; v[4 * k + 1] = a.y; v[4 * k + 2] = a.z; v[4 * k + 3] = a.w;
        }
        float o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float s = 0.0f;
#pragma unroll
          for (int d = 0; d < kW; ++d) s += v[i + d];
          o[i] = s;
        }
        const int64_t i0 = base + 4 * g;
        if (i0 + 3 < n) {
          __stcs(reinterpret_cast<float4 *>(y + i0), make_float4(o[0], o[1], o[2], o[3]));
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (i0 + i < n) __stcs(y + i0 + i, o[i]);
        }
      }
    } else {
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
    }
    __syncthreads();     // every thread is done with this buffer before it is refilled
    const int64_t nn = dyn ? int64_t(s_next) : next + gridDim.x;
    tl = next;
    next = nn;
  }
  win_wait<0>();
  if (stop_it >= 0 && t == 0) {
    // Record the timeout, and give the bulk copies that may still be in flight
    // (this tile's and the next one's) a bounded time to land before the
    // block's shared memory goes away.
    atomicOr(&g_win_status, 1u);
    win_bar_wait(bar0 + 8u * uint32_t(stop_it & 1), uint32_t(stop_it >> 1) & 1u, wait_limit_ns);
    if (next_issued)
      win_bar_wait(bar0 + 8u * uint32_t((stop_it + 1) & 1), uint32_t((stop_it + 1) >> 1) & 1u,
                   wait_limit_ns);
  }
  if (dyn && t == 0 && atomicAdd(&tilectr[1], 1ull) == gridDim.x - 1ull) {
    // The last block done: every fetch has happened, so reset for the next call.
    tilectr[0] = 0;
    tilectr[1] = 0;
    __threadfence();
  }
}

std::atomic<int64_t> g_win_wait_limit_ns{int64_t(10) * 1000 * 1000 * 1000};
std::atomic<int> g_win_drop_block{-1};

// Tile counters, kWinRegions pairs (next tile, blocks done); each call takes
// the next pair, and its last block resets it (up to kWinRegions calls in flight).
constexpr int kWinRegions = 16;
__device__ unsigned long long g_win_tiles[kWinRegions][2];
std::atomic<unsigned int> g_win_epoch{0};

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
  const int yvec = (reinterpret_cast<uintptr_t>(y) & 15u) == 0 ? 1 : 0;
  // A tile counter where several blocks share an SM.
  unsigned long long *tilectr = nullptr;
  if (grid >= 2 * int64_t(dev.sm_count)) {
    e = cudaGetSymbolAddress(reinterpret_cast<void **>(&tilectr), g_win_tiles);
    if (e != cudaSuccess) return e;
    tilectr += 2 * (g_win_epoch.fetch_add(1, std::memory_order_relaxed) % kWinRegions);
  }
  kernel<<<unsigned(grid), kWinThreads, kWinSmemBytes, stream>>>(
      n, W, x, y, vec, yvec, g_win_wait_limit_ns.load(std::memory_order_relaxed),
      g_win_drop_block.load(std::memory_order_relaxed), tilectr);
  return cudaGetLastError();
}

}  // namespace

void window_set_test_hooks(int drop_block, int64_t wait_limit_ns) {
  g_win_drop_block.store(drop_block, std::memory_order_relaxed);
  g_win_wait_limit_ns.store(wait_limit_ns > 0 ? wait_limit_ns : int64_t(10) * 1000 * 1000 * 1000,
                            std::memory_order_relaxed);
}

cudaError_t window_device_status(unsigned int *status, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(status, g_win_status, sizeof(unsigned int));
  if (e != cudaSuccess || !clear) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_win_status, &zero, sizeof(unsigned int));
}

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
