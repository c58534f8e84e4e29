// reduce_softmax.cu -- the tiled reduction and the row softmax.
//
// "Tiling Strategies", section 5 ("Tiling Beyond GEMM"), lists two kernels
// beside GEMM that tile their input: a reduction, whose input is cut into
// chunks with partial sums kept in shared memory, and a softmax, which makes
// two passes over the same data (the maximum, then the normalisation) and so
// should hold that data on chip between them.  Section 4's table gives a
// reduction one tile per block of 256-1024 threads.  Both are bound by HBM
// bandwidth on GB300: each input value is read from HBM once.
//
// Array sum (sum_f32): two launches, no atomics, so the result is the same bits
// on every call.
//   1. sum_partials_kernel: a grid of G <= max(4 x SMs, 512) blocks of 512
//      threads.  Thread g of the P = 512 G threads adds, in its four lanes, the
//      16-byte vectors g, g + P, g + 2P, ... of the 16-byte-aligned body (four
//      streaming loads in flight per step).  Of the at most six leading and
//      trailing scalars outside the body, thread g < 6 takes one first.  The
//      lanes combine pairwise, the block reduces (warp shuffles, then one
//      value per warp through shared memory), and block b writes partials[b].
//   2. sum_final_kernel: one block of 1024 threads reduces the G partials.
//   Every value passes through at most ceil(n / 2^20) + 28 additions on its way
//   to the result (P >= 2^18 whenever the grid is capped).
//
// Row softmax (softmax_rows_f32): y_{r,j} = e^{x_{r,j} - m_r} / sum_k e^{x_{r,k} - m_r}
// with m_r the row maximum.  Which unit owns a row depends on its length:
//   * cols <= 1024: one warp per row, the row in the warp's registers
//     (lane l holds columns l, l + 32, ...); shuffles reduce max and sum.
//   * cols <= 49152: one block per row (128-1024 threads by length).  Pass 1
//     copies the row into shared memory (16-byte streaming loads when the rows
//     are 16-byte aligned) while taking the maximum; pass 2 replaces each
//     staged value by e^{x - m} and sums them; the stores scale by 1 / s.
//     Each thread touches only its own staged columns, so consecutive rows
//     need no barrier on the staging buffer, only on the reduction scratch.
//   * longer rows: one block of 1024 threads per row, three passes over
//     global memory (max, sum, normalise); the second and third reads of a row
//     come from L2 when the rows in flight fit there.
// Arithmetic: t = fl(x - m), e = expf(t) (CUDA's, within 2 ulp), s summed in
// FP32 (each thread in ascending column order, then a shuffle tree), y = e * fl(1/s).
// y may be x itself (in place): every row is read completely before any of its
// outputs is written, and only coherent loads are used.
#include <atomic>
#include <cmath>
#include <cstdint>

#include "tmm_internal.h"

namespace tmm {
namespace {

// ------------------------------------------------------------------ reductions

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;   // identical in every lane: each step adds the same two values in both lanes
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide sum or max; every thread gets the result.  scratch holds 32 floats.
// Contains two barriers: all threads of the block must call it.
template <bool kMax>
__device__ __forceinline__ float block_reduce(float v, float *scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = kMax ? warp_max(v) : warp_sum(v);
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  const int nwarps = blockDim.x >> 5;
  float w = lane < nwarps ? scratch[lane] : (kMax ? -INFINITY : 0.0f);
  w = kMax ? warp_max(w) : warp_sum(w);
  __syncthreads();   // scratch may be rewritten by the next call
  return w;
}

// ------------------------------------------------------------------ array sum

constexpr int kSumThreads = 512;
constexpr int kSumFinalThreads = kSumMaxPartials;   // one partial per thread

__global__ void __launch_bounds__(kSumThreads)
sum_partials_kernel(int64_t nvec, const float4 *__restrict__ body, const float *__restrict__ x,
                    int head, int64_t tail_at, int tail, float *__restrict__ partials) {
  __shared__ float scratch[32];
  const int64_t P = int64_t(gridDim.x) * kSumThreads;
  const int64_t g = int64_t(blockIdx.x) * kSumThreads + threadIdx.x;
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  if (g < head) acc.x = x[g];
  else if (g < head + tail) acc.x = x[tail_at + (g - head)];
  int64_t v = g;
  for (; v + 3 * P < nvec; v += 4 * P) {
    const float4 a = __ldcs(body + v);
    const float4 b = __ldcs(body + v + P);
    const float4 c = __ldcs(body + v + 2 * P);
    const float4 d = __ldcs(body + v + 3 * P);
    acc.x += a.x; acc.y += a.y; acc.z += a.z; acc.w += a.w;
    acc.x += b.x; acc.y += b.y; acc.z += b.z; acc.w += b.w;
    acc.x += c.x; acc.y += c.y; acc.z += c.z; acc.w += c.w;
    acc.x += d.x; acc.y += d.y; acc.z += d.z; acc.w += d.w;
  }
  for (; v < nvec; v += P) {
    const float4 a = __ldcs(body + v);
    acc.x += a.x; acc.y += a.y; acc.z += a.z; acc.w += a.w;
  }
  const float s = block_reduce<false>((acc.x + acc.y) + (acc.z + acc.w), scratch);
  if (threadIdx.x == 0) partials[blockIdx.x] = s;
}

__global__ void __launch_bounds__(kSumFinalThreads)
sum_final_kernel(int G, const float *__restrict__ partials, float *__restrict__ out) {
  __shared__ float scratch[32];
  const float v = int(threadIdx.x) < G ? partials[threadIdx.x] : 0.0f;
  const float s = block_reduce<false>(v, scratch);
  if (threadIdx.x == 0) *out = s;
}

// ------------------------------------------------------------------ softmax

constexpr int kWarpRowThreads = 256;      // 8 rows at a time per block

template <int kPer>   // columns per lane: cols <= 32 kPer
__global__ void __launch_bounds__(kWarpRowThreads)
softmax_warp_kernel(int64_t rows, int cols, const float *x, int64_t ldx, float *y, int64_t ldy) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = int64_t(gridDim.x) * (kWarpRowThreads / 32);
  for (int64_t r = int64_t(blockIdx.x) * (kWarpRowThreads / 32) + (threadIdx.x >> 5); r < rows;
       r += warps) {
    const float *xr = x + r * ldx;
    float *yr = y + r * ldy;
    float v[kPer];
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int j = lane + 32 * i;
      v[i] = j < cols ? __ldcs(xr + j) : -INFINITY;
      m = fmaxf(m, v[i]);
    }
    m = warp_max(m);
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int j = lane + 32 * i;
      v[i] = j < cols ? expf(v[i] - m) : 0.0f;
      s += v[i];
    }
    s = warp_sum(s);
    const float inv = 1.0f / s;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int j = lane + 32 * i;
      if (j < cols) __stcs(yr + j, v[i] * inv);
    }
  }
}

// One block per row, the row staged in shared memory.  kVec: rows start on
// 16-byte boundaries (x, y 16-byte aligned, ldx and ldy multiples of 4).
template <int kThreads, bool kVec>
__global__ void __launch_bounds__(kThreads)
softmax_staged_kernel(int64_t rows, int cols, const float *x, int64_t ldx, float *y,
                      int64_t ldy) {
  extern __shared__ __align__(16) float row[];
  __shared__ float scratch[32];
  const int t = threadIdx.x;
  const int nv = kVec ? cols >> 2 : 0;     // 16-byte vectors of the row
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const float *xr = x + r * ldx;
    float *yr = y + r * ldy;
    // Pass 1: stage the row, taking the maximum on the way.
    float m = -INFINITY;
    for (int q = t; q < nv; q += kThreads) {
      const float4 a = __ldcs(reinterpret_cast<const float4 *>(xr) + q);
      reinterpret_cast<float4 *>(row)[q] = a;
      m = fmaxf(fmaxf(m, fmaxf(a.x, a.y)), fmaxf(a.z, a.w));
    }
    for (int j = 4 * nv + t; j < cols; j += kThreads) {
      const float a = __ldcs(xr + j);
      row[j] = a;
      m = fmaxf(m, a);
    }
    m = block_reduce<true>(m, scratch);
    // Pass 2: exponentials in place, and their sum.
    float s = 0.0f;
    for (int q = t; q < nv; q += kThreads) {
      float4 a = reinterpret_cast<float4 *>(row)[q];
      a.x = expf(a.x - m); s += a.x;
      a.y = expf(a.y - m); s += a.y;
      a.z = expf(a.z - m); s += a.z;
      a.w = expf(a.w - m); s += a.w;
      reinterpret_cast<float4 *>(row)[q] = a;
    }
    for (int j = 4 * nv + t; j < cols; j += kThreads) {
      const float e = expf(row[j] - m);
      row[j] = e;
      s += e;
    }
    s = block_reduce<false>(s, scratch);
    const float inv = 1.0f / s;
    for (int q = t; q < nv; q += kThreads) {
      float4 a = reinterpret_cast<const float4 *>(row)[q];
      a.x *= inv; a.y *= inv; a.z *= inv; a.w *= inv;
      __stcs(reinterpret_cast<float4 *>(yr) + q, a);
    }
    for (int j = 4 * nv + t; j < cols; j += kThreads) __stcs(yr + j, row[j] * inv);
  }
}

constexpr int kLongRowThreads = 1024;

// Rows too long to stage: three passes over global memory.
__global__ void __launch_bounds__(kLongRowThreads)
softmax_long_kernel(int64_t rows, int cols, const float *x, int64_t ldx, float *y,
                    int64_t ldy) {
  __shared__ float scratch[32];
  const int t = threadIdx.x;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const float *xr = x + r * ldx;
    float *yr = y + r * ldy;
    float m = -INFINITY;
    for (int j = t; j < cols; j += kLongRowThreads) m = fmaxf(m, xr[j]);
    m = block_reduce<true>(m, scratch);
    float s = 0.0f;
    for (int j = t; j < cols; j += kLongRowThreads) s += expf(xr[j] - m);
    s = block_reduce<false>(s, scratch);
    const float inv = 1.0f / s;
    // Same thread, same columns, same order as the sum: every x_j is read
    // before this thread writes y_j, so y may be x.
    for (int j = t; j < cols; j += kLongRowThreads) yr[j] = expf(xr[j] - m) * inv;
  }
}

// Per-device launch facts for one kernel instantiation, set up on first use.
struct KernelSetup {
  std::atomic<uint64_t> configured{0};
  std::atomic<int> blocks_per_sm[64];
};

template <class Kernel>
cudaError_t blocks_per_sm(KernelSetup &st, Kernel kernel, int threads, int smem,
                          const DeviceInfo &dev, int *out) {
  const uint64_t bit = uint64_t(1) << (dev.id & 63);
  if (!(st.configured.load(std::memory_order_acquire) & bit)) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kMaxStagedRowBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    st.configured.fetch_or(bit, std::memory_order_release);
  }
  int nb = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, threads, smem);
  if (e != cudaSuccess) return e;
  *out = nb > 0 ? nb : 1;
  return cudaSuccess;
}

template <int kThreads, bool kVec>
cudaError_t launch_staged(int64_t rows, int cols, const float *x, int64_t ldx, float *y,
                          int64_t ldy, const DeviceInfo &dev, cudaStream_t stream) {
  static KernelSetup st;
  auto kernel = softmax_staged_kernel<kThreads, kVec>;
  const int smem = ((cols + 3) & ~3) * int(sizeof(float));
  int nb = 1;
  cudaError_t e = blocks_per_sm(st, kernel, kThreads, smem, dev, &nb);
  if (e != cudaSuccess) return e;
  const int64_t grid = std::min<int64_t>(rows, int64_t(dev.sm_count) * nb);
  kernel<<<unsigned(grid), kThreads, smem, stream>>>(rows, cols, x, ldx, y, ldy);
  return cudaGetLastError();
}

template <int kThreads>
cudaError_t launch_staged_any(int64_t rows, int cols, const float *x, int64_t ldx, float *y,
                              int64_t ldy, bool vec, const DeviceInfo &dev,
                              cudaStream_t stream) {
  return vec ? launch_staged<kThreads, true>(rows, cols, x, ldx, y, ldy, dev, stream)
             : launch_staged<kThreads, false>(rows, cols, x, ldx, y, ldy, dev, stream);
}

template <int kPer>
cudaError_t launch_warp_rows(int64_t rows, int cols, const float *x, int64_t ldx, float *y,
                             int64_t ldy, const DeviceInfo &dev, cudaStream_t stream) {
  constexpr int kRowsPerBlock = kWarpRowThreads / 32;
  const int64_t blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  const int64_t grid = std::min<int64_t>(blocks, int64_t(dev.sm_count) * 8);
  softmax_warp_kernel<kPer><<<unsigned(grid), kWarpRowThreads, 0, stream>>>(rows, cols, x, ldx,
                                                                           y, ldy);
  return cudaGetLastError();
}

}  // namespace

int64_t sum_grid_blocks(int64_t n, const DeviceInfo &dev) {
  const int64_t per_block = int64_t(kSumThreads) * 4 * 4;   // four vectors per thread
  const int64_t cap = std::max<int64_t>(int64_t(dev.sm_count) * 4, 512);
  return std::max<int64_t>(1, std::min<int64_t>((n + per_block - 1) / per_block,
                                                std::min<int64_t>(cap, kSumFinalThreads)));
}

cudaError_t launch_sum(int64_t n, const float *x, float *out, float *partials,
                       const DeviceInfo &dev, cudaStream_t stream) {
  if (n == 0) return cudaMemsetAsync(out, 0, sizeof(float), stream);
  const uintptr_t addr = reinterpret_cast<uintptr_t>(x);
  const int64_t head = std::min<int64_t>(n, int64_t(((16 - (addr & 15)) & 15) >> 2));
  const int64_t nvec = (n - head) >> 2;
  const int64_t tail_at = head + 4 * nvec;
  const int tail = int(n - tail_at);
  const int G = int(sum_grid_blocks(n, dev));
  sum_partials_kernel<<<G, kSumThreads, 0, stream>>>(
      nvec, reinterpret_cast<const float4 *>(x + head), x, int(head), tail_at, tail, partials);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  sum_final_kernel<<<1, kSumFinalThreads, 0, stream>>>(G, partials, out);
  return cudaGetLastError();
}

cudaError_t launch_softmax_rows(int64_t rows, int cols, const float *x, int64_t ldx, float *y,
                                int64_t ldy, const DeviceInfo &dev, cudaStream_t stream) {
  if (cols <= 32) return launch_warp_rows<1>(rows, cols, x, ldx, y, ldy, dev, stream);
  if (cols <= 64) return launch_warp_rows<2>(rows, cols, x, ldx, y, ldy, dev, stream);
  if (cols <= 128) return launch_warp_rows<4>(rows, cols, x, ldx, y, ldy, dev, stream);
  if (cols <= 256) return launch_warp_rows<8>(rows, cols, x, ldx, y, ldy, dev, stream);
  if (cols <= 512) return launch_warp_rows<16>(rows, cols, x, ldx, y, ldy, dev, stream);
  if (cols <= 1024) return launch_warp_rows<32>(rows, cols, x, ldx, y, ldy, dev, stream);
  if (cols <= kMaxStagedRowBytes / int(sizeof(float))) {
    const bool vec = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15u) ==
                         0 &&
                     (ldx & 3) == 0 && (ldy & 3) == 0;
    if (cols <= 2048) return launch_staged_any<128>(rows, cols, x, ldx, y, ldy, vec, dev, stream);
    if (cols <= 8192) return launch_staged_any<256>(rows, cols, x, ldx, y, ldy, vec, dev, stream);
    if (cols <= 16384)
      return launch_staged_any<512>(rows, cols, x, ldx, y, ldy, vec, dev, stream);
    return launch_staged_any<1024>(rows, cols, x, ldx, y, ldy, vec, dev, stream);
  }
  const int64_t grid = std::min<int64_t>(rows, int64_t(dev.sm_count) * 2);
  softmax_long_kernel<<<unsigned(grid), kLongRowThreads, 0, stream>>>(rows, cols, x, ldx, y, ldy);
  return cudaGetLastError();
}

}  // namespace tmm
