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
// Array sum (sum_f32): two launches, and a fixed order of additions, so the
// result is the same bits on every call.
//   1. sum_partials_kernel: the 16-byte-aligned body is cut into G <= 16384
//      chunks of V >= 8192 vectors (V a multiple of 2048); resident blocks of
//      512 threads take chunks from a counter, and partials[c] receives chunk
//      c's sum: thread t adds, in its four lanes, the chunk's vectors t,
//      t + 512, ... (four streaming loads in flight per step), the lanes
//      combine pairwise and the block reduces (warp shuffles, then one value
//      per warp through shared memory).
//   2. sum_final_kernel: one block of 1024 threads; thread t takes one of the
//      at most six scalars outside the body (t < 6), adds partials t,
//      t + 1024, ... in order, and the block reduces.
//   Every value passes through at most V / 512 + ceil(G / 1024) + 22 <=
//   ceil(n / 2^25) + 54 additions on its way to the result.
//
// Row softmax (softmax_rows_f32): y_{r,j} = e^{x_{r,j} - m_r} / sum_k e^{x_{r,k} - m_r}
// with m_r the row maximum.  Rows of up to 65536 columns are read from HBM once
// and written once; what holds them on chip between the two passes depends on
// their length:
//   * up to 2048 columns (rows on 16-byte boundaries, cols % 4 == 0; 1024
//     otherwise): a group of 1-32 lanes per row, the row in registers (lane s
//     holds columns or 16-byte vectors s, s + group, ...); group shuffles
//     reduce max and sum.  Short rows share a warp (32 / group rows at once).
//   * up to 16384 columns: one block per row.  The row is copied into shared
//     memory with cp.async, two buffers deep, so the next row's copies are in
//     flight while this one is reduced; pass 1 takes the maximum, pass 2
//     replaces each staged value by e^{x - m} and sums them, and the stores
//     scale by 1 / s.
//   * up to 65536 columns: a cluster of 2-8 blocks per row, each staging one
//     chunk, the partial maxima and sums combined through distributed shared
//     memory (softmax_staged_kernel describes the exchange).
//   * longer rows: G blocks per row of a cooperative grid, meeting through
//     global memory; each reads its columns twice, a running (maximum, sum)
//     pass and the normalise pass, whose reads come from L2 because the rows
//     in flight are sized to fit there (softmax_grid_kernel).
// Arithmetic: t = fl(x - m), e = expf(t) (CUDA's, within 2 ulp), s summed in
// FP32 in a fixed order (each thread in ascending column order, then a shuffle
// tree, then the cluster's chunks in rank order), y = e * fl(1 / s) (in a
// cluster, e^{x - m_c} * fl(e^{m_c - m} / s)).  Past 65536 columns the sum is
// a running one (each rise of a thread's maximum rescales its sum, one more
// product and one more expf), and the G parts merge in a fixed order.
// y may be x itself (in place): every row (chunk) is read completely before
// any of its outputs is written, and only coherent loads are used.
#include <atomic>
#include <cmath>
#include <cstdint>

#include <cooperative_groups.h>

#include "tmm_internal.h"

namespace cg = cooperative_groups;

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
constexpr int kSumFinalThreads = 1024;
constexpr int kSumChunkVecsMin = 8192;     // 16-byte vectors per chunk, at least (128 KiB)
static_assert(kSumChunkVecsMin % (4 * kSumThreads) == 0, "whole groups of four per thread");
constexpr int kSumRegions = 16;            // calls in flight at once, at most
__device__ unsigned long long g_sum_chunks[kSumRegions][2];   // (next chunk, blocks done)

// Chunk c of the body is vectors [c V, min((c + 1) V, nvec)).  A block takes
// its first chunk by its index and each later one from the counter (taken
// while it sums the one before, so the counter's latency is hidden): blocks
// that the warp schedulers favour take more chunks.  Thread t of the block
// adds, in its four lanes, the chunk's vectors t, t + 512, ... (four loads in
// flight per step); the lanes combine pairwise, the block reduces, and
// partials[c] holds the chunk's sum -- the same bits whichever block took it.
__global__ void __launch_bounds__(kSumThreads)
sum_partials_kernel(int64_t nvec, int64_t V, int64_t G, const float4 *__restrict__ body,
                    float *__restrict__ partials, unsigned long long *ctr) {
  __shared__ float scratch[32];
  __shared__ long long s_next;
  const int t = threadIdx.x;
  int64_t c = blockIdx.x;
  if (t == 0) s_next = (long long)(gridDim.x + atomicAdd(&ctr[0], 1ull));
  __syncthreads();
  int64_t cn = s_next;   // the chunk after c
  while (c < G) {
    unsigned long long tok = 0;
    if (t == 0) tok = atomicAdd(&ctr[0], 1ull);   // the chunk after cn
    const int64_t v0 = c * V;
    const int64_t v1 = v0 + V < nvec ? v0 + V : nvec;
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    int64_t v = v0 + t;
    for (; v + 3 * kSumThreads < v1; v += 4 * kSumThreads) {
      const float4 a = __ldcs(body + v);
      const float4 b = __ldcs(body + v + kSumThreads);
      const float4 cc = __ldcs(body + v + 2 * kSumThreads);
      const float4 d = __ldcs(body + v + 3 * kSumThreads);
      acc.x += a.x; acc.y += a.y; acc.z += a.z; acc.w += a.w;
      acc.x += b.x; acc.y += b.y; acc.z += b.z; acc.w += b.w;
      acc.x += cc.x; acc.y += cc.y; acc.z += cc.z; acc.w += cc.w;
      acc.x += d.x; acc.y += d.y; acc.z += d.z; acc.w += d.w;
    }
    for (; v < v1; v += kSumThreads) {
      const float4 a = __ldcs(body + v);
      acc.x += a.x; acc.y += a.y; acc.z += a.z; acc.w += a.w;
    }
    const float sum = block_reduce<false>((acc.x + acc.y) + (acc.z + acc.w), scratch);
    if (t == 0) {
      partials[c] = sum;
      s_next = (long long)(gridDim.x + tok);
    }
    __syncthreads();
    c = cn;
    cn = s_next;
    __syncthreads();   // every thread has read s_next before it is rewritten
  }
  if (t == 0 && atomicAdd(&ctr[1], 1ull) == gridDim.x - 1ull) {
    // The last block done: every fetch has happened, so reset for the next call.
    ctr[0] = 0;
    ctr[1] = 0;
    __threadfence();
  }
}

// Thread t adds the at most six scalars outside the body (thread t < head +
// tail takes one) and then partials t, t + 1024, ... in order; the block
// reduces (warp shuffles, then one value per warp through shared memory).
__global__ void __launch_bounds__(kSumFinalThreads)
sum_final_kernel(int64_t G, const float *__restrict__ partials, const float *__restrict__ x,
                 int head, int64_t tail_at, int tail, float *__restrict__ out) {
  __shared__ float scratch[32];
  const int t = threadIdx.x;
  float v = 0.0f;
  if (t < head) v = x[t];
  else if (t < head + tail) v = x[tail_at + (t - head)];
  for (int64_t k = t; k < G; k += kSumFinalThreads) v += partials[k];
  const float s = block_reduce<false>(v, scratch);
  if (t == 0) *out = s;
}

// ------------------------------------------------------------------ softmax

__device__ __forceinline__ void cp_async_16(float *dst, const float *src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_4(float *dst, const float *src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(d), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

constexpr int kWarpRowThreads = 256;      // 8 warps per block
constexpr int kMaxCluster = 16;           // blocks sharing one row, at most

template <int kW>   // max over each aligned group of kW lanes (a power of 2)
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
  for (int o = kW / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

template <int kW>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = kW / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Rows owned by groups of kW lanes (32 / kW rows per warp at a time), any
// alignment: lane s of a group holds columns s, s + kW, ... (cols <= kW kPer).
// The whole row stays in registers; group shuffles reduce max and sum.
template <int kW, int kPer>
__global__ void __launch_bounds__(kWarpRowThreads)
softmax_warp_kernel(int64_t rows, int cols, const float *x, int64_t ldx, float *y, int64_t ldy) {
  constexpr int kRowsPerWarp = 32 / kW;
  const int lane = threadIdx.x & 31, sub = lane % kW;
  const int64_t groups = (rows + kRowsPerWarp - 1) / kRowsPerWarp;
  const int64_t warps = int64_t(gridDim.x) * (kWarpRowThreads / 32);
  for (int64_t gi = int64_t(blockIdx.x) * (kWarpRowThreads / 32) + (threadIdx.x >> 5);
       gi < groups; gi += warps) {
    const int64_t r = gi * kRowsPerWarp + lane / kW;
    const bool live = r < rows;
    const float *xr = x + (live ? r : 0) * ldx;
    float v[kPer];
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int j = sub + kW * i;
      v[i] = (live && j < cols) ? __ldcs(xr + j) : -INFINITY;
      m = fmaxf(m, v[i]);
    }
    m = group_max<kW>(m);
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int j = sub + kW * i;
      v[i] = (live && j < cols) ? expf(v[i] - m) : 0.0f;
      s += v[i];
    }
    s = group_sum<kW>(s);
    const float inv = 1.0f / s;
    if (live) {
      float *yr = y + r * ldy;
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int j = sub + kW * i;
        if (j < cols) __stcs(yr + j, v[i] * inv);
      }
    }
  }
}

// The same with 16-byte accesses: rows start on 16-byte boundaries and
// cols % 4 == 0; lane s of a group holds vectors s, s + kW, ... (cols <= 4 kW kVec).
template <int kW, int kVec>
__global__ void __launch_bounds__(kWarpRowThreads)
softmax_warp_vec_kernel(int64_t rows, int cols, const float *x, int64_t ldx, float *y,
                        int64_t ldy) {
  constexpr int kRowsPerWarp = 32 / kW;
  const int lane = threadIdx.x & 31, sub = lane % kW;
  const int nv = cols >> 2;
  const int64_t groups = (rows + kRowsPerWarp - 1) / kRowsPerWarp;
  const int64_t warps = int64_t(gridDim.x) * (kWarpRowThreads / 32);
  for (int64_t gi = int64_t(blockIdx.x) * (kWarpRowThreads / 32) + (threadIdx.x >> 5);
       gi < groups; gi += warps) {
    const int64_t r = gi * kRowsPerWarp + lane / kW;
    const bool live = r < rows;
    const float4 *xr = reinterpret_cast<const float4 *>(x + (live ? r : 0) * ldx);
    const float4 none = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    float4 v[kVec];
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < kVec; ++i) {
      const int q = sub + kW * i;
      v[i] = (live && q < nv) ? __ldcs(xr + q) : none;
      m = fmaxf(fmaxf(m, fmaxf(v[i].x, v[i].y)), fmaxf(v[i].z, v[i].w));
    }
    m = group_max<kW>(m);
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < kVec; ++i) {
      const bool ok = live && sub + kW * i < nv;
      v[i].x = ok ? expf(v[i].x - m) : 0.0f; s += v[i].x;
      v[i].y = ok ? expf(v[i].y - m) : 0.0f; s += v[i].y;
      v[i].z = ok ? expf(v[i].z - m) : 0.0f; s += v[i].z;
      v[i].w = ok ? expf(v[i].w - m) : 0.0f; s += v[i].w;
    }
    s = group_sum<kW>(s);
    const float inv = 1.0f / s;
    if (live) {
      float4 *yr = reinterpret_cast<float4 *>(y + r * ldy);
#pragma unroll
      for (int i = 0; i < kVec; ++i) {
        const int q = sub + kW * i;
        if (q < nv)
          __stcs(yr + q, make_float4(v[i].x * inv, v[i].y * inv, v[i].z * inv, v[i].w * inv));
      }
    }
  }
}

// Rows shared by G blocks that meet through global memory (softmax_grid_kernel).
constexpr int kGridThreads = 512;
constexpr int kGridChunk = 32768;          // columns per block, at most (a multiple of 4)
constexpr int kGridMaxBlocks = 2048;       // blocks of one launch, at most
constexpr int kGridKeep = 4;               // vectors per thread kept in shared memory
constexpr int kGridRegions = 16;           // calls in flight at once, at most
__device__ unsigned int g_sm_counters[kGridRegions][2 * kGridMaxBlocks];
__device__ float2 g_sm_pairs[kGridRegions][2 * kGridMaxBlocks];
__device__ unsigned int g_softmax_status;

// How the G blocks sharing a row meet: block b takes part b % G of row unit
// b / G; U units are in flight.  Slot (it % 2) U + unit of a call's region
// holds a counter and G (maximum, sum) pairs.
struct RowExchange {
  int G, U;                  // blocks per row, rows in flight
  unsigned int *counters;    // 2 U row slots of this call's region, zeroed before launch
  float2 *pairs;             // 2 U x G partial (maximum, sum) pairs
  int64_t wait_limit_ns;
  int drop_block;            // testing hook: this block never counts itself in (-1: none)
};

struct GridRowsParams {
  int64_t rows;
  int cols, chunk;
  const float *x;
  int64_t ldx;
  float *y;
  int64_t ldy;
  RowExchange ex;
};

__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int *p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// The row's (m, s) from the pairs of the G blocks sharing it, for iteration
// `it` of row unit `unit`; (m, s) is this block's pair (needed in thread 0
// only).  Thread 0 stores the pair in the row's slot, counts the block in
// (fence, then an atomic increment) and waits (bounded) until all G blocks
// have; the first warp then merges the G pairs -- lane l takes parts l,
// l + 32, ... in order, then a fixed shuffle tree -- so every block of the row
// gets the same result.  Slots alternate between two sets by iteration
// parity, and a slot's counter grows by G per use: a block stores into a slot
// again only after the following row's wait, which every block of its row
// passes only after reading the slot.  On timeout thread 0 records bit 0 of
// g_softmax_status and stops waiting (the results are then not valid).  All
// threads must call; one barrier; *row_pair is rewritten by the next call, so
// the block must pass another barrier in between.
__device__ __forceinline__ float2 exchange_row_pair(const RowExchange &ex, int unit, int part,
                                                    int it, float m, float s, bool &timed_out,
                                                    float2 *row_pair) {
  const int t = threadIdx.x, lane = t & 31;
  if (t < 32) {
    const int slot = (it & 1) * ex.U + unit;
    float2 *pairs = ex.pairs + int64_t(slot) * ex.G;
    if (t == 0) {
      pairs[part] = make_float2(m, s);
      if (int(blockIdx.x) != ex.drop_block) {
        __threadfence();
        atomicAdd(&ex.counters[slot], 1u);
      }
      const unsigned int target = unsigned(ex.G) * unsigned(it / 2 + 1);
      const uint64_t t0 = globaltimer_ns();
      while (!timed_out && ld_acquire_gpu(&ex.counters[slot]) < target) {
        if (int64_t(globaltimer_ns() - t0) > ex.wait_limit_ns) {
          atomicOr(&g_softmax_status, 1u);
          timed_out = true;
        }
        __nanosleep(64);
      }
    }
    __syncwarp();
    float mm = -INFINITY;
    for (int k = lane; k < ex.G; k += 32) mm = fmaxf(mm, __ldcg(&pairs[k].x));
    mm = warp_max(mm);
    float ss = 0.0f;
    for (int k = lane; k < ex.G; k += 32) {
      const float2 q = __ldcg(&pairs[k]);
      if (q.y != 0.0f) ss += q.y * expf(q.x - mm);
    }
    ss = warp_sum(ss);
    if (t == 0) *row_pair = make_float2(mm, ss);
  }
  __syncthreads();
  return *row_pair;
}

// Rows staged in shared memory, one row per block, or per cluster of C blocks
// (kCluster) for rows longer than one block should hold.
//
// kVec: rows start on 16-byte boundaries (x, y 16-byte aligned, ldx and ldy
// multiples of 4; chunk is a multiple of 4).  kDouble: two staging buffers;
// the next row's asynchronous copies are in flight while the current row is
// reduced and stored (the page's double buffering, across rows).  Thread t
// copies, reads and writes only the columns it owns (vectors t, t + T, ...,
// then the scalars 4 nv + t, ...), so a buffer needs no barrier between its
// uses; only the reduction scratch does.  When a block of up to 256 threads
// has whole vectors, at most kRegVecs per thread, each thread reads its
// vectors from the buffer once and keeps them in registers for all three
// passes.
//
// A cluster splits each row into C chunks: block c stages columns
// [c chunk, (c + 1) chunk), takes its maximum m_c and s_c = sum e^{x - m_c}
// over them, and thread k pushes (m_c, s_c) into slot c of block k's shared
// memory (distributed shared memory).  After one cluster barrier every block
// reads the C slots in rank order, so all of them form the same
//     m = max_c m_c,   s = sum_c s_c e^{m_c - m},
// which equals sum_j e^{x_j - m} (e^{x - m} = e^{x - m_c} e^{m_c - m}), and
// scales its staged e^{x - m_c} by e^{m_c - m} / s.  A chunk that is all
// -inf has s_c = 0 and adds nothing.  The slots alternate between two sets
// by row parity: a block writes a set again only after passing the barrier of
// the following row, which every block reaches after reading that set.
constexpr int kRegVecs = 8;   // a thread's staged vectors held in registers, at most

template <int kThreads, bool kVec, bool kDouble, bool kCluster>
__global__ void __launch_bounds__(kThreads)
softmax_staged_kernel(int64_t rows, int cols, int chunk, const float *x, int64_t ldx, float *y,
                      int64_t ldy, unsigned long long *rowctr) {
  extern __shared__ __align__(16) float stage[];
  __shared__ float scratch[32];
  __shared__ float2 slots[2][kMaxCluster];
  __shared__ long long s_next;
  const int t = threadIdx.x;
  int C = 1, c = 0;
  int64_t unit = blockIdx.x, units = gridDim.x;
  if (kCluster) {
    cg::cluster_group cl = cg::this_cluster();
    C = int(cl.num_blocks());
    c = int(cl.block_rank());
    unit = blockIdx.x / C;
    units = gridDim.x / C;
  }
  const int c0 = c * chunk;
  const int len = max(0, min(cols - c0, chunk));   // columns of this block
  const int nv = kVec ? len >> 2 : 0;               // 16-byte vectors of them
  const int chunk_pad = (chunk + 3) & ~3;
  auto copy_row = [&](float *buf, int64_t r) {
    const float *xr = x + r * ldx + c0;
    for (int q = t; q < nv; q += kThreads) cp_async_16(buf + 4 * q, xr + 4 * q);
    for (int j = 4 * nv + t; j < len; j += kThreads) cp_async_4(buf + j, xr + j);
  };
  // Rows: a block's first is its index; with a row counter (one block per
  // row, double-buffered) each later one is taken from the counter while the
  // block works on the one before, so blocks the warp schedulers favour take
  // more rows and all finish together (measured: with fixed strides the last
  // blocks ended 40 % after the first).  A row's result does not depend on the
  // block that computes it.
  // Blocks of up to 256 threads only (measured: 3-13 % faster for rows of
  // 2560-4096 columns; with 512-thread blocks 10-17 % slower).
  constexpr bool kDyn = !kCluster && kDouble && kThreads <= 256;
  const bool dyn = kDyn && rowctr != nullptr;
  int64_t r = unit;
  int64_t rn = r + units;   // the row after r
  if (dyn) {
    if (t == 0) s_next = (long long)(units + int64_t(atomicAdd(&rowctr[0], 1ull)));
    __syncthreads();
    rn = s_next;
  }
  if (kDouble) {
    if (r < rows) copy_row(stage, r);
    cp_async_commit();
  }
  for (int it = 0; r < rows; ++it) {
    // The row after rn: taken now, its number needed only after pass 1, so
    // the counter's latency is hidden behind the pass.
    unsigned long long tok = 0;
    if (dyn && t == 0) tok = atomicAdd(&rowctr[0], 1ull);
    float *row = stage + (kDouble ? (it & 1) * chunk_pad : 0);
    if (kDouble) {
      if (rn < rows) copy_row(stage + ((it + 1) & 1) * chunk_pad, rn);
      cp_async_commit();
      cp_async_wait<1>();        // this thread's copies of row r have landed
    } else {
      copy_row(row, r);
      cp_async_commit();
      cp_async_wait<0>();
    }
    // Whole vectors only, and few enough: the thread's vectors are read from
    // the staged row once, into registers, and the passes run there.  Blocks of
    // up to 256 threads only (measured: 1-9 % faster there; with 512 threads the
    // registers cost a resident block per SM, 12 % slower).
    const bool regs = kVec && kThreads <= 256 && 4 * nv == len && nv <= kRegVecs * kThreads;
    float4 a[kRegVecs];
    float m = -INFINITY, s = 0.0f;
    if (regs) {
      // Pass 1: the maximum (of this block's columns).
#pragma unroll
      for (int i = 0; i < kRegVecs; ++i) {
        const int q = t + i * kThreads;
        if (q < nv) {
          a[i] = reinterpret_cast<const float4 *>(row)[q];
          m = fmaxf(fmaxf(m, fmaxf(a[i].x, a[i].y)), fmaxf(a[i].z, a[i].w));
        }
      }
      m = block_reduce<true>(m, scratch);
      if (dyn && t == 0) s_next = (long long)(units + int64_t(tok));   // read after the next barrier
      // In a cluster, an all -inf chunk takes 0 as its reference: its terms are 0 either way.
      const float ref = (kCluster && m == -INFINITY) ? 0.0f : m;
      // Pass 2: the exponentials, and their sum (same order as below).
#pragma unroll
      for (int i = 0; i < kRegVecs; ++i)
        if (t + i * kThreads < nv) {
          a[i].x = expf(a[i].x - ref); s += a[i].x;
          a[i].y = expf(a[i].y - ref); s += a[i].y;
          a[i].z = expf(a[i].z - ref); s += a[i].z;
          a[i].w = expf(a[i].w - ref); s += a[i].w;
        }
    } else {
      // Pass 1: the maximum (of this block's columns).
      for (int q = t; q < nv; q += kThreads) {
        const float4 v = reinterpret_cast<const float4 *>(row)[q];
        m = fmaxf(fmaxf(m, fmaxf(v.x, v.y)), fmaxf(v.z, v.w));
      }
      for (int j = 4 * nv + t; j < len; j += kThreads) m = fmaxf(m, row[j]);
      m = block_reduce<true>(m, scratch);
      if (dyn && t == 0) s_next = (long long)(units + int64_t(tok));   // read after the next barrier
      const float ref = (kCluster && m == -INFINITY) ? 0.0f : m;
      // Pass 2: exponentials in place, and their sum.
      for (int q = t; q < nv; q += kThreads) {
        float4 v = reinterpret_cast<float4 *>(row)[q];
        v.x = expf(v.x - ref); s += v.x;
        v.y = expf(v.y - ref); s += v.y;
        v.z = expf(v.z - ref); s += v.z;
        v.w = expf(v.w - ref); s += v.w;
        reinterpret_cast<float4 *>(row)[q] = v;
      }
      for (int j = 4 * nv + t; j < len; j += kThreads) {
        const float e = expf(row[j] - ref);
        row[j] = e;
        s += e;
      }
    }
    s = block_reduce<false>(s, scratch);
    const int64_t rnn = dyn ? int64_t(s_next) : rn + units;
    float scale;
    if (kCluster) {
      cg::cluster_group cl = cg::this_cluster();
      float2 *set = slots[it & 1];
      if (t < C) *cl.map_shared_rank(&set[c], t) = make_float2(m, s);
      cl.sync();
      float mm = -INFINITY;
      for (int k = 0; k < C; ++k) mm = fmaxf(mm, set[k].x);
      float ss = 0.0f;
      for (int k = 0; k < C; ++k)
        if (set[k].y != 0.0f) ss += set[k].y * expf(set[k].x - mm);
      if (mm == -INFINITY) scale = __int_as_float(0x7fc00000);   // all -inf: NaN, as the formula
      else scale = s != 0.0f ? expf(m - mm) / ss : 0.0f;
    } else {
      scale = 1.0f / s;
    }
    float *yr = y + r * ldy + c0;
    if (regs) {
#pragma unroll
      for (int i = 0; i < kRegVecs; ++i) {
        const int q = t + i * kThreads;
        if (q < nv)
          __stcs(reinterpret_cast<float4 *>(yr) + q,
                 make_float4(a[i].x * scale, a[i].y * scale, a[i].z * scale, a[i].w * scale));
      }
    } else {
      for (int q = t; q < nv; q += kThreads) {
        float4 v = reinterpret_cast<const float4 *>(row)[q];
        v.x *= scale; v.y *= scale; v.z *= scale; v.w *= scale;
        __stcs(reinterpret_cast<float4 *>(yr) + q, v);
      }
      for (int j = 4 * nv + t; j < len; j += kThreads) __stcs(yr + j, row[j] * scale);
    }
    r = rn;
    rn = rnn;
  }
  cp_async_wait<0>();
  if (kCluster) cg::this_cluster().sync();
  if (dyn && t == 0 && atomicAdd(&rowctr[1], 1ull) == gridDim.x - 1ull) {
    // The last block done: every fetch has happened, so reset for the next call.
    rowctr[0] = 0;
    rowctr[1] = 0;
    __threadfence();
  }
}

// Running (maximum, sum) of one thread's terms: s = sum e^{x - m}.  When the
// maximum rises to m', s is first scaled by e^{m - m'}; while m is -inf every
// term is e^{-inf} = 0 (reference 0), so s stays 0.
__device__ __forceinline__ void online_add(float &m, float &s, float mx, const float *v, int n) {
  if (mx > m) {
    s = s != 0.0f ? s * expf(m - mx) : s;
    m = mx;
  }
  const float ref = m == -INFINITY ? 0.0f : m;
  for (int i = 0; i < n; ++i) s += expf(v[i] - ref);
}

// (m, s) <- the pair for the union of two sets of terms: m = max, s = sum of
// s_i e^{m_i - m}.  Symmetric bit for bit (IEEE addition commutes), so both
// lanes of a shuffle exchange hold the same result.
__device__ __forceinline__ void online_merge(float &m, float &s, float m2, float s2) {
  const float mm = fmaxf(m, m2);
  float r = s != 0.0f ? s * expf(m - mm) : 0.0f;
  if (s2 != 0.0f) r += s2 * expf(m2 - mm);
  m = mm;
  s = r;
}

// Long rows: a cooperative grid of resident blocks, G blocks per row (block b
// takes part b % G of row unit b / G), U = grid / G rows in flight, so that
// the rows in flight -- about grid x kGridChunk floats -- fit in L2.  Pass 1
// reads the block's columns once, each thread keeping a running (m, s)
// (online_add: at most one rescale per four columns), and the block's threads
// merge theirs (shuffle tree, then the warps' pairs in order); the G blocks
// of the row then meet (exchange_row_pair).  Pass 2 re-reads the block's
// columns -- mostly from L2 -- and writes y.  (Measured against staging the
// chunks in shared memory with one double-buffered block per SM, meeting the
// same way: 131072 columns 4950 against 3486 GB/s; several blocks per SM keep
// more loads in flight than one staging block does.)
template <bool kVec>
__global__ void __launch_bounds__(kGridThreads)
softmax_grid_kernel(const GridRowsParams p) {
  constexpr int T = kGridThreads;
  extern __shared__ __align__(16) float4 keep[];   // kGridKeep x T vectors (kVec only)
  __shared__ float2 scratch[32];
  __shared__ float2 row_pair;
  const int b = blockIdx.x;
  const int u = b / p.ex.G, part = b - u * p.ex.G;
  if (u >= p.ex.U) return;
  const int c0 = part * p.chunk;
  const int len = max(0, min(p.cols - c0, p.chunk));
  const int nv = kVec ? len >> 2 : 0;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  bool timed_out = false;   // thread 0: once a wait has run out, later ones are skipped
  int it = 0;
  for (int64_t r = u; r < p.rows; r += p.ex.U, ++it) {
    const float *xr = p.x + r * p.ldx + c0;
    float m = -INFINITY, s = 0.0f;
    // This thread's vectors are t + i T, i < n; the first kGridKeep of them
    // are kept in shared memory for pass 2 (keep[i T + t]).
    const int n = nv > t ? (nv - 1 - t) / T + 1 : 0;
    if (kVec) {
      const float4 *xv = reinterpret_cast<const float4 *>(xr);
      int i = 0;
      for (; i + 3 < n; i += 4) {
        float4 a[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) a[k] = xv[t + (i + k) * T];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (i + k < kGridKeep) keep[(i + k) * T + t] = a[k];
          const float v[4] = {a[k].x, a[k].y, a[k].z, a[k].w};
          online_add(m, s, fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3])), v, 4);
        }
      }
      for (; i < n; ++i) {
        const float4 a = xv[t + i * T];
        if (i < kGridKeep) keep[i * T + t] = a;
        const float v[4] = {a.x, a.y, a.z, a.w};
        online_add(m, s, fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3])), v, 4);
      }
    }
    {
      int j = 4 * nv + t;
      for (; j + 3 * T < len; j += 4 * T) {
        float v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = xr[j + k * T];
#pragma unroll
        for (int k = 0; k < 4; ++k) online_add(m, s, v[k], &v[k], 1);
      }
      for (; j < len; j += T) {
        const float v = xr[j];
        online_add(m, s, v, &v, 1);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      online_merge(m, s, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, s, o));
    if (lane == 0) scratch[warp] = make_float2(m, s);
    __syncthreads();
    float bm = -INFINITY, bs = 0.0f;
    if (t == 0)
      for (int k = 0; k < T / 32; ++k) online_merge(bm, bs, scratch[k].x, scratch[k].y);
    const float2 rp = exchange_row_pair(p.ex, u, part, it, bm, bs, timed_out, &row_pair);
    const float mm = rp.x;
    const float inv = mm == -INFINITY ? __int_as_float(0x7fc00000) : 1.0f / rp.y;
    float *yr = p.y + r * p.ldy + c0;
    auto out4 = [&](float4 a) {
      return make_float4(expf(a.x - mm) * inv, expf(a.y - mm) * inv, expf(a.z - mm) * inv,
                         expf(a.w - mm) * inv);
    };
    // Pass 2, each thread's vectors backwards: the latest read are the
    // likeliest to be still in L2, and the earliest are in shared memory.
    if (kVec) {
      const float4 *xv = reinterpret_cast<const float4 *>(xr);
      float4 *yv = reinterpret_cast<float4 *>(yr);
      int i = n - 1;
      for (; i - 3 >= kGridKeep; i -= 4) {
        float4 a[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) a[k] = xv[t + (i - k) * T];
#pragma unroll
        for (int k = 0; k < 4; ++k) __stcs(yv + t + (i - k) * T, out4(a[k]));
      }
      for (; i >= kGridKeep; --i) __stcs(yv + t + i * T, out4(xv[t + i * T]));
      for (; i >= 0; --i) __stcs(yv + t + i * T, out4(keep[i * T + t]));
    }
    {
      const int j0 = 4 * nv + t;
      int i = len > j0 ? (len - 1 - j0) / T : -1;
      for (; i >= 3; i -= 4) {
        float v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = xr[j0 + (i - k) * T];
#pragma unroll
        for (int k = 0; k < 4; ++k) __stcs(yr + j0 + (i - k) * T, expf(v[k] - mm) * inv);
      }
      for (; i >= 0; --i) __stcs(yr + j0 + i * T, expf(xr[j0 + i * T] - mm) * inv);
    }
  }
}

std::atomic<unsigned int> g_grid_epoch{0};
std::atomic<unsigned int> g_rows_epoch{0};

// Row counters of softmax_staged_kernel, kGridRegions pairs (next row, blocks
// done); each call takes the next pair, and its last block resets it.
__device__ unsigned long long g_sm_rows[kGridRegions][2];

cudaError_t row_counter(unsigned long long **ctr) {
  unsigned long long *base = nullptr;
  cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void **>(&base), g_sm_rows);
  if (e != cudaSuccess) return e;
  *ctr = base + 2 * (g_rows_epoch.fetch_add(1, std::memory_order_relaxed) % kGridRegions);
  return cudaSuccess;
}
std::atomic<int64_t> g_sm_wait_limit_ns{int64_t(10) * 1000 * 1000 * 1000};
std::atomic<int> g_sm_drop_block{-1};

// This call's exchange: the next of the kGridRegions regions, its 2 U counters
// zeroed on `stream` ahead of the launch.
cudaError_t make_exchange(int G, int64_t U, cudaStream_t stream, RowExchange *ex) {
  const unsigned int region = g_grid_epoch.fetch_add(1, std::memory_order_relaxed) % kGridRegions;
  unsigned int *counters = nullptr;
  float2 *pairs = nullptr;
  cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void **>(&counters), g_sm_counters);
  if (e != cudaSuccess) return e;
  e = cudaGetSymbolAddress(reinterpret_cast<void **>(&pairs), g_sm_pairs);
  if (e != cudaSuccess) return e;
  ex->G = G;
  ex->U = int(U);
  ex->counters = counters + size_t(region) * 2 * kGridMaxBlocks;
  ex->pairs = pairs + size_t(region) * 2 * kGridMaxBlocks;
  ex->wait_limit_ns = g_sm_wait_limit_ns.load(std::memory_order_relaxed);
  ex->drop_block = g_sm_drop_block.load(std::memory_order_relaxed);
  return cudaMemsetAsync(ex->counters, 0, size_t(2) * size_t(U) * sizeof(unsigned int), stream);
}

// Per-device launch facts for one kernel instantiation, set up on first use.
struct KernelSetup {
  std::atomic<uint64_t> configured{0};
};

// Stage plan for rows too long for a warp: how many blocks share a row, how
// many columns each stages, and whether two buffers fit.
struct StagePlan {
  int cluster;   // blocks per row (1, 2, 4 or 8)
  int chunk;     // columns per block, a multiple of 4 when cluster > 1
  bool dbl;      // double-buffered
};

constexpr int kSingleBlockCols = 16384;   // rows up to this length: one block per row
constexpr int kChunkTarget = 8192;        // longer rows: chunks of at most this many columns ...
constexpr int kClusterLimit = 8;          // ... over at most this many blocks
constexpr int kMaxChunk = kMaxStagedRowBytes / int(sizeof(float));
static_assert(kClusterLimit <= kMaxCluster, "exchange slots are sized for kMaxCluster blocks");

bool plan_stage(int cols, StagePlan *p) {
  int C = 1, chunk = cols;
  if (cols > kSingleBlockCols) {
    while (chunk > kChunkTarget && C < kClusterLimit) {
      C *= 2;
      chunk = (((cols + C - 1) / C) + 3) & ~3;
    }
  }
  if (chunk > kMaxChunk) return false;
  p->cluster = C;
  p->chunk = chunk;
  p->dbl = 2 * ((chunk + 3) & ~3) * int(sizeof(float)) <= kMaxStagedRowBytes;
  return true;
}

// Threads per block for a chunk of the given length (measured on GB300 over
// rows of 2048 to 393216 columns: a lone block wants 8-16 columns per thread,
// a block in a cluster about 32, since it also waits at the cluster barrier).
int staged_threads(int chunk, int cluster) {
  if (cluster > 1) return chunk <= 8192 ? 256 : (chunk <= 16384 ? 512 : 1024);
  if (chunk <= 4096) return 128;
  if (chunk <= 16384) return 512;
  return 1024;
}

template <int kThreads, bool kVec, bool kDouble, bool kCluster>
cudaError_t launch_staged(int64_t rows, int cols, const StagePlan &plan, const float *x,
                          int64_t ldx, float *y, int64_t ldy, const DeviceInfo &dev,
                          cudaStream_t stream) {
  static KernelSetup st;
  auto kernel = softmax_staged_kernel<kThreads, kVec, kDouble, kCluster>;
  const int chunk_pad = (plan.chunk + 3) & ~3;
  const int smem = (kDouble ? 2 : 1) * chunk_pad * int(sizeof(float));
  const uint64_t bit = uint64_t(1) << (dev.id & 63);
  if (!(st.configured.load(std::memory_order_acquire) & bit)) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kMaxStagedRowBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    if (kCluster) {
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
    st.configured.fetch_or(bit, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = size_t(smem);
  cfg.stream = stream;
  int64_t units = 0;
  if (kCluster) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(plan.cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(unsigned(plan.cluster) * 64, 1, 1);   // shape only, for the query
    int clusters = 0;
    cudaError_t e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (clusters <= 0) return cudaErrorInvalidConfiguration;
    units = std::min<int64_t>(rows, clusters);
    cfg.gridDim = dim3(unsigned(units * plan.cluster), 1, 1);
  } else {
    int nb = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, kThreads, smem);
    if (e != cudaSuccess) return e;
    units = std::min<int64_t>(rows, int64_t(dev.sm_count) * (nb > 0 ? nb : 1));
    cfg.gridDim = dim3(unsigned(units), 1, 1);
  }
  unsigned long long *rowctr = nullptr;
  // A row counter only where several blocks share an SM (with one block per
  // SM there is no imbalance to remove).
  if (!kCluster && kDouble && kThreads <= 256 && units >= 2 * int64_t(dev.sm_count)) {
    cudaError_t e = row_counter(&rowctr);
    if (e != cudaSuccess) return e;
  }
  return cudaLaunchKernelEx(&cfg, kernel, rows, cols, plan.chunk, x, ldx, y, ldy, rowctr);
}

template <int kThreads>
cudaError_t launch_staged_any(int64_t rows, int cols, const StagePlan &plan, const float *x,
                              int64_t ldx, float *y, int64_t ldy, bool vec, const DeviceInfo &dev,
                              cudaStream_t stream) {
#define TMM_STAGED(V, D, K) \
  launch_staged<kThreads, V, D, K>(rows, cols, plan, x, ldx, y, ldy, dev, stream)
  if (plan.cluster > 1) {
    if (vec) return plan.dbl ? TMM_STAGED(true, true, true) : TMM_STAGED(true, false, true);
    return plan.dbl ? TMM_STAGED(false, true, true) : TMM_STAGED(false, false, true);
  }
  if (vec) return plan.dbl ? TMM_STAGED(true, true, false) : TMM_STAGED(true, false, false);
  return plan.dbl ? TMM_STAGED(false, true, false) : TMM_STAGED(false, false, false);
#undef TMM_STAGED
}

// Rows from this length on take softmax_grid_kernel (measured on GB300: from
// here on it beats a cluster staging the row; below, staging wins).
constexpr int kGridRowCols = 65537;

template <bool kVec>
cudaError_t launch_grid_rows(int64_t rows, int cols, const float *x, int64_t ldx, float *y,
                             int64_t ldy, const DeviceInfo &dev, cudaStream_t stream) {
  static KernelSetup st;
  static std::atomic<int> blocks_per_sm[64];
  auto kernel = softmax_grid_kernel<kVec>;
  const size_t smem = kVec ? size_t(kGridKeep) * kGridThreads * sizeof(float4) : 0;
  const uint64_t bit = uint64_t(1) << (dev.id & 63);
  if (!(st.configured.load(std::memory_order_acquire) & bit)) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem));
    if (e != cudaSuccess) return e;
    // The default carveout: a larger L1 serves some of pass 2's re-reads
    // (measured: the maximum shared carveout loses 10-15 %).
    int nb = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, kGridThreads, smem);
    if (e != cudaSuccess) return e;
    if (nb < 1) return cudaErrorInvalidConfiguration;
    blocks_per_sm[dev.id & 63].store(nb, std::memory_order_relaxed);
    st.configured.fetch_or(bit, std::memory_order_release);
  }
  const int64_t grid = std::min<int64_t>(
      int64_t(blocks_per_sm[dev.id & 63].load(std::memory_order_relaxed)) * dev.sm_count,
      kGridMaxBlocks);
  GridRowsParams prm = {};
  prm.rows = rows;
  prm.cols = cols;
  const int G = int(std::min<int64_t>((int64_t(cols) + kGridChunk - 1) / kGridChunk, grid));
  prm.chunk = int((((int64_t(cols) + G - 1) / G) + 3) & ~int64_t(3));
  prm.x = x;
  prm.ldx = ldx;
  prm.y = y;
  prm.ldy = ldy;
  cudaError_t e = make_exchange(G, std::min<int64_t>(grid / G, rows), stream, &prm.ex);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(unsigned(int64_t(prm.ex.U) * prm.ex.G), 1, 1);
  cfg.blockDim = dim3(kGridThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, kernel, prm);
}

int64_t warp_grid(int64_t units, const DeviceInfo &dev) {
  constexpr int kWarps = kWarpRowThreads / 32;
  return std::max<int64_t>(1, std::min<int64_t>((units + kWarps - 1) / kWarps,
                                                int64_t(dev.sm_count) * 8));
}

template <int kW, int kPer>
cudaError_t launch_warp_rows(int64_t rows, int cols, const float *x, int64_t ldx, float *y,
                             int64_t ldy, const DeviceInfo &dev, cudaStream_t stream) {
  const int64_t grid = warp_grid((rows + 32 / kW - 1) / (32 / kW), dev);
  softmax_warp_kernel<kW, kPer><<<unsigned(grid), kWarpRowThreads, 0, stream>>>(
      rows, cols, x, ldx, y, ldy);
  return cudaGetLastError();
}

template <int kW, int kVec>
cudaError_t launch_warp_vec(int64_t rows, int cols, const float *x, int64_t ldx, float *y,
                            int64_t ldy, const DeviceInfo &dev, cudaStream_t stream) {
  const int64_t grid = warp_grid((rows + 32 / kW - 1) / (32 / kW), dev);
  softmax_warp_vec_kernel<kW, kVec><<<unsigned(grid), kWarpRowThreads, 0, stream>>>(
      rows, cols, x, ldx, y, ldy);
  return cudaGetLastError();
}

}  // namespace

cudaError_t softmax_device_status(unsigned int *status, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(status, g_softmax_status, sizeof(unsigned int));
  if (e != cudaSuccess || !clear) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_softmax_status, &zero, sizeof(unsigned int));
}

void softmax_set_test_hooks(int drop_block, int64_t wait_limit_ns) {
  g_sm_drop_block.store(drop_block, std::memory_order_relaxed);
  g_sm_wait_limit_ns.store(wait_limit_ns > 0 ? wait_limit_ns : int64_t(10) * 1000 * 1000 * 1000,
                           std::memory_order_relaxed);
}

// Chunk length (a multiple of 4 x kSumThreads vectors) and count for nvec vectors.
void sum_chunks(int64_t nvec, int64_t *V, int64_t *G) {
  constexpr int64_t kGroup = 4 * kSumThreads;
  int64_t v = (nvec + kSumMaxPartials - 1) / kSumMaxPartials;
  v = v > kSumChunkVecsMin ? v : kSumChunkVecsMin;
  v = (v + kGroup - 1) / kGroup * kGroup;
  *V = v;
  *G = (nvec + v - 1) / v;
}

std::atomic<unsigned int> g_sum_epoch{0};

cudaError_t launch_sum(int64_t n, const float *x, float *out, float *partials,
                       const DeviceInfo &dev, cudaStream_t stream) {
  if (n == 0) return cudaMemsetAsync(out, 0, sizeof(float), stream);
  const uintptr_t addr = reinterpret_cast<uintptr_t>(x);
  const int64_t head = std::min<int64_t>(n, int64_t(((16 - (addr & 15)) & 15) >> 2));
  const int64_t nvec = (n - head) >> 2;
  const int64_t tail_at = head + 4 * nvec;
  const int tail = int(n - tail_at);
  int64_t V = 0, G = 0;
  sum_chunks(nvec, &V, &G);
  if (G > 0) {
    static KernelSetup st;
    static std::atomic<int> blocks_per_sm[64];
    const uint64_t bit = uint64_t(1) << (dev.id & 63);
    if (!(st.configured.load(std::memory_order_acquire) & bit)) {
      int nb = 0;
      cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, sum_partials_kernel,
                                                                    kSumThreads, 0);
      if (e != cudaSuccess) return e;
      blocks_per_sm[dev.id & 63].store(nb > 0 ? nb : 1, std::memory_order_relaxed);
      st.configured.fetch_or(bit, std::memory_order_release);
    }
    const int64_t grid = std::min<int64_t>(
        G, int64_t(blocks_per_sm[dev.id & 63].load(std::memory_order_relaxed)) * dev.sm_count);
    unsigned long long *ctr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void **>(&ctr), g_sum_chunks);
    if (e != cudaSuccess) return e;
    ctr += 2 * (g_sum_epoch.fetch_add(1, std::memory_order_relaxed) % kSumRegions);
    sum_partials_kernel<<<unsigned(grid), kSumThreads, 0, stream>>>(
        nvec, V, G, reinterpret_cast<const float4 *>(x + head), partials, ctr);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  sum_final_kernel<<<1, kSumFinalThreads, 0, stream>>>(G, partials, x, int(head), tail_at, tail,
                                                       out);
  return cudaGetLastError();
}

cudaError_t launch_softmax_rows(int64_t rows, int cols, const float *x, int64_t ldx, float *y,
                                int64_t ldy, const DeviceInfo &dev, cudaStream_t stream) {
  // Rows that start on 16-byte boundaries and hold whole vectors.
  const bool aligned =
      ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15u) == 0 &&
      (ldx & 3) == 0 && (ldy & 3) == 0;
#define TMM_WARP(W, P) launch_warp_rows<W, P>(rows, cols, x, ldx, y, ldy, dev, stream)
#define TMM_WVEC(W, V) launch_warp_vec<W, V>(rows, cols, x, ldx, y, ldy, dev, stream)
  if (aligned && (cols & 3) == 0 && cols <= 2048) {
    if (cols <= 4) return TMM_WVEC(1, 1);
    if (cols <= 8) return TMM_WVEC(2, 1);
    if (cols <= 16) return TMM_WVEC(4, 1);
    if (cols <= 32) return TMM_WVEC(8, 1);
    if (cols <= 64) return TMM_WVEC(16, 1);
    if (cols <= 128) return TMM_WVEC(32, 1);
    if (cols <= 256) return TMM_WVEC(32, 2);
    if (cols <= 512) return TMM_WVEC(32, 4);
    if (cols <= 1024) return TMM_WVEC(32, 8);
    return TMM_WVEC(32, 16);
  }
  if (cols <= 4) return TMM_WARP(1, 4);
  if (cols <= 8) return TMM_WARP(2, 4);
  if (cols <= 16) return TMM_WARP(4, 4);
  if (cols <= 32) return TMM_WARP(8, 4);
  if (cols <= 64) return TMM_WARP(16, 4);
  if (cols <= 128) return TMM_WARP(32, 4);
  if (cols <= 256) return TMM_WARP(32, 8);
  if (cols <= 512) return TMM_WARP(32, 16);
  if (cols <= 1024) return TMM_WARP(32, 32);
#undef TMM_WARP
#undef TMM_WVEC
  if (cols >= kGridRowCols)
    return aligned ? launch_grid_rows<true>(rows, cols, x, ldx, y, ldy, dev, stream)
                   : launch_grid_rows<false>(rows, cols, x, ldx, y, ldy, dev, stream);
  StagePlan plan;
  if (plan_stage(cols, &plan)) {
    switch (staged_threads(plan.chunk, plan.cluster)) {
      case 128: return launch_staged_any<128>(rows, cols, plan, x, ldx, y, ldy, aligned, dev, stream);
      case 256: return launch_staged_any<256>(rows, cols, plan, x, ldx, y, ldy, aligned, dev, stream);
      case 512: return launch_staged_any<512>(rows, cols, plan, x, ldx, y, ldy, aligned, dev, stream);
      default: return launch_staged_any<1024>(rows, cols, plan, x, ldx, y, ldy, aligned, dev, stream);
    }
  }
  return aligned ? launch_grid_rows<true>(rows, cols, x, ldx, y, ldy, dev, stream)
                 : launch_grid_rows<false>(rows, cols, x, ldx, y, ldy, dev, stream);
}

}  // namespace tmm
