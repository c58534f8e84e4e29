// gemm_tc3.cu -- FP32 product on the tcgen05 tensor cores with split-TF32 operands.
//
// The product C = A x B is the same as gemm_f32's; only the arithmetic units
// differ.  Each FP32 operand x is split into two TF32 values, hi (x with its
// low 13 mantissa bits cleared) and lo (x - hi, exact in FP32, rounded to the
// nearest TF32).  Then
//     a b = a_hi b_hi + a_hi b_lo + a_lo b_hi + a_lo b_lo,
// and the last term (about 2^-22 |a b|) is dropped: three TF32 tensor-core
// products, accumulated in FP32, give a result within FP32 accuracy.  Small
// integers (|x| < 2^11) are exact TF32 values (lo = 0), so integer-valued
// inputs stay exact.
//
// Structure (two pre-pass launches and one product launch per call):
//   1. split pre-pass -- A into A_hi, A_lo (M x Kp, K-major) and B, transposed,
//      into B_hi, B_lo (N x Kp, K-major), in the caller's workspace; Kp is K
//      rounded up to 32 with zeros, so every K-slice is whole.  The tensor
//      core reads a TF32 operand by ignoring the low 13 bits of an FP32 word,
//      which is exactly hi, so an operand already stored K-major with aligned
//      rows is read as its own hi and only its lo is written;
//   2. product kernel, for M > 128 on block pairs (gemm_tc3_pair_kernel,
//      described before it: 256 x 256 tiles, tcgen05.mma.cta_group::2,
//      persistent), else one 128 x 256 tile per block (gemm_tc3_kernel), with
//      three roles in each block:
//      * copy (one thread): TMA (tensor-map bulk copies, 64-byte swizzle)
//        loads K-slices of 16 of the four operands into a ring of stages;
//      * tensor core (one thread): tcgen05.mma.kind::tf32, three per K-step,
//        into one of two tensor-memory accumulators (128 lanes x 256 FP32
//        columns each), switching buffers every kTcChunk values of K;
//      * accumulate (eight warps): as each chunk completes, read it with
//        tcgen05.ld and add it into FP32 registers (round to nearest), then
//        release the buffer; after the last chunk, store C.
//      The tensor core's own FP32 accumulation does not round to nearest
//      (measured: error growing linearly in K); bounding each tensor-memory
//      sum to kTcChunk values of K and adding the chunks on the CUDA cores
//      keeps the product within FP32 accuracy at any K.
// Scheduling: tiles in row-major order, so the tiles in flight move through K
// together and share the A and B panels in L2.  When the tile count leaves the
// last wave at most half full, each of its tiles is split into two halves of
// the K range, run side by side: the unit holding the lower half stores its
// partial sums into C and raises a flag (one per accumulate warp), the unit
// holding the upper half waits for it (bounded), adds, and stores the total --
// in that fixed order, so results are deterministic.  The last wave then takes
// half the time.  With at most half as many tiles as slots, every tile is cut
// into up to four K-parts on chunk boundaries in the same way: the first part
// stores and raises its flag, and each later part waits for the previous one's
// flag, adds C, stores and (unless it is the last) raises its own.  A part's
// units come in item order, so a waiting block or pair always waits for one
// launched before it: no wait depends on a block that has not started.
// Epilogue: each accumulate warp holds 32 rows (one per lane) of 128 columns;
// it stores them through a 4 KiB staging buffer in shared memory, transposed
// so that every store instruction writes whole 128-byte lines of C.
// This follows the block-tile / staged-slab schedule of "CMU DLSys Lecture 12"
// section 5 and the double buffering of "Tiling Strategies" section 3; the
// register tile is replaced by a tensor-memory accumulator.
//
// Every mbarrier wait is bounded (globaltimer); on timeout the block records
// bit 1 in its device status word, stops issuing work, waits (bounded) for its
// copies in flight, frees its tensor memory and exits.
#include <cuda.h>

#include <algorithm>
#include <atomic>
#include <cstdint>

#include "bounds_check.cuh"
#include "tmm_internal.h"

namespace tmm {

// Status word: bit 1 when a bounded wait ran out of time, bit 2 when a range
// check of the bounds-checked build failed.
__device__ unsigned int g_tc3_status;
// Split-tile flags, one per (tail block, accumulate warp): kTc3FlagRegions
// rings; a call uses region epoch % kTc3FlagRegions and raises flags to its epoch.
constexpr int kTc3FlagRegions = 16;
constexpr int kTc3MaxBlocks = 1024;   // tail blocks of one call
constexpr int kTc3FlagsPerBlock = 8;   // = the accumulate warps
__device__ unsigned int g_tc3_flags[kTc3FlagRegions * kTc3MaxBlocks * kTc3FlagsPerBlock];

namespace {

constexpr int kTcBM = 128;
constexpr int kTcBN = 256;
constexpr int kTcBK = 16;                          // floats per K-slice: one 64-byte swizzle row
constexpr int kTcStages = 4;
constexpr int kTcChunk = 256;                      // K values per tensor-memory sum
constexpr int kTcAccWarps = 8;                     // accumulate / epilogue warps
constexpr int kTcThreads = 32 * (2 + kTcAccWarps); // copy warp, tensor-core warp, 8 more
constexpr int kKPad = 32;                          // workspace K is a multiple of this
constexpr uint32_t kATileBytes = kTcBM * kTcBK * 4;   // 8 KiB
constexpr uint32_t kBTileBytes = kTcBN * kTcBK * 4;   // 16 KiB
constexpr uint32_t kStageBytes = 2 * kATileBytes + 2 * kBTileBytes;
constexpr uint32_t kTmemCols = 2 * kTcBN;         // two FP32 accumulators of kTcBN columns
constexpr uint32_t kBarrierBytes = 8 * (2 * kTcStages + 5) + 8;
constexpr uint32_t kStagingBytes = kTcAccWarps * 32 * 32 * 4;   // 4 KiB per accumulate warp
constexpr uint32_t kTcSmemBytes =
    1024 + kTcStages * kStageBytes + kBarrierBytes + 128 + kStagingBytes;
constexpr uint32_t kMaxSmemPerBlock = 232448;   // 227 KiB, the opt-in limit of one block
static_assert(kTcSmemBytes <= kMaxSmemPerBlock, "ring, barriers and staging fit one block");

static_assert(kTcBK * 4 == 64, "one K-slice row is one 64-byte swizzle row");
static_assert(kTcChunk % kTcBK == 0 && kKPad % kTcBK == 0, "chunks are whole slices");
static_assert(kStageBytes % 1024 == 0 && kATileBytes % 1024 == 0 && kBTileBytes % 1024 == 0,
              "tiles stay 1024-byte aligned");

// Instruction descriptor of tcgen05.mma.kind::tf32: D = F32 (bits 4-5 = 1),
// A = B = TF32 (bits 7-9, 10-12 = 2), both K-major (bits 15, 16 = 0),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t kIdescTf32 = (1u << 4) | (2u << 7) | (2u << 10) |
                                (uint32_t(kTcBN >> 3) << 17) | (uint32_t(kTcBM >> 4) << 24);

// Shared-memory matrix descriptor of a K-major operand tile with 64-byte
// swizzle: start address >> 4 (bits 0-13), leading byte offset (unused for
// swizzled K-major tiles; 16 B) >> 4 (bits 16-29), stride byte offset = 8 rows
// x 64 B = 512 B >> 4 (bits 32-45), descriptor version 1 (bits 46-47),
// layout 4 = 64-byte swizzle (bits 61-63).
__device__ __forceinline__ uint64_t sw64_desc(uint32_t smem_addr) {
  return uint64_t((smem_addr >> 4) & 0x3FFFu) | (uint64_t(1) << 16) |
         (uint64_t(512 >> 4) << 32) | (uint64_t(1) << 46) | (uint64_t(4) << 61);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
// Wait for phase `parity` of the barrier to complete; false after limit_ns.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (int64_t(timer_ns() - t0) > limit_ns) return false;
  return true;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %3, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %4, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(accumulate), "r"(kIdescTf32)
      : "memory");
}
// Arrive on `bar` once every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
// 8 consecutive FP32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_load_8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// hi: x truncated to TF32; lo: the exact remainder rounded to the nearest TF32.
__device__ __forceinline__ void split_tf32(float x, float &hi, float &lo) {
  hi = __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
  const float r = x - hi;
  lo = __uint_as_float((__float_as_uint(r) + 0x1000u) & 0xFFFFE000u);
}

// ---- split pre-pass -----------------------------------------------------------

// Rows of K values (M x K, ld) -> hi, lo (M x Kp), zeros for k >= K.  Thread
// handles 4 consecutive k of one row; rows advance with the grid's y extent.
// write_hi = 0: only lo is written (the product then reads hi from the operand
// itself -- see launch_tc3).
__global__ void tc3_split_a_kernel(int M, int K, int Kp, const float *__restrict__ A, int64_t lda,
                                   int vec_load, int write_hi, float *__restrict__ hi,
                                   float *__restrict__ lo) {
  const int k = 4 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (k >= Kp) return;
  for (int m = blockIdx.y; m < M; m += gridDim.y) {
    const float *a = A + int64_t(m) * lda;
    float x[4];
    if (vec_load && k + 4 <= K) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (TMM_IN_BOUNDS(in_matrix(a + k, A, M, K, lda, 4), &g_tc3_status))
        v = *reinterpret_cast<const float4 *>(a + k);
      x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        x[j] = k + j < K && TMM_IN_BOUNDS(in_matrix(a + k + j, A, M, K, lda), &g_tc3_status)
                   ? a[k + j] : 0.0f;
    }
    float h[4], l[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) split_tf32(x[j], h[j], l[j]);
    const int64_t o = int64_t(m) * Kp + k;
    if (write_hi && TMM_IN_BOUNDS(in_matrix(hi + o, hi, M, Kp, Kp, 4), &g_tc3_status))
      *reinterpret_cast<float4 *>(hi + o) = make_float4(h[0], h[1], h[2], h[3]);
    if (TMM_IN_BOUNDS(in_matrix(lo + o, lo, M, Kp, Kp, 4), &g_tc3_status))
      *reinterpret_cast<float4 *>(lo + o) = make_float4(l[0], l[1], l[2], l[3]);
  }
}

// K rows of N values (K x N, ldb) -> hi, lo transposed (N x Kp), zeros for
// k >= K; 32 x 32 tiles through shared memory.
__global__ void tc3_split_bt_kernel(int K, int N, int Kp, const float *__restrict__ B, int64_t ldb,
                                    float *__restrict__ hi, float *__restrict__ lo) {
  // The product kernel may be scheduled now; it waits for this grid to finish
  // before its first read of the split operands.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ float tile[32][33];
  const int k0 = blockIdx.y * 32, n0 = blockIdx.x * 32;
  const int tx = threadIdx.x, ty = threadIdx.y;   // 32 x 8
#pragma unroll
  for (int j = 0; j < 32; j += 8) {
    const int k = k0 + ty + j, n = n0 + tx;
    tile[ty + j][tx] = (k < K && n < N && TMM_IN_BOUNDS(in_matrix(B + int64_t(k) * ldb + n, B,
                                                                   K, N, ldb),
                                                         &g_tc3_status))
                           ? B[int64_t(k) * ldb + n] : 0.0f;
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < 32; j += 8) {
    const int n = n0 + ty + j, k = k0 + tx;
    if (n < N && k < Kp) {
      float h, l;
      split_tf32(tile[tx][ty + j], h, l);
      if (TMM_IN_BOUNDS(in_matrix(hi + int64_t(n) * Kp + k, hi, N, Kp, Kp) &&
                            in_matrix(lo + int64_t(n) * Kp + k, lo, N, Kp, Kp),
                        &g_tc3_status)) {
        hi[int64_t(n) * Kp + k] = h;
        lo[int64_t(n) * Kp + k] = l;
      }
    }
  }
}

// ---- product kernel ---------------------------------------------------------------

struct Tc3Params {
  int M, N, Kp;
  float *C;
  int64_t ldc;
  int tiles_m, tiles_n;
  int slices;            // K-slices per tile
  int dp_tiles;          // items [0, dp_tiles) are whole tiles
  int parts;             // K-parts of each tile from dp_tiles on (1: none split)
  int chunks;            // ceil(slices / slices per chunk); parts end on chunk bounds
  int items;             // dp_tiles + parts x (split tiles): the work list
  unsigned int epoch;    // this call's flag value (never 0)
  int vec_store;         // C 16-byte aligned and ldc % 4 == 0
  int64_t wait_limit_ns;
  int drop_signal_block; // testing hook: this block never raises its flags (-1: none)
};

__device__ __forceinline__ void tc3_tile_coords(int tile, int tiles_n, int &tm, int &tn) {
  tm = tile / tiles_n;
  tn = tile - tm * tiles_n;
}

// This block's work items (tile, K-slice range): items b, b + stride, ...
// of the list [whole tiles, split units]; `unit` >= 0 numbers the items that
// share a split tile, `parts` consecutive units per tile (part 0 holds the
// lowest K-range; the last part, which stores the total, the highest).  The one-block kernel launches one block per item;
// the pair kernel one pair per resident slot, each pair walking its items in
// order.  Whole tiles are a multiple of the stride whenever units exist, so
// all units fall in the last round, each on its own pair and alongside its
// partners.
struct Tc3Work {
  int idx, stride;
  __device__ __forceinline__ void init(const Tc3Params &, int first, int step) {
    idx = first;
    stride = step;
  }
  __device__ __forceinline__ bool next(const Tc3Params &p, int &tile, int &kb, int &ke,
                                       int &unit) {
    if (idx >= p.items) return false;
    const int b = idx;
    idx += stride;
    if (b < p.dp_tiles) {
      tile = b;
      kb = 0;
      ke = p.slices;
      unit = -1;
      return true;
    }
    unit = b - p.dp_tiles;
    const int part = unit % p.parts;
    tile = p.dp_tiles + unit / p.parts;
    constexpr int kSlicesPerChunk = kTcChunk / kTcBK;
    kb = (part * p.chunks / p.parts) * kSlicesPerChunk;
    ke = part + 1 == p.parts ? p.slices : ((part + 1) * p.chunks / p.parts) * kSlicesPerChunk;
    return true;
  }
};

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int *p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(unsigned int *p, unsigned int v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
static_assert(kTc3FlagsPerBlock == kTcAccWarps, "one flag per accumulate warp");

__device__ __forceinline__ void st_shared_v4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}
__device__ __forceinline__ float4 ld_shared_v4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ float f4_get(const float4 &v, int j) {
  return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}

// Stores one accumulate warp's 32 x 128 block of C -- lane l holds row
// row_base + l, acc[j] its column col0 + j -- through the warp's 4 KiB staging
// buffer `stg` in shared memory.  Each 32 x 32 part is written there row by
// row and read back transposed, so that 8 lanes cover 128 contiguous bytes of
// one row and one instruction stores 4 whole cache lines (a direct store from
// the row-per-lane layout touches 32 lines with 16 bytes each).  16-byte
// chunk q of staged row r sits at position q ^ (r % 8), which keeps both the
// row-wise writes and the transposed reads free of bank conflicts.
// adds_prev: add the partial sums that C already holds (the running sum of the
// earlier K-parts), loaded kStoreBatch vectors at a time before the first of
// their stores.
__device__ __forceinline__ void store_c_block(const Tc3Params &p, const float (&acc)[kTcBN / 2],
                                              int row_base, int col0, uint32_t stg, int lane,
                                              bool adds_prev) {
  const int rsub = lane >> 3;   // row within each group of four
  const int cq = lane & 7;      // 16-byte chunk within the 32 columns
  constexpr int kStoreBatch = 2;   // groups of four rows loaded and stored together
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    __syncwarp();   // the previous part's transposed reads are done
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (TMM_IN_BOUNDS(in_region(lane * 128 + ((q ^ (lane & 7)) << 4), 1024, 4), &g_tc3_status))
        st_shared_v4(stg + uint32_t(lane * 128 + ((q ^ (lane & 7)) << 4)), acc[32 * b + 4 * q],
                     acc[32 * b + 4 * q + 1], acc[32 * b + 4 * q + 2], acc[32 * b + 4 * q + 3]);
    __syncwarp();
    const int col = col0 + 32 * b + 4 * cq;
    const bool vec = p.vec_store && col + 4 <= p.N;
#pragma unroll
    for (int h = 0; h < 8 / kStoreBatch; ++h) {
      float4 v[kStoreBatch], w[kStoreBatch];
#pragma unroll
      for (int u = 0; u < kStoreBatch; ++u) {
        const int r = 4 * (kStoreBatch * h + u) + rsub;
        v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (TMM_IN_BOUNDS(in_region(r * 128 + ((cq ^ (r & 7)) << 4), 1024, 4), &g_tc3_status))
          v[u] = ld_shared_v4(stg + uint32_t(r * 128 + ((cq ^ (r & 7)) << 4)));
        w[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      if (adds_prev && vec) {
#pragma unroll
        for (int u = 0; u < kStoreBatch; ++u) {
          const int row = row_base + 4 * (kStoreBatch * h + u) + rsub;
          if (row < p.M && TMM_IN_BOUNDS(in_matrix(p.C + int64_t(row) * p.ldc + col, p.C, p.M,
                                                   p.N, p.ldc, 4),
                                         &g_tc3_status))
            w[u] = __ldcg(reinterpret_cast<const float4 *>(p.C + int64_t(row) * p.ldc + col));
        }
      }
#pragma unroll
      for (int u = 0; u < kStoreBatch; ++u) {
        const int row = row_base + 4 * (kStoreBatch * h + u) + rsub;
        if (row >= p.M) continue;
        float *c_row = p.C + int64_t(row) * p.ldc;
        if (vec) {
          float4 o = v[u];
          if (adds_prev) {
            o.x = w[u].x + o.x; o.y = w[u].y + o.y; o.z = w[u].z + o.z; o.w = w[u].w + o.w;
          }
          if (TMM_IN_BOUNDS(in_matrix(c_row + col, p.C, p.M, p.N, p.ldc, 4), &g_tc3_status))
            *reinterpret_cast<float4 *>(c_row + col) = o;
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (col + j < p.N &&
                TMM_IN_BOUNDS(in_matrix(c_row + col + j, p.C, p.M, p.N, p.ldc), &g_tc3_status)) {
              float o = f4_get(v[u], j);
              if (adds_prev) o = __ldcg(c_row + col + j) + o;
              c_row[col + j] = o;
            }
        }
      }
    }
  }
}

// 320 threads: with 3 warps on some SM sub-partitions (16K registers each),
// at most 168 registers per thread.
__global__ void __launch_bounds__(kTcThreads, 1)
gemm_tc3_kernel(const __grid_constant__ CUtensorMap map_ahi,
                const __grid_constant__ CUtensorMap map_alo,
                const __grid_constant__ CUtensorMap map_bhi,
                const __grid_constant__ CUtensorMap map_blo, const Tc3Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;            // 1024-aligned stage ring
  const uint32_t bar_full = base + kTcStages * kStageBytes;
  const uint32_t bar_empty = bar_full + 8 * kTcStages;
  const uint32_t bar_tfull = bar_empty + 8 * kTcStages;    // accumulator b holds a finished chunk
  const uint32_t bar_tempty = bar_tfull + 16;              // accumulator b drained
  const uint32_t bar_drain = bar_tempty + 16;              // every product issued has completed
  const uint32_t tmem_slot = bar_drain + 8;
  const uint32_t staging = (tmem_slot + 8 + 127u) & ~127u;  // kTcAccWarps x 4 KiB
  volatile uint32_t *tmem_slot_ptr =
      reinterpret_cast<volatile uint32_t *>(smem_raw + (tmem_slot - raw));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kSlicesPerChunk = kTcChunk / kTcBK;
  unsigned int *flags =
      g_tc3_flags + (p.epoch % kTc3FlagRegions) * (kTc3MaxBlocks * kTc3FlagsPerBlock);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull + 8 * b, 1);
      mbar_init(bar_tempty + 8 * b, kTcAccWarps);
    }
    mbar_init(bar_drain, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     tmem_slot),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_d = *tmem_slot_ptr;

  bool timed_out = false;
  Tc3Work work;
  work.init(p, int(blockIdx.x), int(gridDim.x));
  int tile, kb, ke, unit;
  if (threadIdx.x == 0) {
    // Copy role: TMA loads of each work item's slices into the ring.
    int r = 0;   // ring position (slices issued so far)
    while (!timed_out && work.next(p, tile, kb, ke, unit)) {
      int tm, tn;
      tc3_tile_coords(tile, p.tiles_n, tm, tn);
      const int m0 = tm * kTcBM, n0 = tn * kTcBN;
      for (int i = kb; i < ke; ++i, ++r) {
        const int s = r % kTcStages;
        if (r >= kTcStages &&
            !mbar_wait(bar_empty + 8 * s, uint32_t((r / kTcStages) - 1) & 1u, p.wait_limit_ns)) {
          timed_out = true;
          break;
        }
        const uint32_t full = bar_full + 8 * s;
        const uint32_t st = base + s * kStageBytes;
        const int kx = i * kTcBK;
        mbar_arrive_expect_tx(full, kStageBytes);
        tma_load_2d(st, &map_ahi, kx, m0, full);
        tma_load_2d(st + kATileBytes, &map_alo, kx, m0, full);
        tma_load_2d(st + 2 * kATileBytes, &map_bhi, kx, n0, full);
        tma_load_2d(st + 2 * kATileBytes + kBTileBytes, &map_blo, kx, n0, full);
      }
    }
    if (timed_out) {
      // Let the copies already in flight land before the block goes away.
      for (int i = r > kTcStages ? r - kTcStages : 0; i < r; ++i)
        mbar_wait(bar_full + 8 * (i % kTcStages), uint32_t(i / kTcStages) & 1u, p.wait_limit_ns);
    }
  } else if (threadIdx.x == 32) {
    // Tensor-core role: three TF32 products per K-step of 8, small terms first,
    // each chunk of kSlicesPerChunk slices into accumulator (chunk count % 2).
    int r = 0;   // ring position
    int q = 0;   // chunks started so far
    while (!timed_out && work.next(p, tile, kb, ke, unit)) {
      for (int i = kb; i < ke && !timed_out; ++i, ++r) {
        const int s = r % kTcStages;
        const bool chunk_start = ((i - kb) % kSlicesPerChunk) == 0;
        if (chunk_start) {
          if (q >= 2 && !mbar_wait(bar_tempty + 8 * (q & 1), uint32_t((q >> 1) - 1) & 1u,
                                   p.wait_limit_ns)) {
            timed_out = true;
            break;
          }
          ++q;
        }
        const int buf = (q - 1) & 1;
        if (!mbar_wait(bar_full + 8 * s, uint32_t(r / kTcStages) & 1u, p.wait_limit_ns)) {
          timed_out = true;
          break;
        }
        tc_fence_after();
        const uint32_t st = base + s * kStageBytes;
        const uint32_t d = tmem_d + uint32_t(buf * kTcBN);
#pragma unroll
        for (int kk = 0; kk < kTcBK / 8; ++kk) {
          const uint32_t koff = 32u * kk;   // 8 TF32 values along K
          const uint64_t a_hi = sw64_desc(st + koff);
          const uint64_t a_lo = sw64_desc(st + kATileBytes + koff);
          const uint64_t b_hi = sw64_desc(st + 2 * kATileBytes + koff);
          const uint64_t b_lo = sw64_desc(st + 2 * kATileBytes + kBTileBytes + koff);
          mma_tf32(d, a_lo, b_hi, (chunk_start && kk == 0) ? 0u : 1u);
          mma_tf32(d, a_hi, b_lo, 1u);
          mma_tf32(d, a_hi, b_hi, 1u);
        }
        mma_commit(bar_empty + 8 * s);   // stage s is free once these products have read it
        if ((i - kb) % kSlicesPerChunk == kSlicesPerChunk - 1 || i == ke - 1)
          mma_commit(bar_tfull + 8 * buf);   // accumulator buf holds a finished chunk
      }
    }
    mma_commit(bar_drain);
    if (!mbar_wait(bar_drain, 0u, p.wait_limit_ns)) timed_out = true;
  } else if (warp >= 2) {
    // Accumulate role: warp w reads TMEM lanes 32 (w % 4).. (its rows), columns
    // half * 128.. of each finished chunk, and adds them in FP32 registers.
    // Warp w of a split tile's owner adds what warp w of the partner block
    // stored (the same rows and columns), so the two meet through one flag per
    // warp, without any block-level barrier.
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int acc_warp = warp - 2;
    int q = 0;   // chunks consumed so far
    while (!timed_out && work.next(p, tile, kb, ke, unit)) {
      float acc[kTcBN / 2];
#pragma unroll
      for (int j = 0; j < kTcBN / 2; ++j) acc[j] = 0.0f;
      const int chunks = (ke - kb + kSlicesPerChunk - 1) / kSlicesPerChunk;
      for (int c = 0; c < chunks; ++c, ++q) {
        const int buf = q & 1;
        // The whole warp takes one decision: tcgen05.ld below is warp-collective.
        const bool ready =
            mbar_wait(bar_tfull + 8 * buf, uint32_t(q >> 1) & 1u, p.wait_limit_ns);
        if (!__all_sync(0xffffffffu, ready)) {
          timed_out = true;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_d + (uint32_t(32 * quarter) << 16) +
                               uint32_t(buf * kTcBN + half * (kTcBN / 2));
#pragma unroll
        for (int cc = 0; cc < kTcBN / 2; cc += 8) {
          float v[8];
          __syncwarp();
          tmem_load_8(taddr + uint32_t(cc), v);
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[cc + j] += v[j];
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_tempty + 8 * buf);
      }
      if (timed_out) break;
      int tm, tn;
      tc3_tile_coords(tile, p.tiles_n, tm, tn);
      const int col0 = tn * kTcBN + half * (kTcBN / 2);
      // A split tile's parts run in item order: part q adds the running sum of
      // parts 0 .. q-1 (unit - 1's, in C) to its own, so every wait is for an
      // item dispatched earlier.
      const bool adds_prev = kb > 0;
      if (adds_prev) {
        if (lane == 0) {
          const unsigned int *f = &flags[(unit - 1) * kTc3FlagsPerBlock + acc_warp];
          const uint64_t t0 = timer_ns();
          while (ld_acquire_u32(f) != p.epoch) {
            if (int64_t(timer_ns() - t0) > p.wait_limit_ns) {
              atomicOr(&g_tc3_status, 2u);
              break;
            }
            __nanosleep(128);
          }
        }
        __syncwarp();
      }
      store_c_block(p, acc, tm * kTcBM + 32 * quarter, col0,
                    staging + uint32_t(acc_warp) * 4096u, lane, adds_prev);
      if (ke < p.slices) {
        // Slices [0, ke) of a split tile: this warp's running sum is in C.
        __syncwarp();
        if (lane == 0 && unit != p.drop_signal_block) {
          __threadfence();
          st_release_u32(&flags[unit * kTc3FlagsPerBlock + acc_warp], p.epoch);
        }
      }
    }
  }
  __syncwarp();
  if (timed_out) atomicOr(&g_tc3_status, 2u);

  tc_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_d),
                 "r"(kTmemCols)
                 : "memory");
}

// ---- two-SM product kernel ----------------------------------------------------------
//
// The same product on CTA pairs (a cluster of two blocks on two SMs) with
// tcgen05.mma.cta_group::2: one M = 256, N = 256, K = 8 instruction, issued by
// the pair's first block (the leader), multiplies the 256 rows of A held by
// the two blocks (128 each) with the 256 rows of B^T, also held 128 per block,
// and writes rows 0-127 of the result into the leader's tensor memory and rows
// 128-255 into the other block's.  Each block stages 128 rows of A and 128 of
// B^T per K-slice (32 KiB, against 48 KiB for a 128 x 256 tile alone), so the
// shared-memory traffic per SM, which bounds the one-block kernel, drops by a
// third; the saved space deepens the ring to six stages.
//
// The grid is persistent: one pair per resident slot, each walking its work
// items (Tc3Work), so the ring, the accumulator buffers and the chunk count
// run on from one tile to the next and a tile's stores overlap the next
// tile's first copies and products.  The copy thread starts with
// griddepcontrol.wait: the launch may begin while the split pre-pass is
// finishing (programmatic dependent launch).
//
// Synchronisation across the pair:
//   * each block's copy thread loads its own halves into its own ring; the
//     copies of both blocks complete on the leader's "full" barrier of the
//     stage (cta_group::2 bulk copies may signal the peer's barrier), and the
//     leader's copy thread announces the bytes of both;
//   * the leader's commits arrive on the "empty" and "chunk done" barriers of
//     both blocks at once (multicast), so each block's copy thread and
//     accumulate warps wait on their own barriers;
//   * the accumulate warps of both blocks release an accumulator on the
//     leader's barrier (eight local arrivals and eight remote ones);
//   * tensor memory is allocated and freed by one warp of each block together
//     (cta_group::2), and cluster barriers separate the barrier set-up from the
//     first remote arrival and the last remote arrival from the release.
// Every wait is bounded as in the one-block kernel.

constexpr int kT2Rows = 128;                       // rows of A and of B^T staged per block
constexpr int kT2BM = 2 * kT2Rows;                 // rows of C per pair tile
constexpr int kT2BN = 256;                         // columns of C per pair tile
constexpr int kT2Stages = 6;
constexpr uint32_t kT2TileBytes = kT2Rows * kTcBK * 4;    // 8 KiB
constexpr uint32_t kT2StageBytes = 4 * kT2TileBytes;      // A hi, A lo, B^T hi, B^T lo
constexpr uint32_t kT2BarrierBytes = 8 * (2 * kT2Stages + 5) + 8;
constexpr uint32_t kT2SmemBytes =
    1024 + kT2Stages * kT2StageBytes + kT2BarrierBytes + 128 + kStagingBytes;
static_assert(kT2SmemBytes <= kMaxSmemPerBlock, "ring, barriers and staging fit one block");
static_assert(kT2StageBytes % 1024 == 0 && kT2TileBytes % 1024 == 0, "tiles stay 1024-byte aligned");
static_assert(kT2BN == kTcBN, "each block's accumulator keeps the one-block layout");

// M = 256 (the pair), N = 256.
constexpr uint32_t kIdescTf32Pair = (1u << 4) | (2u << 7) | (2u << 10) |
                                    (uint32_t(kT2BN >> 3) << 17) | (uint32_t(kT2BM >> 4) << 24);

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of both blocks of the pair.
__device__ __forceinline__ void pair_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// The shared::cluster address of `addr` (this block's shared memory) in block `rank`.
__device__ __forceinline__ uint32_t map_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                                  int64_t limit_ns) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = timer_ns();
  while (!mbar_try_wait_cluster(bar, parity))
    if (int64_t(timer_ns() - t0) > limit_ns) return false;
  return true;
}
// Bulk tensor copy into this block's shared memory whose completion is
// counted on `bar`, a shared::cluster address in either block of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, int x,
                                                 int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void mma_tf32_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %3, 0;\n"
      " tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %4, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(accumulate), "r"(kIdescTf32Pair)
      : "memory");
}
// Arrive on the barrier at offset `bar` of every block in `mask` once the pair
// products issued so far by this thread have completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

__global__ void __launch_bounds__(kTcThreads, 1)
gemm_tc3_pair_kernel(const __grid_constant__ CUtensorMap map_ahi,
                     const __grid_constant__ CUtensorMap map_alo,
                     const __grid_constant__ CUtensorMap map_bhi,
                     const __grid_constant__ CUtensorMap map_blo, const Tc3Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;            // same offsets in both blocks
  const uint32_t bar_full = base + kT2Stages * kT2StageBytes;
  const uint32_t bar_empty = bar_full + 8 * kT2Stages;
  const uint32_t bar_tfull = bar_empty + 8 * kT2Stages;
  const uint32_t bar_tempty = bar_tfull + 16;              // used in the leader
  const uint32_t bar_drain = bar_tempty + 16;              // used in the leader
  const uint32_t tmem_slot = bar_drain + 8;
  const uint32_t staging = (tmem_slot + 8 + 127u) & ~127u;  // kTcAccWarps x 4 KiB
  volatile uint32_t *tmem_slot_ptr =
      reinterpret_cast<volatile uint32_t *>(smem_raw + (tmem_slot - raw));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = int(blockIdx.x >> 1);
  constexpr int kSlicesPerChunk = kTcChunk / kTcBK;
  unsigned int *flags =
      g_tc3_flags + (p.epoch % kTc3FlagRegions) * (kTc3MaxBlocks * kTc3FlagsPerBlock);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kT2Stages; ++s) {
      mbar_init(bar_full + 8 * s, 1);     // used in the leader
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull + 8 * b, 1);
      mbar_init(bar_tempty + 8 * b, 2 * kTcAccWarps);
    }
    mbar_init(bar_drain, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     tmem_slot),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  pair_sync();          // both blocks' barriers exist before any arrival crosses the pair
  tc_fence_after();
  const uint32_t tmem_d = *tmem_slot_ptr;

  bool timed_out = false;
  Tc3Work work;
  work.init(p, pair, int(gridDim.x >> 1));
  int tile, kb, ke, unit;
  if (threadIdx.x == 0) {
    // Copy role (both blocks): this block's 128 rows of A and of B^T per slice.
    // The launch may overlap the split pre-pass (programmatic dependent launch):
    // wait until it has completed and its writes are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint32_t leader_full = map_rank(bar_full, 0);
    int r = 0;
    while (!timed_out && work.next(p, tile, kb, ke, unit)) {
      int tm, tn;
      tc3_tile_coords(tile, p.tiles_n, tm, tn);
      const int m0 = tm * kT2BM + int(rank) * kT2Rows;
      const int nb0 = tn * kT2BN + int(rank) * kT2Rows;
      for (int i = kb; i < ke; ++i, ++r) {
        const int s = r % kT2Stages;
        if (r >= kT2Stages &&
            !mbar_wait_cluster(bar_empty + 8 * s, uint32_t((r / kT2Stages) - 1) & 1u,
                               p.wait_limit_ns)) {
          timed_out = true;
          break;
        }
        const uint32_t full = leader_full + 8 * s;
        const uint32_t st = base + s * kT2StageBytes;
        const int kx = i * kTcBK;
        if (leader) mbar_arrive_expect_tx(bar_full + 8 * s, 2 * kT2StageBytes);
        tma_load_2d_pair(st, &map_ahi, kx, m0, full);
        tma_load_2d_pair(st + kT2TileBytes, &map_alo, kx, m0, full);
        tma_load_2d_pair(st + 2 * kT2TileBytes, &map_bhi, kx, nb0, full);
        tma_load_2d_pair(st + 3 * kT2TileBytes, &map_blo, kx, nb0, full);
      }
    }
    if (timed_out && leader) {
      // The leader's barriers count both blocks' copies: once they complete,
      // nothing is in flight into either block.
      for (int i = r > kT2Stages ? r - kT2Stages : 0; i < r; ++i)
        mbar_wait_cluster(bar_full + 8 * (i % kT2Stages), uint32_t(i / kT2Stages) & 1u,
                          p.wait_limit_ns);
    }
  } else if (threadIdx.x == 32 && leader) {
    // Tensor-core role (leader): as in the one-block kernel, on pair instructions.
    int r = 0;
    int q = 0;
    while (!timed_out && work.next(p, tile, kb, ke, unit)) {
      for (int i = kb; i < ke && !timed_out; ++i, ++r) {
        const int s = r % kT2Stages;
        const bool chunk_start = ((i - kb) % kSlicesPerChunk) == 0;
        if (chunk_start) {
          if (q >= 2 && !mbar_wait_cluster(bar_tempty + 8 * (q & 1),
                                           uint32_t((q >> 1) - 1) & 1u, p.wait_limit_ns)) {
            timed_out = true;
            break;
          }
          ++q;
        }
        const int buf = (q - 1) & 1;
        if (!mbar_wait_cluster(bar_full + 8 * s, uint32_t(r / kT2Stages) & 1u,
                               p.wait_limit_ns)) {
          timed_out = true;
          break;
        }
        tc_fence_after();
        const uint32_t st = base + s * kT2StageBytes;
        const uint32_t d = tmem_d + uint32_t(buf * kT2BN);
#pragma unroll
        for (int kk = 0; kk < kTcBK / 8; ++kk) {
          const uint32_t koff = 32u * kk;
          const uint64_t a_hi = sw64_desc(st + koff);
          const uint64_t a_lo = sw64_desc(st + kT2TileBytes + koff);
          const uint64_t b_hi = sw64_desc(st + 2 * kT2TileBytes + koff);
          const uint64_t b_lo = sw64_desc(st + 3 * kT2TileBytes + koff);
          mma_tf32_pair(d, a_lo, b_hi, (chunk_start && kk == 0) ? 0u : 1u);
          mma_tf32_pair(d, a_hi, b_lo, 1u);
          mma_tf32_pair(d, a_hi, b_hi, 1u);
        }
        mma_commit_pair(bar_empty + 8 * s, 3);          // both blocks' stage s is free
        if ((i - kb) % kSlicesPerChunk == kSlicesPerChunk - 1 || i == ke - 1)
          mma_commit_pair(bar_tfull + 8 * buf, 3);      // both halves of accumulator buf ready
      }
    }
    mma_commit_pair(bar_drain, 1);
    if (!mbar_wait(bar_drain, 0u, p.wait_limit_ns)) timed_out = true;
  } else if (warp >= 2) {
    // Accumulate role (both blocks): this block's 128 rows of the pair tile.
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int acc_warp = warp - 2;
    const uint32_t tempty = leader ? bar_tempty : map_rank(bar_tempty, 0);
    int q = 0;
    while (!timed_out && work.next(p, tile, kb, ke, unit)) {
      float acc[kT2BN / 2];
#pragma unroll
      for (int j = 0; j < kT2BN / 2; ++j) acc[j] = 0.0f;
      const int chunks = (ke - kb + kSlicesPerChunk - 1) / kSlicesPerChunk;
      for (int c = 0; c < chunks; ++c, ++q) {
        const int buf = q & 1;
        const bool ready =
            mbar_wait_cluster(bar_tfull + 8 * buf, uint32_t(q >> 1) & 1u, p.wait_limit_ns);
        if (!__all_sync(0xffffffffu, ready)) {
          timed_out = true;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_d + (uint32_t(32 * quarter) << 16) +
                               uint32_t(buf * kT2BN + half * (kT2BN / 2));
#pragma unroll
        for (int cc = 0; cc < kT2BN / 2; cc += 8) {
          float v[8];
          __syncwarp();
          tmem_load_8(taddr + uint32_t(cc), v);
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[cc + j] += v[j];
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader) mbar_arrive(tempty + 8 * buf);
          else mbar_arrive_remote(tempty + 8 * buf);
        }
      }
      if (timed_out) break;
      int tm, tn;
      tc3_tile_coords(tile, p.tiles_n, tm, tn);
      const int col0 = tn * kT2BN + half * (kT2BN / 2);
      const int flag = int(rank) * kTcAccWarps + acc_warp;   // per block of the pair and warp
      const bool adds_prev = kb > 0;   // slices [0, kb): unit - 1's running sum, in C
      if (adds_prev) {
        if (lane == 0) {
          const unsigned int *f = &flags[(unit - 1) * 2 * kTcAccWarps + flag];
          const uint64_t t0 = timer_ns();
          while (ld_acquire_u32(f) != p.epoch) {
            if (int64_t(timer_ns() - t0) > p.wait_limit_ns) {
              atomicOr(&g_tc3_status, 2u);
              break;
            }
            __nanosleep(128);
          }
        }
        __syncwarp();
      }
      store_c_block(p, acc, tm * kT2BM + int(rank) * kT2Rows + 32 * quarter, col0,
                    staging + uint32_t(acc_warp) * 4096u, lane, adds_prev);
      if (ke < p.slices) {
        __syncwarp();
        if (lane == 0 && unit != p.drop_signal_block) {
          __threadfence();
          st_release_u32(&flags[unit * 2 * kTcAccWarps + flag], p.epoch);
        }
      }
    }
  }
  __syncwarp();
  if (timed_out) atomicOr(&g_tc3_status, 2u);

  tc_fence_before();
  __syncthreads();
  pair_sync();          // every remote arrival has landed; neither block uses tensor memory
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_d),
                 "r"(kTmemCols)
                 : "memory");
}

// ---- host side ------------------------------------------------------------------

int64_t pad_k(int64_t K) { return (K + kKPad - 1) / kKPad * kKPad; }
size_t round256(size_t b) { return (b + 255) / 256 * 256; }

// K-major operand: `rows` rows of `kdim` floats, `ld` floats apart; box of
// kTcBK x box_rows, 64-byte swizzle.  Reads past kdim or rows return zeros.
cudaError_t encode_operand(CUtensorMap *map, const float *base, int64_t rows, int64_t kdim,
                           int64_t ld, uint32_t box_rows) {
  return encode_f32_2d(map, base, rows, kdim, ld, uint32_t(kTcBK), box_rows,
                       CU_TENSOR_MAP_SWIZZLE_64B);
}

std::atomic<uint64_t> g_tc3_configured{0};
std::atomic<int> g_tc3_blocks_per_sm[64];
std::atomic<int64_t> g_tc3_wait_limit_ns{int64_t(10) * 1000 * 1000 * 1000};
std::atomic<unsigned int> g_tc3_epoch{0};
std::atomic<int> g_tc3_drop_signal_block{-1};

// Work split shared by both kernels: whole tiles, and when the last wave is at
// most half full, its tiles in two K-parts; with at most half as many tiles as
// slots, every tile in up to kTc3MaxParts K-parts of at least two chunks each,
// one slot each (measured: each hand-over of a running sum costs about half a
// chunk's products, so one-chunk parts lose more than they gain).
constexpr int kTc3MaxParts = 4;
// Returns the item count (the caller rejects one past the int range).
int64_t plan_tiles(Tc3Params &prm, int64_t tiles, int64_t slots, int max_units, int slices) {
  constexpr int kSlicesPerChunk = kTcChunk / kTcBK;
  const int64_t chunks = (slices + kSlicesPerChunk - 1) / kSlicesPerChunk;
  const int64_t rem = slots > 0 ? tiles % slots : 0;
  prm.slices = slices;
  prm.chunks = int(chunks);
  prm.parts = 1;
  prm.dp_tiles = int(tiles);
  if (tiles > slots && rem > 0 && 2 * rem <= slots && 2 * rem <= max_units && chunks >= 2) {
    prm.parts = 2;
    prm.dp_tiles = int(tiles - rem);
  } else if (tiles > 0 && 2 * tiles <= slots && chunks >= 4) {
    int64_t parts = std::min<int64_t>({slots / tiles, chunks / 2, int64_t(kTc3MaxParts)});
    if (parts * tiles <= max_units) {
      prm.parts = int(parts);
      prm.dp_tiles = 0;
    }
  }
  const int64_t items = prm.dp_tiles + prm.parts * (tiles - prm.dp_tiles);
  prm.items = int(items);
  return items;
}

unsigned int next_epoch() {
  unsigned int ep = g_tc3_epoch.fetch_add(1, std::memory_order_relaxed) + 1;
  if (ep == 0) ep = g_tc3_epoch.fetch_add(1, std::memory_order_relaxed) + 1;
  return ep;
}

std::atomic<uint64_t> g_tc3_pair_configured{0};
std::atomic<int> g_tc3_pair_slots[64];

cudaError_t launch_tc3_pairs(const GemmProblem &p, const DeviceInfo &dev, int64_t Kp,
                             const CUtensorMap (&maps)[4], cudaStream_t stream) {
  auto kernel = gemm_tc3_pair_kernel;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.blockDim = dim3(kTcThreads, 1, 1);
  cfg.dynamicSmemBytes = kT2SmemBytes;
  cfg.stream = stream;
  const uint64_t bit = uint64_t(1) << (dev.id & 63);
  if (!(g_tc3_pair_configured.load(std::memory_order_acquire) & bit)) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(kT2SmemBytes));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(2 * 64, 1, 1);   // shape only, for the query
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (clusters < 1) return cudaErrorLaunchOutOfResources;
    g_tc3_pair_slots[dev.id & 63].store(clusters, std::memory_order_relaxed);
    g_tc3_pair_configured.fetch_or(bit, std::memory_order_release);
  }
  const int64_t slots = g_tc3_pair_slots[dev.id & 63].load(std::memory_order_relaxed);
  const int64_t tiles_m = (p.M + kT2BM - 1) / kT2BM;
  const int64_t tiles_n = (p.N + kT2BN - 1) / kT2BN;
  const int64_t tiles = tiles_m * tiles_n;
  Tc3Params prm = {};
  prm.M = int(p.M);
  prm.N = int(p.N);
  prm.Kp = int(Kp);
  prm.C = p.C;
  prm.ldc = p.ldc;
  prm.tiles_m = int(tiles_m);
  prm.tiles_n = int(tiles_n);
  // Split units use flags per (unit, block of the pair, warp): half as many units fit.
  const int64_t items = plan_tiles(prm, tiles, slots, kTc3MaxBlocks / 2, int(Kp / kTcBK));
  if (tiles > 0x7fffffff || items > 0x7fffffff) return cudaErrorInvalidConfiguration;
  prm.vec_store = ((reinterpret_cast<uintptr_t>(p.C) & 15u) == 0 && p.ldc % 4 == 0) ? 1 : 0;
  prm.wait_limit_ns = g_tc3_wait_limit_ns.load(std::memory_order_relaxed);
  prm.drop_signal_block = g_tc3_drop_signal_block.load(std::memory_order_relaxed);
  prm.epoch = next_epoch();
  // Persistent: one pair per resident slot, each walking its items; the next
  // tile's copies and products start while the previous tile is being stored.
  cfg.gridDim = dim3(unsigned(2 * std::min<int64_t>(items, slots)), 1, 1);
  // Start the blocks (barriers, tensor memory) while the split pre-pass
  // finishes; the copy thread waits for it before reading (griddepcontrol.wait).
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, maps[0], maps[1], maps[2], maps[3], prm);
}

}  // namespace

size_t tc3_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  // In 128-bit arithmetic: with sizes up to 2^31 - 1 the count reaches about
  // 2^68 bytes, which size_t cannot hold; such products get SIZE_MAX.
  const __int128 Kp = pad_k(K);
  const auto part = [](__int128 b) { return (b + 255) / 256 * 256; };
  const __int128 total = 2 * part(__int128(M) * Kp * 4) + 2 * part(__int128(N) * Kp * 4);
  return total >= __int128(SIZE_MAX) ? SIZE_MAX : size_t(total);
}

cudaError_t launch_tc3(const GemmProblem &p, const DeviceInfo &dev, void *workspace,
                       cudaStream_t stream) {
  cudaError_t e = tensor_map_encoder_ready();
  if (e != cudaSuccess) return e;
  const int64_t Kp = pad_k(p.K);
  char *ws = static_cast<char *>(workspace);
  float *a_hi = reinterpret_cast<float *>(ws);
  float *a_lo = reinterpret_cast<float *>(ws + round256(size_t(p.M) * Kp * 4));
  float *b_hi = reinterpret_cast<float *>(ws + 2 * round256(size_t(p.M) * Kp * 4));
  float *b_lo = reinterpret_cast<float *>(ws + 2 * round256(size_t(p.M) * Kp * 4) +
                                          round256(size_t(p.N) * Kp * 4));

  // The tensor core reads a TF32 operand from an FP32 word by ignoring its low
  // 13 mantissa bits -- exactly the hi of the split (measured: products from
  // raw FP32 words and from masked ones agree bit for bit).  So an operand
  // already stored K-major (A as M x K, B as N x K) whose rows start on
  // 16-byte boundaries serves as its own hi: only lo is written for it.
  const bool raw_a = !p.transa && p.K > 0 &&
                     (reinterpret_cast<uintptr_t>(p.A) & 15u) == 0 && p.lda % 4 == 0;
  const bool raw_b = p.transb && p.K > 0 &&
                     (reinterpret_cast<uintptr_t>(p.B) & 15u) == 0 && p.ldb % 4 == 0;

  // 1. split pre-pass: op(A) -> M x Kp and op(B)^T -> N x Kp, K-major.  An
  // operand stored with K contiguous (A as M x K, B as N x K) is split row by
  // row; one stored with K as its rows (A as K x M, B as K x N) is transposed.
  {
    auto split_rows = [&](const float *src, int64_t ld, int64_t rows, float *hi, float *lo,
                          bool write_hi) {
      const bool vec = (reinterpret_cast<uintptr_t>(src) & 15u) == 0 && ld % 4 == 0;
      const dim3 grid(unsigned((Kp / 4 + 255) / 256), unsigned(std::min<int64_t>(rows, 65535)));
      tc3_split_a_kernel<<<grid, 256, 0, stream>>>(int(rows), int(p.K), int(Kp), src, ld,
                                                   vec ? 1 : 0, write_hi ? 1 : 0, hi, lo);
      return cudaGetLastError();
    };
    auto split_transposed = [&](const float *src, int64_t ld, int64_t cols, float *hi,
                                float *lo) {
      const dim3 grid(unsigned((cols + 31) / 32), unsigned(Kp / 32));
      tc3_split_bt_kernel<<<grid, dim3(32, 8), 0, stream>>>(int(p.K), int(cols), int(Kp), src,
                                                            ld, hi, lo);
      return cudaGetLastError();
    };
    e = p.transa ? split_transposed(p.A, p.lda, p.M, a_hi, a_lo)
                 : split_rows(p.A, p.lda, p.M, a_hi, a_lo, !raw_a);
    if (e != cudaSuccess) return e;
    e = p.transb ? split_rows(p.B, p.ldb, p.N, b_hi, b_lo, !raw_b)
                 : split_transposed(p.B, p.ldb, p.N, b_hi, b_lo);
    if (e != cudaSuccess) return e;
  }

  // 2. product kernel: on block pairs once A has more rows than one block's
  // tile (each block then stages 128 rows of B^T as well), else one block per
  // tile.  (Measured: pairs are faster at every K from 128 up once M > 128.)
  const bool pairs = p.M > kTcBM;
  CUtensorMap maps[4];
  const uint32_t b_box = pairs ? uint32_t(kT2Rows) : uint32_t(kTcBN);
  e = raw_a ? encode_operand(&maps[0], p.A, p.M, p.K, p.lda, kTcBM)
            : encode_operand(&maps[0], a_hi, p.M, Kp, Kp, kTcBM);
  if (e != cudaSuccess) return e;
  e = raw_b ? encode_operand(&maps[2], p.B, p.N, p.K, p.ldb, b_box)
            : encode_operand(&maps[2], b_hi, p.N, Kp, Kp, b_box);
  if (e != cudaSuccess) return e;
  if ((e = encode_operand(&maps[1], a_lo, p.M, Kp, Kp, kTcBM)) != cudaSuccess ||
      (e = encode_operand(&maps[3], b_lo, p.N, Kp, Kp, b_box)) != cudaSuccess)
    return e;
  if (pairs) return launch_tc3_pairs(p, dev, Kp, maps, stream);
  const uint64_t bit = uint64_t(1) << (dev.id & 63);
  if (!(g_tc3_configured.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(gemm_tc3_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kTcSmemBytes));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gemm_tc3_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    int nb = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, gemm_tc3_kernel, kTcThreads,
                                                      kTcSmemBytes);
    if (e != cudaSuccess) return e;
    if (nb < 1) return cudaErrorLaunchOutOfResources;
    g_tc3_blocks_per_sm[dev.id & 63].store(nb, std::memory_order_relaxed);
    g_tc3_configured.fetch_or(bit, std::memory_order_release);
  }
  // One block per tile; a last wave at most half full is split along K.
  const int64_t tiles_m = (p.M + kTcBM - 1) / kTcBM;
  const int64_t tiles_n = (p.N + kTcBN - 1) / kTcBN;
  const int64_t tiles = tiles_m * tiles_n;
  const int64_t slots =
      int64_t(g_tc3_blocks_per_sm[dev.id & 63].load(std::memory_order_relaxed)) * dev.sm_count;
  Tc3Params prm = {};
  prm.M = int(p.M);
  prm.N = int(p.N);
  prm.Kp = int(Kp);
  prm.C = p.C;
  prm.ldc = p.ldc;
  prm.tiles_m = int(tiles_m);
  prm.tiles_n = int(tiles_n);
  const int64_t grid = plan_tiles(prm, tiles, slots, kTc3MaxBlocks, int(Kp / kTcBK));   // one block per item
  if (tiles > 0x7fffffff || grid > 0x7fffffff) return cudaErrorInvalidConfiguration;
  prm.vec_store = ((reinterpret_cast<uintptr_t>(p.C) & 15u) == 0 && p.ldc % 4 == 0) ? 1 : 0;
  prm.wait_limit_ns = g_tc3_wait_limit_ns.load(std::memory_order_relaxed);
  prm.drop_signal_block = g_tc3_drop_signal_block.load(std::memory_order_relaxed);
  prm.epoch = next_epoch();

  gemm_tc3_kernel<<<unsigned(grid), kTcThreads, kTcSmemBytes, stream>>>(maps[0], maps[1],
                                                                       maps[2], maps[3], prm);
  return cudaGetLastError();
}

cudaError_t tc3_device_status(unsigned int *status, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(status, g_tc3_status, sizeof(unsigned int));
  if (e != cudaSuccess || !clear) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_tc3_status, &zero, sizeof(unsigned int));
}

void tc3_plan_for_testing(int64_t M, int64_t N, int64_t K, int pairs, int64_t slots,
                          int64_t out[6]) {
  const int64_t BM = pairs ? kT2BM : kTcBM, BN = pairs ? kT2BN : kTcBN;
  const int64_t tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  Tc3Params prm = {};
  const int64_t items = plan_tiles(prm, tiles, slots, pairs ? kTc3MaxBlocks / 2 : kTc3MaxBlocks,
                                   int(pad_k(K) / kTcBK));
  out[0] = tiles;
  out[1] = items;
  out[2] = prm.dp_tiles;
  out[3] = prm.parts;
  out[4] = prm.chunks;
  out[5] = prm.slices;
}

void tc3_set_test_hooks(int drop_signal_block, int64_t wait_limit_ns) {
  g_tc3_drop_signal_block.store(drop_signal_block, std::memory_order_relaxed);
  g_tc3_wait_limit_ns.store(wait_limit_ns > 0 ? wait_limit_ns : int64_t(10) * 1000 * 1000 * 1000,
                            std::memory_order_relaxed);
}

}  // namespace tmm
