// gemm_simt.cu -- two-level tiled FP32 product on the CUDA cores (FFMA).
//
// Tiling ("Tiling Strategies" sections 2-4, "CMU DLSys Lecture 12" section 5):
//   * block tile: each 128-thread block (4 warps, 2 x 2) owns a 128 x 128 tile
//     of C; two blocks are resident per SM;
//   * K-slices of BK = 16 flow through a ring of kStages shared-memory stages
//     filled by asynchronous copies (cp.async).  This generalises the double
//     buffer of "Tiling Strategies" section 3: the copies of the next
//     kStages - 1 slices are in flight while one slice is consumed, and no
//     register holds staged data;
//   * thread tile: each thread owns a 16 x 8 tile of C (128 accumulators) and
//     performs one outer product per k, 16 + 8 operands for 128 FFMA, with the
//     operands of step k+1 loaded from shared memory while step k's FFMAs
//     issue ("Tiling Hierarchy on GPUs", "Register Tiling", "Register
//     prefetching", "Reducing Overhead Slots").
//
// Shared-memory layout.  The A slab is stored transposed, a[k][m], so a
// thread's rows of A at one k are 16-byte vectors; it is filled by 4-byte
// copies, each warp copying 4 rows x 8 consecutive k (four 32-byte global
// sectors) into 32 distinct banks (row length BM + 4 floats).  The B slab
// keeps its global layout b[k][n] and is filled by 16-byte copies of whole
// 512-byte row segments when B is 16-byte aligned (4-byte copies otherwise).
//
// Warp tiling ("Tiling Hierarchy on GPUs", "Warp Tiling"): each warp covers a
// 64 x 64 region of C; lane (lm, ln), lm in 0..3, ln in 0..7, owns rows
// lm*4 + 16t + i and columns ln*4 + 32c + j (t < 4, c < 2, i, j < 4).  A
// 128-bit shared load is served at most 16 lanes per wavefront, and the two
// quarter-warps of a half-warp share a wavefront only when they read disjoint
// words with lanes that share a word paired up.  With quarter q = lane / 8,
//     lm = lane % 2 + 2 (q % 2),
//     ln = (lane / 2) % 4 + 4 ((q % 2) xor (q / 2)),
// every fragment load, of A or of B, takes two wavefronts, the minimum.
//
// Tails ("CMU DLSys Lecture 12" section 5): copies outside M, N or K are
// zero-filled (source size 0), which adds nothing to the sums, and only
// entries inside M x N are stored.
//
// Scheduling: tiles are numbered along a grouped raster -- kGroupM tile-rows
// are walked column by column -- so blocks resident at the same time share
// the A row-panels and B column-panels they read through L2.
#include <atomic>

#include "tmm_internal.h"

namespace tmm {
namespace {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int BK = 16;
constexpr int kStages = 4;
constexpr int TM = 16;                       // thread tile rows
constexpr int TN = 8;                        // thread tile columns
constexpr int kWarpsM = 2, kWarpsN = 2;
constexpr int kThreads = 32 * kWarpsM * kWarpsN;  // 128
constexpr int kAsLd = BM + 4;                // row of the transposed A slab (floats)
constexpr int kBsLd = BN;
constexpr int kStageFloats = BK * kAsLd + BK * kBsLd;
constexpr int kSmemBytes = kStages * kStageFloats * 4;
constexpr int kGroupM = 16;
constexpr int kKUnroll = 4;                  // k steps per iteration of the inner loop

static_assert(BM == kWarpsM * 4 * TM && BN == kWarpsN * 8 * TN, "warp tile is 4 x 8 lanes");
static_assert(BM * BK == kThreads * 16, "each thread copies 16 elements of the A slab");
static_assert(BK * BN == kThreads * 16, "each thread copies 16 elements of the B slab");
static_assert(BK % kKUnroll == 0 && kKUnroll % 2 == 0, "inner loop ping-pongs fragments");

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Asynchronous global->shared copies; a false predicate copies zero bytes and
// zero-fills the destination.  The source is then not read, and is replaced by
// `safe` (an address inside the operand) all the same.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const float *src, bool pred,
                                           const float *safe) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst),
               "l"(pred ? src : safe), "r"(pred ? 4 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_16(uint32_t dst, const float *src, bool pred,
                                            const float *safe) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst),
               "l"(pred ? src : safe), "r"(pred ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void tile_coords(int tile, int tiles_m, int tiles_n, int &tm,
                                            int &tn) {
  const int per_group = kGroupM * tiles_n;
  const int group = tile / per_group;
  const int first_m = group * kGroupM;
  const int rows = min(tiles_m - first_m, kGroupM);
  const int in_group = tile - group * per_group;
  tm = first_m + in_group % rows;
  tn = in_group / rows;
}

// kVecB:     B is 16-byte aligned and ldb, N are multiples of 4 (16-byte copies).
// kVecStore: C is 16-byte aligned and ldc, N are multiples of 4.
template <bool kVecB, bool kVecStore>
__global__ void __launch_bounds__(kThreads, 2)
gemm_simt_kernel(int M, int N, int K,
                 const float *__restrict__ A, int64_t lda,
                 const float *__restrict__ B, int64_t ldb,
                 float *__restrict__ C, int64_t ldc, int tiles_m, int tiles_n) {
  extern __shared__ __align__(16) float smem[];

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  int tm, tn;
  tile_coords(blockIdx.x, tiles_m, tiles_n, tm, tn);
  const int m0 = tm * BM;
  const int n0 = tn * BN;

  // ---- copy assignment -------------------------------------------------------
  // A: element `it` (0..15) of this thread is row a_r0 + 16 (it/2), k a_k0 + 8 (it%2).
  const int a_r0 = (lane >> 3) + 4 * warp;
  const int a_k0 = lane & 7;
  uint32_t a_rows_ok = 0;                      // bit r: row a_r0 + 16 r inside M
#pragma unroll
  for (int r = 0; r < 8; ++r) a_rows_ok |= uint32_t(m0 + a_r0 + 16 * r < M) << r;
  const float *a_src = A + int64_t(min(m0 + a_r0, M - 1)) * lda + a_k0;
  const int64_t a_row_step = 16 * lda;
  const uint32_t a_dst0 = smem_addr(smem) + 4u * (a_k0 * kAsLd + a_r0);

  // B: vectorised, vector v (0..3) is k row b_k0 + 4v, columns b_n0..b_n0+3;
  //    scalar, element it (0..15) is k row b_k0 + 4 (it/4), column lane + 32 (it%4).
  const int b_k0 = tid >> 5;
  const int b_n0 = kVecB ? (tid & 31) * 4 : lane;
  const float *b_src = B + int64_t(b_k0) * ldb + min(n0 + b_n0, N - 1);
  const int64_t b_row4_step = 4 * ldb;
  const uint32_t b_dst0 = smem_addr(smem) + 4u * (BK * kAsLd + b_k0 * kBsLd + b_n0);

  const int num_slices = (K + BK - 1) / BK;

  auto issue_slice = [&](int s, int stage) {
    const int k0 = s * BK;
    const uint32_t st_off = 4u * stage * kStageFloats;
    const float *a = a_src + k0;
#pragma unroll
    for (int it = 0; it < 16; ++it) {
      const int r = it >> 1, h = it & 1;
      const bool ok = ((a_rows_ok >> r) & 1u) && (k0 + a_k0 + 8 * h < K);
      cp_async_4(a_dst0 + st_off + 4u * (8 * h * kAsLd + 16 * r), a + r * a_row_step + 8 * h,
                 ok, A);
    }
    const float *b = b_src + int64_t(k0) * ldb;
    if (kVecB) {
      const bool col_ok = n0 + b_n0 < N;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const bool ok = col_ok && (k0 + b_k0 + 4 * v < K);
        cp_async_16(b_dst0 + st_off + 4u * (4 * v * kBsLd), b + v * b_row4_step, ok, B);
      }
    } else {
#pragma unroll
      for (int it = 0; it < 16; ++it) {
        const int v = it >> 2, c = it & 3;
        const bool ok = (n0 + b_n0 + 32 * c < N) && (k0 + b_k0 + 4 * v < K);
        cp_async_4(b_dst0 + st_off + 4u * (4 * v * kBsLd + 32 * c), b + v * b_row4_step + 32 * c,
                   ok, B);
      }
    }
  };

  // ---- fragment placement ----------------------------------------------------
  const int q = lane >> 3;
  const int lm = (lane & 1) + 2 * (q & 1);
  const int ln = ((lane >> 1) & 3) + 4 * ((q & 1) ^ (q >> 1));
  const int wm = warp / kWarpsN, wn = warp % kWarpsN;
  const int a_off = wm * (4 * TM) + lm * 4;   // + 16 t
  const int b_off = wn * (8 * TN) + ln * 4;   // + 32 c

  float acc[TM][TN];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) acc[i][j] = 0.0f;

  auto load_frag = [&](const float *st, int k, float (&af)[TM], float (&bf)[TN]) {
    const float *as = st + k * kAsLd + a_off;
    const float *bs = st + BK * kAsLd + k * kBsLd + b_off;
#pragma unroll
    for (int t = 0; t < TM / 4; ++t) {
      const float4 v = *reinterpret_cast<const float4 *>(as + 16 * t);
      af[4 * t + 0] = v.x; af[4 * t + 1] = v.y; af[4 * t + 2] = v.z; af[4 * t + 3] = v.w;
    }
#pragma unroll
    for (int c = 0; c < TN / 4; ++c) {
      const float4 v = *reinterpret_cast<const float4 *>(bs + 32 * c);
      bf[4 * c + 0] = v.x; bf[4 * c + 1] = v.y; bf[4 * c + 2] = v.z; bf[4 * c + 3] = v.w;
    }
  };
  auto outer_product = [&](const float (&af)[TM], const float (&bf)[TN]) {
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(af[i], bf[j], acc[i][j]);
  };

  // ---- pipeline ----------------------------------------------------------------
#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < num_slices) issue_slice(s, s);
    cp_async_commit();
  }

  float af[2][TM], bf[2][TN];
  int stage = 0;
  for (int s = 0; s < num_slices; ++s) {
    cp_async_wait<kStages - 2>();   // slice s has landed (this thread's copies) ...
    __syncthreads();                // ... and everyone's; slice s-1's stage is free
    {
      const int sn = s + kStages - 1;
      int stage_n = stage + kStages - 1;
      if (stage_n >= kStages) stage_n -= kStages;
      if (sn < num_slices) issue_slice(sn, stage_n);
      cp_async_commit();
    }
    const float *st = smem + stage * kStageFloats;
    load_frag(st, 0, af[0], bf[0]);
#pragma unroll 1
    for (int kk = 0; kk < BK; kk += kKUnroll) {
#pragma unroll
      for (int u = 0; u < kKUnroll; ++u) {
        const int k = kk + u;
        if (u + 1 < kKUnroll || k + 1 < BK) load_frag(st, k + 1, af[(u + 1) & 1], bf[(u + 1) & 1]);
        outer_product(af[u & 1], bf[u & 1]);
      }
    }
    if (++stage == kStages) stage = 0;
  }
  cp_async_wait<0>();

  // ---- epilogue: accumulator (4t + i, 4c + j) is C[m0 + a_off + 16t + i][n0 + b_off + 32c + j]
  const int row0 = m0 + a_off;
  const int col0 = n0 + b_off;
  float *c_base = C + int64_t(row0) * ldc + col0;
#pragma unroll
  for (int t = 0; t < TM / 4; ++t) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int dr = 16 * t + i;
      if (row0 + dr >= M) continue;
      float *c_row = c_base + int64_t(dr) * ldc;
      const float *a = acc[4 * t + i];
#pragma unroll
      for (int c = 0; c < TN / 4; ++c) {
        const int dc = 32 * c;
        if (kVecStore) {
          if (col0 + dc < N)
            *reinterpret_cast<float4 *>(c_row + dc) =
                make_float4(a[4 * c], a[4 * c + 1], a[4 * c + 2], a[4 * c + 3]);
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (col0 + dc + j < N) c_row[dc + j] = a[4 * c + j];
        }
      }
    }
  }
}

// Dynamic shared memory above 48 KiB needs an opt-in per kernel and device.
std::atomic<uint64_t> g_smem_configured[4];

template <bool kVecB, bool kVecStore>
cudaError_t launch_variant(const GemmProblem &p, const DeviceInfo &dev, cudaStream_t stream) {
  auto kernel = gemm_simt_kernel<kVecB, kVecStore>;
  const int variant = (kVecB ? 2 : 0) + (kVecStore ? 1 : 0);
  const uint64_t bit = uint64_t(1) << (dev.id & 63);
  if (!(g_smem_configured[variant].load(std::memory_order_acquire) & bit)) {
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    g_smem_configured[variant].fetch_or(bit, std::memory_order_release);
  }
  const int64_t tiles_m = (p.M + BM - 1) / BM;
  const int64_t tiles_n = (p.N + BN - 1) / BN;
  if (tiles_m * tiles_n > 0x7fffffff) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(tiles_m * tiles_n), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, kernel, int(p.M), int(p.N), int(p.K), p.A, p.lda, p.B, p.ldb,
                            p.C, p.ldc, int(tiles_m), int(tiles_n));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

cudaError_t launch_simt(const GemmProblem &p, const DeviceInfo &dev, cudaStream_t stream) {
  const bool vec_b = aligned16(p.B) && p.ldb % 4 == 0 && p.N % 4 == 0;
  const bool vec_store = aligned16(p.C) && p.ldc % 4 == 0 && p.N % 4 == 0;
  if (vec_b)
    return vec_store ? launch_variant<true, true>(p, dev, stream)
                     : launch_variant<true, false>(p, dev, stream);
  return vec_store ? launch_variant<false, true>(p, dev, stream)
                   : launch_variant<false, false>(p, dev, stream);
}

}  // namespace tmm
