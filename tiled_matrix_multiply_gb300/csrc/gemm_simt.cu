// gemm_simt.cu -- two-level tiled FP32 product on the CUDA cores (FFMA).
//
// Tiling ("Tiling Strategies" sections 2-4, "CMU DLSys Lecture 12" section 5):
//   * block tile: each 256-thread block owns a BM x BN = 128 x 128 tile of C;
//   * K-slices of BK = 8: the block stages the BM x BK slab of A and the
//     BK x BN slab of B in shared memory, double buffered ("Tiling
//     Strategies" section 3): the global loads of slice t+1 are in flight
//     (held in registers) while slice t is consumed, and are written to the
//     other buffer just before it is needed, so one barrier per slice suffices;
//   * thread tile: each thread owns an 8 x 8 tile of C in 64 accumulators and
//     performs one outer product per k (8 + 8 operands, 64 FFMA), with the
//     operands of step k+1 loaded from shared memory while step k's FFMAs
//     issue ("Tiling Hierarchy on GPUs", "Register Tiling", "Register
//     prefetching").
//
// Shared-memory layout.  The A slab is stored transposed, a[k][m], so a
// thread's 8 rows of A at one k are two 16-byte vectors; the row length is
// padded to BM + 4 floats, which makes the transposing stores conflict-free
// (each warp writes 16 rows x 2 k-quads that land in 32 distinct banks).  The
// B slab keeps its global layout b[k][n].  A warp covers a 32 x 64 region of
// C with its lanes as 4 (rows) x 8 (columns), each lane's 8 x 8 tile split
// into 4 x 4 quadrants 16 rows / 32 columns apart: every fragment load of a
// warp then reads 4 (A) or 8 (B) distinct 16-byte vectors of one 128-byte
// line -- one shared-memory wavefront, the other lanes served by broadcast.
//
// Tails ("CMU DLSys Lecture 12" section 5, single-buffer schedule): loads
// outside M, N or K are replaced by zeros, which add nothing to the sums, and
// only entries inside M x N are stored.
//
// Scheduling: tiles are numbered along a grouped raster -- kGroupM tile-rows
// are walked column by column -- so blocks resident at the same time share
// the A row-panels and B column-panels they read through L2.
#include "tmm_internal.h"

namespace tmm {
namespace {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int BK = 8;
constexpr int TM = 8;
constexpr int TN = 8;
constexpr int kThreads = (BM / TM) * (BN / TN);  // 256
constexpr int kAsLd = BM + 4;                    // padded row of the transposed A slab
constexpr int kBsLd = BN;
constexpr int kGroupM = 16;

static_assert(kThreads == 256, "thread mapping below assumes 256 threads");
static_assert(BM * BK == kThreads * 4 && BN * BK == kThreads * 4,
              "each thread stages one 4-element vector of A and of B per slice");

struct __align__(16) SimtSmem {
  float a[2][BK][kAsLd];
  float b[2][BK][kBsLd];
};

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

// kVecLoad: A and B are 16-byte aligned, lda, ldb, K and N are multiples of 4,
//           so every staged 4-vector is either wholly inside or wholly outside.
// kVecStore: C is 16-byte aligned and ldc, N are multiples of 4.
template <bool kVecLoad, bool kVecStore>
__global__ void __launch_bounds__(kThreads, 2)
gemm_simt_kernel(int M, int N, int K,
                 const float *__restrict__ A, int64_t lda,
                 const float *__restrict__ B, int64_t ldb,
                 float *__restrict__ C, int64_t ldc, int tiles_m, int tiles_n) {
  __shared__ SimtSmem sm;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  int tm, tn;
  tile_coords(blockIdx.x, tiles_m, tiles_n, tm, tn);
  const int m0 = tm * BM;
  const int n0 = tn * BN;

  // Staging assignment: A vector = row a_row, k offset a_k (4 consecutive k);
  // B vector = k row b_k, columns b_n..b_n+3.
  const int a_row = tid >> 1;
  const int a_k = (tid & 1) * 4;
  const int b_k = tid >> 5;
  const int b_n = (tid & 31) * 4;
  const bool a_row_ok = m0 + a_row < M;
  const int b_col = n0 + b_n;
  const float *a_src = A + int64_t(a_row_ok ? m0 + a_row : 0) * lda + a_k;
  const float *b_src = B + int64_t(b_k) * ldb + (b_col < N ? b_col : 0);
  const int64_t b_step = int64_t(BK) * ldb;

  // Fragment assignment: warp (wm, wn) covers rows wm*32.., columns wn*64..;
  // lane (lm, ln) reads A at rows a_off, a_off+16 and B at columns b_off, b_off+32.
  const int wm = warp >> 1, wn = warp & 1;
  const int lm = lane >> 3, ln = lane & 7;
  const int a_off = wm * 32 + lm * 4;
  const int b_off = wn * 64 + ln * 4;

  float acc[TM][TN];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) acc[i][j] = 0.0f;

  float4 a_st, b_st;

  // Stage the slice starting at k0 into registers; a_src/b_src point at it.
  auto load_slice = [&](int k0) {
    if (kVecLoad) {
      const bool a_ok = a_row_ok && (k0 + a_k < K);
      const bool b_ok = (b_col < N) && (k0 + b_k < K);
      a_st = a_ok ? *reinterpret_cast<const float4 *>(a_src) : make_float4(0, 0, 0, 0);
      b_st = b_ok ? *reinterpret_cast<const float4 *>(b_src) : make_float4(0, 0, 0, 0);
    } else {
      float av[4], bv[4];
      const bool b_k_ok = k0 + b_k < K;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        av[j] = (a_row_ok && k0 + a_k + j < K) ? a_src[j] : 0.0f;
        bv[j] = (b_k_ok && b_col + j < N) ? b_src[j] : 0.0f;
      }
      a_st = make_float4(av[0], av[1], av[2], av[3]);
      b_st = make_float4(bv[0], bv[1], bv[2], bv[3]);
    }
  };
  auto store_slice = [&](int buf) {
    sm.a[buf][a_k + 0][a_row] = a_st.x;
    sm.a[buf][a_k + 1][a_row] = a_st.y;
    sm.a[buf][a_k + 2][a_row] = a_st.z;
    sm.a[buf][a_k + 3][a_row] = a_st.w;
    *reinterpret_cast<float4 *>(&sm.b[buf][b_k][b_n]) = b_st;
  };
  auto load_frag = [&](int buf, int k, float (&af)[TM], float (&bf)[TN]) {
    const float4 a0 = *reinterpret_cast<const float4 *>(&sm.a[buf][k][a_off]);
    const float4 a1 = *reinterpret_cast<const float4 *>(&sm.a[buf][k][a_off + 16]);
    const float4 b0 = *reinterpret_cast<const float4 *>(&sm.b[buf][k][b_off]);
    const float4 b1 = *reinterpret_cast<const float4 *>(&sm.b[buf][k][b_off + 32]);
    af[0] = a0.x; af[1] = a0.y; af[2] = a0.z; af[3] = a0.w;
    af[4] = a1.x; af[5] = a1.y; af[6] = a1.z; af[7] = a1.w;
    bf[0] = b0.x; bf[1] = b0.y; bf[2] = b0.z; bf[3] = b0.w;
    bf[4] = b1.x; bf[5] = b1.y; bf[6] = b1.z; bf[7] = b1.w;
  };

  load_slice(0);
  store_slice(0);
  __syncthreads();

  float af[TM], bf[TN];
  int cur = 0;
  for (int k0 = 0; k0 < K; k0 += BK) {
    const bool has_next = k0 + BK < K;
    if (has_next) {
      a_src += BK;
      b_src += b_step;
      load_slice(k0 + BK);
    }
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      load_frag(cur, k, af, bf);
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(af[i], bf[j], acc[i][j]);
    }
    if (has_next) {
      store_slice(cur ^ 1);
      __syncthreads();
    }
    cur ^= 1;
  }

  // Epilogue: row i of the thread tile is m0 + a_off + (i/4)*16 + i%4,
  // column j is n0 + b_off + (j/4)*32 + j%4.
  const int row0 = m0 + a_off;
  const int col0 = n0 + b_off;
  float *c_base = C + int64_t(row0) * ldc + col0;
#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int dr = (i >> 2) * 16 + (i & 3);
    if (row0 + dr >= M) continue;
    float *c_row = c_base + int64_t(dr) * ldc;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int dc = h * 32;
      if (kVecStore) {
        if (col0 + dc < N)
          *reinterpret_cast<float4 *>(c_row + dc) =
              make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2], acc[i][4 * h + 3]);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (col0 + dc + j < N) c_row[dc + j] = acc[i][4 * h + j];
      }
    }
  }
}

template <bool kVecLoad, bool kVecStore>
cudaError_t launch_variant(const GemmProblem &p, cudaStream_t stream) {
  const int64_t tiles_m = (p.M + BM - 1) / BM;
  const int64_t tiles_n = (p.N + BN - 1) / BN;
  if (tiles_m * tiles_n > 0x7fffffff) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(tiles_m * tiles_n), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, gemm_simt_kernel<kVecLoad, kVecStore>, int(p.M), int(p.N),
                            int(p.K), p.A, p.lda, p.B, p.ldb, p.C, p.ldc, int(tiles_m),
                            int(tiles_n));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

cudaError_t launch_simt(const GemmProblem &p, const DeviceInfo &, cudaStream_t stream) {
  const bool vec_load = aligned16(p.A) && aligned16(p.B) && p.lda % 4 == 0 &&
                        p.ldb % 4 == 0 && p.K % 4 == 0 && p.N % 4 == 0;
  const bool vec_store = aligned16(p.C) && p.ldc % 4 == 0 && p.N % 4 == 0;
  if (vec_load)
    return vec_store ? launch_variant<true, true>(p, stream)
                     : launch_variant<true, false>(p, stream);
  return vec_store ? launch_variant<false, true>(p, stream)
                   : launch_variant<false, false>(p, stream);
}

}  // namespace tmm
