// gemm_naive.cu -- one output per thread, operands straight from global memory.
//
// "Tiling Strategies" section 2 ("The Problem"): C[i][j] accumulates
// A[i][k] * B[k][j] over ascending k, every operand fetched from global
// memory, so the kernel issues 2 M N K operand loads for M N K FMAs
// (intensity 0.5 FMA per load, "Tiling Hierarchy on GPUs", "Inner Product").
// The launch is the bounds-checked one-thread-per-output pattern of "CMU DLSys
// Lecture 12" section 1, in two dimensions: 16 x 16 threads per block,
// ceil(N/16) x ceil(M/16) blocks, extra threads in the last blocks do nothing.
//
// It is the contrast kernel: its L1/L2 load traffic, not the FMA pipe, bounds it.
#include "bounds_check.cuh"
#include "tmm_internal.h"

namespace tmm {

// Status word of the naive kernel: bit 2 (kStatusBounds) when a range check of
// the bounds-checked build failed.
__device__ unsigned int g_naive_status;

namespace {

constexpr int kNaiveTile = 16;
constexpr int64_t kMaxGridY = 65535;

__global__ void __launch_bounds__(kNaiveTile * kNaiveTile)
gemm_naive_kernel(int64_t M, int64_t N, int64_t K,
                  const float *__restrict__ A, int64_t lda,
                  const float *__restrict__ B, int64_t ldb,
                  float *__restrict__ C, int64_t ldc) {
  const int64_t j = int64_t(blockIdx.x) * kNaiveTile + threadIdx.x;
  // Rows beyond 65535 blocks are covered by striding over the grid's y extent.
  for (int64_t i = int64_t(blockIdx.y) * kNaiveTile + threadIdx.y; i < M;
       i += int64_t(gridDim.y) * kNaiveTile) {
    if (j >= N) continue;
    const float *a = A + i * lda;
    const float *b = B + j;
    float acc = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
      if (TMM_IN_BOUNDS(in_matrix(a + k, A, M, K, lda) && in_matrix(b + k * ldb, B, K, N, ldb),
                        &g_naive_status))
        acc = fmaf(a[k], b[k * ldb], acc);
    }
    if (TMM_IN_BOUNDS(in_matrix(C + i * ldc + j, C, M, N, ldc), &g_naive_status))
      C[i * ldc + j] = acc;
  }
}

}  // namespace

cudaError_t naive_device_status(unsigned int *status, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(status, g_naive_status, sizeof(unsigned int));
  if (e != cudaSuccess || !clear) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_naive_status, &zero, sizeof(unsigned int));
}

cudaError_t launch_naive(const GemmProblem &p, const DeviceInfo &, cudaStream_t stream) {
  const int64_t gx = (p.N + kNaiveTile - 1) / kNaiveTile;
  int64_t gy = (p.M + kNaiveTile - 1) / kNaiveTile;
  if (gy > kMaxGridY) gy = kMaxGridY;
  if (gx > 0x7fffffff) return cudaErrorInvalidConfiguration;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(gx), unsigned(gy), 1);
  cfg.blockDim = dim3(kNaiveTile, kNaiveTile, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, gemm_naive_kernel, p.M, p.N, p.K, p.A, p.lda, p.B,
                            p.ldb, p.C, p.ldc);
}

}  // namespace tmm
