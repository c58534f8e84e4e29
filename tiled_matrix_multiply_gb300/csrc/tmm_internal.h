// tmm_internal.h -- declarations shared by the library's translation units.
// Not part of the public ABI (that is include/tmm_gemm.h).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace tmm {

// One validated product C = A x B (row-major, element strides lda/ldb/ldc).
struct GemmProblem {
  int64_t M, N, K;
  const float *A;
  int64_t lda;
  const float *B;
  int64_t ldb;
  float *C;
  int64_t ldc;
};

// Properties of the current device the launchers size their grids by.
struct DeviceInfo {
  int id;
  int sm_count;
  int cc_major, cc_minor;
  int max_smem_optin;  // bytes of shared memory a block may opt in to
};

// Each launcher enqueues its kernel(s) on `stream` and returns the launch
// status.  Problems reaching a launcher have M, N, K > 0.
cudaError_t launch_naive(const GemmProblem &p, const DeviceInfo &dev, cudaStream_t stream);
cudaError_t launch_simt(const GemmProblem &p, const DeviceInfo &dev, cudaStream_t stream);

}  // namespace tmm
