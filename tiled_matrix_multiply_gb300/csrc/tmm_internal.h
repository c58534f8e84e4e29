// tmm_internal.h -- declarations shared by the library's translation units.
// Not part of the public ABI (that is include/tmm_gemm.h).
#pragma once

#include <algorithm>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace tmm {

// One validated product C = op(A) x op(B) (row-major, element strides
// lda/ldb/ldc).  op(A) is M x K: A itself (stored M x K) or, with transa, the
// transpose of A stored K x M; op(B) is K x N likewise (B stored N x K with transb).
struct GemmProblem {
  int64_t M, N, K;
  const float *A;
  int64_t lda;
  const float *B;
  int64_t ldb;
  float *C;
  int64_t ldc;
  int transa = 0, transb = 0;
};

// Properties of the current device the launchers size their grids by.
struct DeviceInfo {
  int id;
  int sm_count;
  int cc_major, cc_minor;
  int max_smem_optin;  // bytes of shared memory a block may opt in to
};

// A 2-D FP32 tensor map (TMA descriptor): `rows` rows of `cols` floats, `ld`
// floats apart, copied in boxes of box_cols x box_rows; reads outside the
// matrix return zeros.  The base must be 16-byte aligned and ld a multiple of
// 4 (the tensor-map rules); cudaErrorInvalidValue otherwise.
cudaError_t tensor_map_encoder_ready();
cudaError_t encode_f32_2d(CUtensorMap *map, const float *base, int64_t rows, int64_t cols,
                          int64_t ld, uint32_t box_cols, uint32_t box_rows,
                          CUtensorMapSwizzle swizzle);

// Each launcher enqueues its kernel(s) on `stream` and returns the launch
// status.  Problems reaching a launcher have M, N, K > 0.
cudaError_t launch_naive(const GemmProblem &p, const DeviceInfo &dev, cudaStream_t stream);
// Status word of the naive kernel (bit 2: a range check of the bounds-checked
// build failed), read from the current device, optionally cleared.
cudaError_t naive_device_status(unsigned int *status, bool clear);
cudaError_t launch_simt(const GemmProblem &p, const DeviceInfo &dev, cudaStream_t stream);

// Operand restaging for the tiled product's TMA copies (operand_stage.cu):
// dst[r][c] = src[r][c] (stage_rows) or dst[c][r] = src[r][c]
// (stage_transpose) for r < rows, c < cols, with any source pitch and a
// destination pitch ld_dst; launched on `stream`.
cudaError_t stage_rows(const float *src, int64_t ld_src, int64_t rows, int64_t cols, float *dst,
                       int64_t ld_dst, const DeviceInfo &dev, cudaStream_t stream);
cudaError_t stage_transpose(const float *src, int64_t ld_src, int64_t rows, int64_t cols,
                            float *dst, int64_t ld_dst, const DeviceInfo &dev,
                            cudaStream_t stream);
// Stream-ordered scratch from the library's memory pool of the device (kept
// for reuse after it is freed); a failed allocation leaves no pending CUDA
// error behind.
cudaError_t scratch_alloc(void **ptr, size_t bytes, const DeviceInfo &dev, cudaStream_t stream);
cudaError_t scratch_free(void *ptr, cudaStream_t stream);
// Status word of the restaging copies (bit 2: a range check of the
// bounds-checked build failed), optionally cleared.
cudaError_t stage_device_status(unsigned int *status, bool clear);

// Split-TF32 tensor-core path: workspace bytes for an M x N x K product
// (SIZE_MAX when the count does not fit in size_t), and the launch (split
// pre-pass + product kernel); `workspace` is 256-byte aligned.
size_t tc3_workspace_bytes(int64_t M, int64_t N, int64_t K);
cudaError_t launch_tc3(const GemmProblem &p, const DeviceInfo &dev, void *workspace,
                       cudaStream_t stream);
cudaError_t tc3_device_status(unsigned int *status, bool clear);
// Fixed scratch of gemm_f32_tc3_noalloc: its size, and its address on the
// current device (looked up on every call).
size_t tc3_noalloc_scratch_bytes();
cudaError_t tc3_noalloc_scratch(void **ptr);
void tc3_set_test_hooks(int drop_signal_block, int64_t wait_limit_ns);
// The tensor-core kernels' work list, for host tests (see tmm_testing_tc3_plan).
void tc3_plan_for_testing(int64_t M, int64_t N, int64_t K, int pairs, int64_t slots,
                          int64_t out[6]);

// Sliding-window sums (y_i = sum_{d<W} x_{i+d}, i < n); 1 <= W <= kMaxWindow.
constexpr int kMaxWindow = 129;
cudaError_t window_device_status(unsigned int *status, bool clear);
void window_set_test_hooks(int drop_block, int64_t wait_limit_ns);
cudaError_t softmax_device_status(unsigned int *status, bool clear);
void softmax_set_test_hooks(int drop_block, int64_t wait_limit_ns);
cudaError_t launch_window_sum(int64_t n, int W, const float *x, float *y,
                              const DeviceInfo &dev, cudaStream_t stream);

// Device status word of the tiled kernel (bit 0: a bounded wait ran out of
// time); read from the current device, optionally cleared.
cudaError_t simt_device_status(unsigned int *status, bool clear);
// Testing hooks of the tiled kernel's stream-K waits (see tmm_gemm.h).
void simt_set_test_hooks(int drop_signal_block, int64_t wait_limit_ns);
// The tiled kernels' work split, for host tests (see tmm_testing_simt_plan).
void simt_plan_for_testing(int64_t M, int64_t N, int64_t K, int wide, int vec_c, int may_reduce,
                           int64_t slots, int64_t out[9]);

// Array sum: a first launch writes one partial per chunk of the input (at most
// kSumMaxPartials, in a caller-supplied workspace), a second adds them.
constexpr int kSumMaxPartials = 16384;
cudaError_t launch_sum(int64_t n, const float *x, float *out, float *partials,
                       const DeviceInfo &dev, cudaStream_t stream);

// Row softmax; rows of up to kMaxStagedRowBytes are staged in shared memory.
constexpr int kMaxStagedRowBytes = 49152 * 4;
cudaError_t launch_softmax_rows(int64_t rows, int cols, const float *x, int64_t ldx, float *y,
                                int64_t ldy, const DeviceInfo &dev, cudaStream_t stream);

}  // namespace tmm
