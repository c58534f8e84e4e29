// gemm_abi.cpp -- the extern "C" boundary: argument checks, device checks,
// path selection and launch-status reporting.  No device memory is allocated.
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "bounds_check.cuh"
#include "tmm_gemm.h"
#include "tmm_internal.h"

namespace {

thread_local char g_last_error[256] = "";

int fail(int code, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
bool g_dev_known[kMaxDevices] = {};
tmm::DeviceInfo g_dev_info[kMaxDevices];

// Properties of the current device, queried once per device.
int current_device(tmm::DeviceInfo *out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(TMM_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return fail(TMM_ERR_UNSUPPORTED_DEVICE, "device ordinal %d out of range", dev);
  {
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (g_dev_known[dev]) {
      *out = g_dev_info[dev];
      return TMM_OK;
    }
  }
  tmm::DeviceInfo info = {};
  info.id = dev;
  if ((e = cudaDeviceGetAttribute(&info.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) ||
      (e = cudaDeviceGetAttribute(&info.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) ||
      (e = cudaDeviceGetAttribute(&info.sm_count, cudaDevAttrMultiProcessorCount, dev)) ||
      (e = cudaDeviceGetAttribute(&info.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                  dev)))
    return fail(TMM_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
  if (info.cc_major != 10 || info.cc_minor != 3)
    return fail(TMM_ERR_UNSUPPORTED_DEVICE,
                "device %d has compute capability %d.%d; this library is built for 10.3 (sm_103a)",
                dev, info.cc_major, info.cc_minor);
  {
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    g_dev_info[dev] = info;
    g_dev_known[dev] = true;
  }
  *out = info;
  return TMM_OK;
}

// a * b + c without int64 overflow; false when it would overflow.
bool span_ok(int64_t rows, int64_t ld, int64_t cols) {
  if (rows <= 0 || cols <= 0) return true;
  const __int128 last = (__int128)(rows - 1) * ld + cols;
  return last <= (__int128)(INT64_MAX / 4);
}

// Byte range [lo, hi) spanned by the rows x cols window of a row-major matrix.
void byte_span(const void *p, int64_t rows, int64_t ld, int64_t cols, uintptr_t *lo,
               uintptr_t *hi) {
  *lo = reinterpret_cast<uintptr_t>(p);
  *hi = *lo + uintptr_t(((rows - 1) * ld + cols) * int64_t(sizeof(float)));
}

bool overlaps(uintptr_t a_lo, uintptr_t a_hi, uintptr_t b_lo, uintptr_t b_hi) {
  return a_lo < b_hi && b_lo < a_hi;
}

// Checks shared by every entry point; on success *nothing_to_do tells whether
// the call is a no-op (M == 0 or N == 0).  transa/transb select how A and B
// are stored: A as M x K (0) or K x M (1), B as K x N (0) or N x K (1).
int check_args(const char *who, int64_t M, int64_t N, int64_t K, int transa, int transb,
               const float *A, int64_t lda, const float *B, int64_t ldb, const float *C,
               int64_t ldc, bool *nothing_to_do) {
  *nothing_to_do = false;
  if ((transa != 0 && transa != 1) || (transb != 0 && transb != 1))
    return fail(TMM_ERR_INVALID_ARG, "%s: transa and transb must be 0 or 1", who);
  if (M < 0 || N < 0 || K < 0)
    return fail(TMM_ERR_INVALID_ARG, "%s: negative size (M=%lld N=%lld K=%lld)", who,
                (long long)M, (long long)N, (long long)K);
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX)
    return fail(TMM_ERR_INVALID_ARG, "%s: sizes above 2^31-1 are not supported", who);
  const int64_t a_rows = transa ? K : M, a_cols = transa ? M : K;
  const int64_t b_rows = transb ? N : K, b_cols = transb ? K : N;
  const int64_t min_lda = a_cols > 1 ? a_cols : 1, min_ldb = b_cols > 1 ? b_cols : 1;
  const int64_t min_ldc = N > 1 ? N : 1;
  if (lda < min_lda || ldb < min_ldb || ldc < min_ldc)
    return fail(TMM_ERR_INVALID_ARG,
                "%s: leading dimension too small (lda=%lld ldb=%lld ldc=%lld for stored A %lldx%lld, "
                "B %lldx%lld, C %lldx%lld)",
                who, (long long)lda, (long long)ldb, (long long)ldc, (long long)a_rows,
                (long long)a_cols, (long long)b_rows, (long long)b_cols, (long long)M,
                (long long)N);
  if (M == 0 || N == 0) {
    *nothing_to_do = true;
    return TMM_OK;
  }
  if (C == nullptr) return fail(TMM_ERR_INVALID_ARG, "%s: C is NULL", who);
  if (K > 0 && (A == nullptr || B == nullptr))
    return fail(TMM_ERR_INVALID_ARG, "%s: A or B is NULL", who);
  if (!span_ok(a_rows, lda, a_cols) || !span_ok(b_rows, ldb, b_cols) || !span_ok(M, ldc, N))
    return fail(TMM_ERR_INVALID_ARG, "%s: matrix extent overflows 64-bit byte offsets", who);
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) |
       reinterpret_cast<uintptr_t>(C)) & 3u)
    return fail(TMM_ERR_INVALID_ARG, "%s: pointers must be 4-byte aligned", who);
  if (K > 0) {
    uintptr_t c_lo, c_hi, a_lo, a_hi, b_lo, b_hi;
    byte_span(C, M, ldc, N, &c_lo, &c_hi);
    byte_span(A, a_rows, lda, a_cols, &a_lo, &a_hi);
    byte_span(B, b_rows, ldb, b_cols, &b_lo, &b_hi);
    if (overlaps(c_lo, c_hi, a_lo, a_hi) || overlaps(c_lo, c_hi, b_lo, b_hi))
      return fail(TMM_ERR_ALIAS, "%s: the byte range of C overlaps A or B", who);
  }
  return TMM_OK;
}

using Launcher = cudaError_t (*)(const tmm::GemmProblem &, const tmm::DeviceInfo &, cudaStream_t);

int run(const char *who, Launcher launch, int transa, int transb, int64_t M, int64_t N,
        int64_t K, const float *A, int64_t lda, const float *B, int64_t ldb, float *C,
        int64_t ldc, tmm_stream_t stream) {
  bool noop = false;
  int rc = check_args(who, M, N, K, transa, transb, A, lda, B, ldb, C, ldc, &noop);
  if (rc != TMM_OK || noop) return rc;
  tmm::DeviceInfo dev;
  if ((rc = current_device(&dev)) != TMM_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (K == 0) {
    // The empty sum: zero the M x N window of C, leaving the row gaps alone.
    e = cudaMemset2DAsync(C, size_t(ldc) * sizeof(float), 0, size_t(N) * sizeof(float),
                          size_t(M), s);
    if (e != cudaSuccess)
      return fail(TMM_ERR_CUDA, "%s: cudaMemset2DAsync: %s", who, cudaGetErrorString(e));
    return TMM_OK;
  }
  tmm::GemmProblem p = {M, N, K, A, lda, B, ldb, C, ldc};
  p.transa = transa;
  p.transb = transb;
  e = launch(p, dev, s);
  if (e != cudaSuccess) return fail(TMM_ERR_CUDA, "%s: launch: %s", who, cudaGetErrorString(e));
  return TMM_OK;
}

}  // namespace

extern "C" {

int gemm_f32(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B,
             int64_t ldb, float *C, int64_t ldc, tmm_stream_t stream) {
  return run("gemm_f32", tmm::launch_simt, 0, 0, M, N, K, A, lda, B, ldb, C, ldc, stream);
}

int gemm_f32_ex(int transa, int transb, int64_t M, int64_t N, int64_t K, const float *A,
                int64_t lda, const float *B, int64_t ldb, float *C, int64_t ldc,
                tmm_stream_t stream) {
  return run("gemm_f32_ex", tmm::launch_simt, transa, transb, M, N, K, A, lda, B, ldb, C, ldc,
             stream);
}

int gemm_f32_naive(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B,
                   int64_t ldb, float *C, int64_t ldc, tmm_stream_t stream) {
  return run("gemm_f32_naive", tmm::launch_naive, 0, 0, M, N, K, A, lda, B, ldb, C, ldc,
             stream);
}

int tmm_check_device(tmm_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return fail(TMM_ERR_CUDA, "tmm_check_device: cudaStreamSynchronize: %s", cudaGetErrorString(e));
  unsigned int simt = 0, tc3 = 0, win = 0, sm = 0, naive = 0, stage = 0;
  e = tmm::simt_device_status(&simt, true);
  if (e == cudaSuccess) e = tmm::tc3_device_status(&tc3, true);
  if (e == cudaSuccess) e = tmm::window_device_status(&win, true);
  if (e == cudaSuccess) e = tmm::softmax_device_status(&sm, true);
  if (e == cudaSuccess) e = tmm::naive_device_status(&naive, true);
  if (e == cudaSuccess) e = tmm::stage_device_status(&stage, true);
  if (e != cudaSuccess)
    return fail(TMM_ERR_CUDA, "tmm_check_device: status read: %s", cudaGetErrorString(e));
  if ((simt | tc3 | naive | stage) & tmm::kStatusBounds)
    return fail(TMM_ERR_BOUNDS,
                "tmm_check_device: a range check of the bounds-checked build failed inside %s",
                (simt & tmm::kStatusBounds)    ? "gemm_f32"
                : (stage & tmm::kStatusBounds) ? "gemm_f32 (operand restaging)"
                : (tc3 & tmm::kStatusBounds)   ? "gemm_f32_tc3"
                                               : "gemm_f32_naive");
  if (simt | tc3 | win | sm)
    return fail(TMM_ERR_DEVICE_TIMEOUT,
                "tmm_check_device: a bounded wait inside %s ran out of time; the affected "
                "results are not valid",
                simt ? "gemm_f32"
                     : (tc3 ? "gemm_f32_tc3" : (win ? "window_sum_f32" : "softmax_rows_f32")));
  return TMM_OK;
}

int tmm_testing_simt_plan(int64_t M, int64_t N, int64_t K, int wide, int vec_c, int may_reduce,
                          int64_t slots, int64_t *out) {
  if (M <= 0 || N <= 0 || K <= 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX ||
      slots <= 0 || out == nullptr)
    return fail(TMM_ERR_INVALID_ARG, "tmm_testing_simt_plan: bad arguments");
  tmm::simt_plan_for_testing(M, N, K, wide, vec_c, may_reduce, slots, out);
  return TMM_OK;
}

int tmm_testing_tc3_plan(int64_t M, int64_t N, int64_t K, int pairs, int64_t slots,
                         int64_t *out) {
  if (M <= 0 || N <= 0 || K <= 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX ||
      slots <= 0 || out == nullptr)
    return fail(TMM_ERR_INVALID_ARG, "tmm_testing_tc3_plan: bad arguments");
  tmm::tc3_plan_for_testing(M, N, K, pairs, slots, out);
  return TMM_OK;
}

int tmm_testing_set_wait_hooks(int drop_signal_block, int64_t wait_limit_ns) {
  tmm::simt_set_test_hooks(drop_signal_block, wait_limit_ns);
  tmm::tc3_set_test_hooks(drop_signal_block, wait_limit_ns);
  tmm::window_set_test_hooks(drop_signal_block, wait_limit_ns);
  tmm::softmax_set_test_hooks(drop_signal_block, wait_limit_ns);
  return TMM_OK;
}

size_t gemm_f32_tc3_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return 0;
  return tmm::tc3_workspace_bytes(M, N, K);
}

int gemm_f32_tc3_ex(int transa, int transb, int64_t M, int64_t N, int64_t K, const float *A,
                    int64_t lda, const float *B, int64_t ldb, float *C, int64_t ldc,
                    void *workspace, size_t workspace_bytes, tmm_stream_t stream) {
  const char *who = "gemm_f32_tc3";
  bool noop = false;
  int rc = check_args(who, M, N, K, transa, transb, A, lda, B, ldb, C, ldc, &noop);
  if (rc != TMM_OK || noop) return rc;
  tmm::DeviceInfo dev;
  if ((rc = current_device(&dev)) != TMM_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (K == 0) {
    cudaError_t e = cudaMemset2DAsync(C, size_t(ldc) * sizeof(float), 0,
                                      size_t(N) * sizeof(float), size_t(M), s);
    if (e != cudaSuccess)
      return fail(TMM_ERR_CUDA, "%s: cudaMemset2DAsync: %s", who, cudaGetErrorString(e));
    return TMM_OK;
  }
  const size_t need = tmm::tc3_workspace_bytes(M, N, K);
  if (need == SIZE_MAX)
    return fail(TMM_ERR_INVALID_ARG, "%s: the workspace size of this product overflows size_t",
                who);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(TMM_ERR_INVALID_ARG, "%s: workspace of %zu bytes needed, %zu given", who, need,
                workspace == nullptr ? size_t(0) : workspace_bytes);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return fail(TMM_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned", who);
  {
    uintptr_t c_lo, c_hi, a_lo, a_hi, b_lo, b_hi;
    byte_span(C, M, ldc, N, &c_lo, &c_hi);
    byte_span(A, transa ? K : M, lda, transa ? M : K, &a_lo, &a_hi);
    byte_span(B, transb ? N : K, ldb, transb ? K : N, &b_lo, &b_hi);
    const uintptr_t w_lo = reinterpret_cast<uintptr_t>(workspace), w_hi = w_lo + need;
    if (overlaps(w_lo, w_hi, c_lo, c_hi) || overlaps(w_lo, w_hi, a_lo, a_hi) ||
        overlaps(w_lo, w_hi, b_lo, b_hi))
      return fail(TMM_ERR_ALIAS, "%s: the workspace overlaps A, B or C", who);
  }
  tmm::GemmProblem p = {M, N, K, A, lda, B, ldb, C, ldc};
  p.transa = transa;
  p.transb = transb;
  cudaError_t e = tmm::launch_tc3(p, dev, workspace, s);
  if (e != cudaSuccess) return fail(TMM_ERR_CUDA, "%s: launch: %s", who, cudaGetErrorString(e));
  return TMM_OK;
}

int gemm_f32_tc3(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B,
                 int64_t ldb, float *C, int64_t ldc, void *workspace, size_t workspace_bytes,
                 tmm_stream_t stream) {
  return gemm_f32_tc3_ex(0, 0, M, N, K, A, lda, B, ldb, C, ldc, workspace, workspace_bytes,
                         stream);
}

int gemm_f32_tc3_noalloc(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                         const float *B, int64_t ldb, float *C, int64_t ldc,
                         tmm_stream_t stream) {
  const char *who = "gemm_f32_tc3_noalloc";
  bool noop = false;
  int rc = check_args(who, M, N, K, 0, 0, A, lda, B, ldb, C, ldc, &noop);
  if (rc != TMM_OK || noop) return rc;
  // The size limit is checked before any CUDA call, so a refused product
  // reaches neither the device nor the scratch.
  const size_t need = K > 0 ? tmm::tc3_workspace_bytes(M, N, K) : 0;
  const size_t limit = tmm::tc3_noalloc_scratch_bytes();
  if (need > limit)
    return fail(TMM_ERR_INVALID_ARG,
                "%s: this product needs %zu bytes of scratch but the fixed scratch holds %zu; "
                "use gemm_f32_tc3 with a caller-supplied workspace",
                who, need, limit);
  tmm::DeviceInfo dev;
  if ((rc = current_device(&dev)) != TMM_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (K == 0) {
    cudaError_t e = cudaMemset2DAsync(C, size_t(ldc) * sizeof(float), 0,
                                      size_t(N) * sizeof(float), size_t(M), s);
    if (e != cudaSuccess)
      return fail(TMM_ERR_CUDA, "%s: cudaMemset2DAsync: %s", who, cudaGetErrorString(e));
    return TMM_OK;
  }
  void *scratch = nullptr;
  cudaError_t e = tmm::tc3_noalloc_scratch(&scratch);
  if (e != cudaSuccess)
    return fail(TMM_ERR_CUDA, "%s: scratch address lookup: %s", who, cudaGetErrorString(e));
  const tmm::GemmProblem p = {M, N, K, A, lda, B, ldb, C, ldc};
  e = tmm::launch_tc3(p, dev, scratch, s);
  if (e != cudaSuccess) return fail(TMM_ERR_CUDA, "%s: launch: %s", who, cudaGetErrorString(e));
  return TMM_OK;
}

int window_sum_f32(int64_t n, int W, const float *x, float *y, tmm_stream_t stream) {
  const char *who = "window_sum_f32";
  if (n < 0 || W < 1 || W > tmm::kMaxWindow)
    return fail(TMM_ERR_INVALID_ARG, "%s: need n >= 0 and 1 <= W <= %d (n=%lld W=%d)", who,
                tmm::kMaxWindow, (long long)n, W);
  if (n == 0) return TMM_OK;
  if (n > (int64_t(1) << 40))
    return fail(TMM_ERR_INVALID_ARG, "%s: n above 2^40 is not supported", who);
  if (x == nullptr || y == nullptr) return fail(TMM_ERR_INVALID_ARG, "%s: x or y is NULL", who);
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 3u)
    return fail(TMM_ERR_INVALID_ARG, "%s: pointers must be 4-byte aligned", who);
  const uintptr_t x_lo = reinterpret_cast<uintptr_t>(x), x_hi = x_lo + uintptr_t(n + W - 1) * 4;
  const uintptr_t y_lo = reinterpret_cast<uintptr_t>(y), y_hi = y_lo + uintptr_t(n) * 4;
  if (overlaps(x_lo, x_hi, y_lo, y_hi))
    return fail(TMM_ERR_ALIAS, "%s: the output overlaps the input", who);
  tmm::DeviceInfo dev;
  int rc = current_device(&dev);
  if (rc != TMM_OK) return rc;
  cudaError_t e = tmm::launch_window_sum(n, W, x, y, dev, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(TMM_ERR_CUDA, "%s: launch: %s", who, cudaGetErrorString(e));
  return TMM_OK;
}

size_t sum_f32_workspace_size(int64_t n) {
  (void)n;
  return size_t(tmm::kSumMaxPartials) * sizeof(float);
}

int sum_f32(int64_t n, const float *x, float *out, void *workspace, size_t workspace_bytes,
            tmm_stream_t stream) {
  const char *who = "sum_f32";
  if (n < 0 || n > (int64_t(1) << 40))
    return fail(TMM_ERR_INVALID_ARG, "%s: need 0 <= n <= 2^40 (n=%lld)", who, (long long)n);
  if (out == nullptr) return fail(TMM_ERR_INVALID_ARG, "%s: out is NULL", who);
  if (reinterpret_cast<uintptr_t>(out) & 3u)
    return fail(TMM_ERR_INVALID_ARG, "%s: out must be 4-byte aligned", who);
  const size_t need = sum_f32_workspace_size(n);
  if (n > 0) {
    if (x == nullptr) return fail(TMM_ERR_INVALID_ARG, "%s: x is NULL", who);
    if (reinterpret_cast<uintptr_t>(x) & 3u)
      return fail(TMM_ERR_INVALID_ARG, "%s: x must be 4-byte aligned", who);
    if (workspace == nullptr || workspace_bytes < need)
      return fail(TMM_ERR_INVALID_ARG, "%s: workspace of %zu bytes needed, %zu given", who, need,
                  workspace == nullptr ? size_t(0) : workspace_bytes);
    if (reinterpret_cast<uintptr_t>(workspace) & 15u)
      return fail(TMM_ERR_INVALID_ARG, "%s: workspace must be 16-byte aligned", who);
    const uintptr_t x_lo = reinterpret_cast<uintptr_t>(x), x_hi = x_lo + uintptr_t(n) * 4;
    const uintptr_t w_lo = reinterpret_cast<uintptr_t>(workspace), w_hi = w_lo + need;
    if (overlaps(x_lo, x_hi, w_lo, w_hi))
      return fail(TMM_ERR_ALIAS, "%s: the workspace overlaps x", who);
  }
  tmm::DeviceInfo dev;
  int rc = current_device(&dev);
  if (rc != TMM_OK) return rc;
  cudaError_t e = tmm::launch_sum(n, x, out, static_cast<float *>(workspace), dev,
                                  reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(TMM_ERR_CUDA, "%s: launch: %s", who, cudaGetErrorString(e));
  return TMM_OK;
}

int softmax_rows_f32(int64_t rows, int64_t cols, const float *x, int64_t ldx, float *y,
                     int64_t ldy, tmm_stream_t stream) {
  const char *who = "softmax_rows_f32";
  if (rows < 0 || cols < 0)
    return fail(TMM_ERR_INVALID_ARG, "%s: negative size (rows=%lld cols=%lld)", who,
                (long long)rows, (long long)cols);
  if (cols > INT32_MAX)
    return fail(TMM_ERR_INVALID_ARG, "%s: cols above 2^31-1 is not supported", who);
  const int64_t min_ld = cols > 1 ? cols : 1;
  if (ldx < min_ld || ldy < min_ld)
    return fail(TMM_ERR_INVALID_ARG, "%s: row stride too small (ldx=%lld ldy=%lld, cols=%lld)",
                who, (long long)ldx, (long long)ldy, (long long)cols);
  if (rows == 0 || cols == 0) return TMM_OK;
  if (x == nullptr || y == nullptr) return fail(TMM_ERR_INVALID_ARG, "%s: x or y is NULL", who);
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 3u)
    return fail(TMM_ERR_INVALID_ARG, "%s: pointers must be 4-byte aligned", who);
  if (!span_ok(rows, ldx, cols) || !span_ok(rows, ldy, cols))
    return fail(TMM_ERR_INVALID_ARG, "%s: matrix extent overflows 64-bit byte offsets", who);
  const bool in_place = x == y && ldx == ldy;
  if (!in_place) {
    uintptr_t x_lo, x_hi, y_lo, y_hi;
    byte_span(x, rows, ldx, cols, &x_lo, &x_hi);
    byte_span(y, rows, ldy, cols, &y_lo, &y_hi);
    if (overlaps(x_lo, x_hi, y_lo, y_hi))
      return fail(TMM_ERR_ALIAS, "%s: y overlaps x without being x itself", who);
  }
  tmm::DeviceInfo dev;
  int rc = current_device(&dev);
  if (rc != TMM_OK) return rc;
  cudaError_t e = tmm::launch_softmax_rows(rows, int(cols), x, ldx, y, ldy, dev,
                                           reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(TMM_ERR_CUDA, "%s: launch: %s", who, cudaGetErrorString(e));
  return TMM_OK;
}

const char *tmm_last_error_string(void) { return g_last_error; }

const char *gemm_last_error_string(void) { return g_last_error; }

int gemm_check_status(tmm_stream_t stream) { return tmm_check_device(stream); }

int tmm_version(void) { return 100; }

}  // extern "C"
