// tensor_map.cpp -- TMA descriptors (CUtensorMap) for the library's kernels.
//
// The encoder is the driver's cuTensorMapEncodeTiled, looked up once through
// the runtime's driver entry-point query, so the library links against the
// CUDA runtime only.
#include <mutex>

#include <cudaTypedefs.h>

#include "tmm_internal.h"

namespace tmm {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_status = cudaSuccess;

}  // namespace

cudaError_t tensor_map_encoder_ready() {
  std::call_once(g_encode_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    g_encode_status = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                       cudaEnableDefault, &q);
    if (g_encode_status == cudaSuccess && (q != cudaDriverEntryPointSuccess || fn == nullptr))
      g_encode_status = cudaErrorNotSupported;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode_status;
}

cudaError_t encode_f32_2d(CUtensorMap *map, const float *base, int64_t rows, int64_t cols,
                          int64_t ld, uint32_t box_cols, uint32_t box_rows,
                          CUtensorMapSwizzle swizzle) {
  cudaError_t e = tensor_map_encoder_ready();
  if (e != cudaSuccess) return e;
  const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(ld) * 4};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base),
                              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace tmm
