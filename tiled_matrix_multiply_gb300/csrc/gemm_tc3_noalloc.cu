// gemm_tc3_noalloc.cu -- fixed scratch for gemm_f32_tc3_noalloc.
//
// gemm_f32_tc3 needs a workspace for the split TF32 operands, which its
// caller allocates.  Some callers cannot allocate device memory at the point
// of the call: code running under a memory manager that owns the whole device
// budget and forbids raw cudaMalloc, code on a latency-critical path where
// cudaMalloc's implicit device synchronisation is not acceptable, or code in a
// context where the CUDA allocation API may not be called at all.  For them
// the workspace lives here, in one statically sized array of device memory
// that the CUDA runtime sets aside when this module is loaded; every GPU that
// loads it holds the array until the process exits.
//
// The array's name is only a host-side stand-in in host code: every call turns
// it into the device address with cudaGetSymbolAddress, with the caller's
// device current, and that address is what the kernels receive.  The lookup
// is not cached: an address kept per device ordinal would outlive the context
// it belongs to (after cudaDeviceReset, or with another context current on the
// same ordinal) and send the kernels to memory that is no longer the array.
// All calls share the array and it keeps the last call's contents; nothing in
// it needs to start at zero (the split pre-pass writes every element the
// product kernel reads).  Calls that overlap on the GPU (for example on two
// streams) race on it.
#include <cstddef>

#include "tmm_internal.h"

namespace {

constexpr size_t kTc3NoallocScratchBytes = size_t(64) << 20;   // 64 MiB per device

}  // namespace

static __device__ __align__(256) unsigned char g_tc3_noalloc_scratch[kTc3NoallocScratchBytes];

namespace tmm {

size_t tc3_noalloc_scratch_bytes() { return kTc3NoallocScratchBytes; }

cudaError_t tc3_noalloc_scratch(void **ptr) {
  // The current device's (and current context's) copy of the array.
  void *p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_tc3_noalloc_scratch);
  if (e != cudaSuccess) return e;
  if (p == nullptr) return cudaErrorInvalidSymbol;
  *ptr = p;
  return cudaSuccess;
}

}  // namespace tmm
