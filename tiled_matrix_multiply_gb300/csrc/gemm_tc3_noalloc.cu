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
// The array's name is only a host-side stand-in in host code: it is turned
// into the device address with cudaGetSymbolAddress, once per device, with
// that device current, and that address is what the kernels receive.  All
// calls share the array and it keeps the last call's contents; nothing in it
// needs to start at zero (the split pre-pass writes every element the product
// kernel reads).  Calls that overlap on the GPU (for example on two streams)
// race on it.
#include <cstddef>
#include <mutex>

#include "tmm_internal.h"

namespace {

constexpr size_t kTc3NoallocScratchBytes = size_t(64) << 20;   // 64 MiB per device

}  // namespace

static __device__ __align__(256) unsigned char g_tc3_noalloc_scratch[kTc3NoallocScratchBytes];

namespace tmm {
namespace {

constexpr int kMaxScratchDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxScratchDevices] = {};

}  // namespace

size_t tc3_noalloc_scratch_bytes() { return kTc3NoallocScratchBytes; }

cudaError_t tc3_noalloc_scratch(int device, void **ptr) {
  if (device < 0 || device >= kMaxScratchDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[device] == nullptr) {
    // The caller has `device` current: the address is that device's copy.
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_tc3_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (p == nullptr) return cudaErrorInvalidSymbol;
    g_scratch_ptr[device] = p;
  }
  *ptr = g_scratch_ptr[device];
  return cudaSuccess;
}

}  // namespace tmm
