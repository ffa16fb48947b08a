// bla_core_forward_noalloc: the gated BLA core forward for callers that
// cannot allocate device memory.  Its scratch (the split-L partial states,
// the combine counters, the error word, the combined state) lives in one
// file-scope device array that every GPU which loads this library holds
// until the process exits.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "../../include/gbla.h"

namespace {

constexpr size_t kScratchBytes = GBLA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device.  The host-side name
// g_scratch is only a stand-in; the address comes from cudaGetSymbolAddress,
// looked up once per device with that device current.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" gbla_status bla_core_forward_noalloc(const gbla_shape* shape, const void* q, const void* k,
                                                const void* v, const float* g, void* o, float* den,
                                                float* state, void* stream) {
  const gbla_status s = gbla_validate_shape(shape);
  if (s != GBLA_OK) return s;
  const size_t need = gbla_workspace_size(shape, GBLA_OP_CORE_FORWARD);
  if (need == 0 || need > kScratchBytes) return GBLA_ERR_WORKSPACE;  // the fixed scratch is too small
  void* ws = nullptr;
  if (scratch_address(&ws) != cudaSuccess) return GBLA_ERR_CUDA;
  // bla_core_forward clears the counters and the error word at the start of
  // every call, so the previous call's contents do not matter.
  return bla_core_forward(shape, q, k, v, g, o, den, state, ws, kScratchBytes, stream);
}
