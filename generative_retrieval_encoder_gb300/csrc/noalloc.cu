// bla_core_forward_noalloc: the gated BLA core forward for callers that
// cannot allocate device memory.  Its scratch (the split-L partial states,
// the combine counters, the error word, the combined state) lives in one
// file-scope device array that every GPU which loads this library holds
// until the process exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>
#include <unordered_map>

#include "../../include/gbla.h"

namespace {

constexpr size_t kScratchBytes = GBLA_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// The unique id of the calling thread's current CUDA context (0 if it cannot
// be read).  A context that is destroyed and re-created (cudaDeviceReset) gets
// a new id, and with it a new copy of g_scratch at a possibly new address.
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

std::mutex g_mu;
struct Entry { unsigned long long ctx; void* ptr; };
std::unordered_map<int, Entry> g_scratch_ptr;  // by device

// Device address of g_scratch on the current device.  The host-side name
// g_scratch is only a stand-in; the address comes from cudaGetSymbolAddress,
// looked up with that device current the first time the device is used, and
// again whenever the device's context has been re-created since.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  // 0 before the runtime has made the device's context current on this
  // thread: the lookup below does that, and the id is read again after it.
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = g_scratch_ptr.find(dev);
  if (it == g_scratch_ptr.end() || ctx == 0 || it->second.ctx != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = Entry{current_context_id(), p};
    *out = p;
    return cudaSuccess;
  }
  *out = it->second.ptr;
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
  if (scratch_address(&ws) != cudaSuccess) {
    (void)cudaGetLastError();
    return GBLA_ERR_CUDA;
  }
  // bla_core_forward clears the counters and the error word at the start of
  // every call, so the previous call's contents do not matter.
  return bla_core_forward(shape, q, k, v, g, o, den, state, ws, kScratchBytes, stream);
}

extern "C" gbla_status bla_core_noalloc_check_device_status(void* stream) {
  void* ws = nullptr;
  if (scratch_address(&ws) != cudaSuccess) {
    (void)cudaGetLastError();
    return GBLA_ERR_CUDA;
  }
  // The error word sits at the start of the scratch, as in any workspace.
  return gbla_check_device_status(ws, stream);
}
