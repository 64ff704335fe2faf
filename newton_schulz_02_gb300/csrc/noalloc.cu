// Allocation-free Newton–Schulz entry point.
//
// Some callers cannot hand this library a workspace from cudaMalloc: code
// embedded in a framework whose caching allocator owns all device memory (a
// raw cudaMalloc there fragments memory and escapes the framework's
// accounting), and latency-critical loops that must not pay the implicit
// device synchronisation cudaMalloc / cudaFree can cause.  For them,
// newton_schulz_batched_noalloc runs the same kernels as
// newton_schulz_batched on a scratch area that is a file-scope __device__
// array of this library instead of a caller workspace.
//
// The array is part of the library's device image: every GPU the library is
// loaded on holds its kStaticScratchBytes until the process exits.  Host code
// cannot use the array's name as a device address; its device address is
// looked up with cudaGetSymbolAddress (with the device current) on the first
// call made in a CUDA context, and kept for later calls in that context.
// The cache is keyed by the context's process-unique id (cuCtxGetId), so an
// address taken in one context is never handed to kernels of another, not
// even of a context created after cudaDeviceReset under a reused handle.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/muon.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t{32} << 20;  // 32 MiB
constexpr int kMaxDevices = 128;

__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

struct ScratchAddr {
  unsigned long long ctx_id = 0;  // context the address was taken in
  void* ptr = nullptr;
};

std::mutex g_scratch_mu;
ScratchAddr g_scratch_addr[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Driver entry points, through the runtime's query (the library links no
// driver stub).
void* driver_fn(const char* name, int version) {
  void* f = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &f, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return f;
}

// Process-unique id of the current context; 0 if no context is current.
cudaError_t current_ctx_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    get_current = reinterpret_cast<CtxGetCurrentFn>(driver_fn("cuCtxGetCurrent", 4000));
    get_id = reinterpret_cast<CtxGetIdFn>(driver_fn("cuCtxGetId", 12000));
  });
  if (get_current == nullptr || get_id == nullptr) return cudaErrorDeviceUninitialized;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  *id = 0;
  if (ctx != nullptr && get_id(ctx, id) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  return cudaSuccess;
}

// Device address of g_static_scratch in the current device's current context.
cudaError_t static_scratch(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  unsigned long long id = 0;
  e = current_ctx_id(&id);
  if (e != cudaSuccess) return e;
  ScratchAddr& a = g_scratch_addr[dev];
  if (id != 0 && a.ptr != nullptr && a.ctx_id == id) {
    *out = a.ptr;
    return cudaSuccess;
  }
  // First call in this context (with no context current yet, the lookup
  // makes the device's primary context current).
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_static_scratch);
  if (e != cudaSuccess) return e;
  if (id == 0) {
    e = current_ctx_id(&id);
    if (e != cudaSuccess) return e;
    if (id == 0) return cudaErrorDeviceUninitialized;
  }
  a.ctx_id = id;
  a.ptr = p;
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" muon_status_t newton_schulz_batched_noalloc(const void* x, muon_dtype_t xdt,
                                                       const muon_view_t* view, int batch,
                                                       void* out, muon_dtype_t odt,
                                                       const muon_ns_schedule_t* schedule,
                                                       uint32_t* device_flags,
                                                       muon_stream_t stream) {
  size_t need = 0;
  muon_status_t s = newton_schulz_workspace_size(view, batch, schedule, &need);
  if (s != MUON_OK) return s;
  if (need > kStaticScratchBytes) return MUON_ERR_WORKSPACE_TOO_SMALL;
  if (device_flags != nullptr && (reinterpret_cast<uintptr_t>(device_flags) & 3u) != 0)
    return MUON_ERR_MISALIGNED;
  void* scratch = nullptr;
  if (static_scratch(&scratch) != cudaSuccess) return MUON_ERR_CUDA;
  s = newton_schulz_batched(x, xdt, view, batch, out, odt, schedule, scratch,
                            kStaticScratchBytes, stream);
  if (s != MUON_OK) return s;
  if (device_flags != nullptr) {
    // The status word is the first 4 bytes of the scratch area.
    if (cudaMemcpyAsync(device_flags, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice,
                        reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
      return MUON_ERR_CUDA;
  }
  return MUON_OK;
}
