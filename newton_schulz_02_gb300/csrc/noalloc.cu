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
// taken once per device with cudaGetSymbolAddress (with that device current)
// on the first call made on that device.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/muon.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t{32} << 20;  // 32 MiB
constexpr int kMaxDevices = 128;

__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device (set up once per device).
cudaError_t static_scratch(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
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
