// Launch counters and optional per-launch CUDA-event timing.
//
// prof_begin/prof_end bracket every kernel launch of the library.  Launches
// and algorithmic work are always counted; when timing is on, an event pair
// is recorded on the launching stream and resolved lazily by
// muon_profile_query / muon_profile_reset.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <vector>

#include "internal.h"

namespace muon {
namespace {

struct KindStats {
  uint64_t launches = 0;
  double ms = 0.0, flops = 0.0, bytes = 0.0;
};

struct Pending {
  int kind;
  cudaEvent_t start, stop;
};

const char* const kNames[kKindCount] = {"prepare", "finalize_norm", "ns_gram", "ns_poly",
                                        "ns_update", "apply", "timeout_check", "adamw",
                                        "ns_gram_poly", "ns_chain"};

std::mutex g_mu;
bool g_timing = false;
KindStats g_stats[kKindCount];
std::vector<Pending> g_pending;
std::vector<cudaEvent_t> g_pool;
cudaEvent_t g_open[kKindCount] = {};

cudaEvent_t take_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Resolve all pending event pairs (caller holds g_mu).
void drain_locked() {
  for (const Pending& p : g_pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(p.stop) == cudaSuccess &&
        cudaEventElapsedTime(&ms, p.start, p.stop) == cudaSuccess)
      g_stats[p.kind].ms += ms;
    g_pool.push_back(p.start);
    g_pool.push_back(p.stop);
  }
  g_pending.clear();
}

}  // namespace

void prof_begin(KernelKind k, cudaStream_t st) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_open[k] = nullptr;
  if (!g_timing) return;
  cudaEvent_t e = take_event();
  if (e != nullptr && cudaEventRecord(e, st) == cudaSuccess) g_open[k] = e;
}

void prof_end(KernelKind k, cudaStream_t st, double alg_flops, double alg_bytes) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_stats[k].launches += 1;
  g_stats[k].flops += alg_flops;
  g_stats[k].bytes += alg_bytes;
  if (g_open[k] == nullptr) return;
  cudaEvent_t e = take_event();
  if (e != nullptr && cudaEventRecord(e, st) == cudaSuccess) {
    g_pending.push_back({static_cast<int>(k), g_open[k], e});
  } else {
    g_pool.push_back(g_open[k]);
  }
  g_open[k] = nullptr;
}

}  // namespace muon

extern "C" {

muon_status_t muon_profile_enable(int on) {
  if (on != 0 && on != 1) return MUON_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(muon::g_mu);
  muon::g_timing = on != 0;
  return MUON_OK;
}

muon_status_t muon_profile_reset(void) {
  std::lock_guard<std::mutex> lk(muon::g_mu);
  muon::drain_locked();
  for (auto& s : muon::g_stats) s = muon::KindStats{};
  return MUON_OK;
}

muon_status_t muon_profile_query(muon_kernel_stats_t* out, int capacity, int* n) {
  if (n == nullptr || capacity < 0 || (capacity > 0 && out == nullptr)) return MUON_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(muon::g_mu);
  muon::drain_locked();
  for (int k = 0; k < muon::kKindCount && k < capacity; ++k) {
    std::memset(out[k].name, 0, sizeof(out[k].name));
    std::strncpy(out[k].name, muon::kNames[k], sizeof(out[k].name) - 1);
    out[k].launches = muon::g_stats[k].launches;
    out[k].total_ms = muon::g_stats[k].ms;
    out[k].alg_flops = muon::g_stats[k].flops;
    out[k].alg_bytes = muon::g_stats[k].bytes;
  }
  *n = muon::kKindCount;
  return MUON_OK;
}

}  // extern "C"
