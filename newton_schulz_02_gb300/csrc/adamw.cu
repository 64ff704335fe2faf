// AdamW partition of the optimizer: the parameters that stay on AdamW next to
// Muon (embeddings, the output head, norm scales and other non-matrix
// tensors, "Muon 优化器" §3), with the per-tensor decay mask of
// "RFC-0023: 对齐 MaxText Muon 优化器实现与 Megatron-LM 完整行为" §方案 2.
// Per element, in fp32:
//
//   m <- beta1*m + (1 - beta1)*g
//   v <- beta2*v + (1 - beta2)*g^2
//   u  = (m / (1 - beta1^t)) / (sqrt(v / (1 - beta2^t)) + eps)
//   W <- W*(1 - lr*wd*mask) - lr*u
//
// One HBM pass (W, G, m, v read; W, m, v written: 22 bytes per parameter for
// bf16 W and G).  All groups of one call go into one launch (up to
// kAdamWMaxGroups groups per launch): the grid strides over fixed-size chunks of
// every tensor of every group, so small tensors (norm scales) and large ones
// (embeddings) share the launch and the grid stays a multiple of the SM count.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "internal.h"

namespace muon {
namespace {

constexpr int kThreads = 256;
constexpr int kVec = 8;                                  // elements per vector access
constexpr int kUnroll = 2;                               // vectors in flight per thread
constexpr int64_t kChunk = int64_t{kThreads} * kVec * kUnroll;  // elements per work item

struct AdamWLaunch {
  int n_groups;
  int64_t item_begin[kAdamWMaxGroups + 1];  // prefix sums of work items per group
  AdamWGroupArgs g[kAdamWMaxGroups];
  float lr, beta1, omb1, beta2, omb2, eps, c1, c2, decay_on;
  uint32_t* flags;
};

__device__ __forceinline__ void ld8(const void* p, int dtype, float (&x)[8]) {
  if (dtype == MUON_BF16) {
    const uint4 u = *static_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(h[k]);
      x[2 * k] = f.x;
      x[2 * k + 1] = f.y;
    }
  } else {
    const float4* q = static_cast<const float4*>(p);
    const float4 a = q[0], b = q[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
}

__device__ __forceinline__ void st8(void* p, int dtype, const float (&x)[8]) {
  if (dtype == MUON_BF16) {
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int k = 0; k < 4; ++k) h[k] = __floats2bfloat162_rn(x[2 * k], x[2 * k + 1]);
    *static_cast<uint4*>(p) = u;
  } else {
    float4* q = static_cast<float4*>(p);
    q[0] = make_float4(x[0], x[1], x[2], x[3]);
    q[1] = make_float4(x[4], x[5], x[6], x[7]);
  }
}

__device__ __forceinline__ float ld1(const void* base, int64_t i, int dtype) {
  return dtype == MUON_BF16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(base)[i])
                            : static_cast<const float*>(base)[i];
}

__device__ __forceinline__ void st1(void* base, int64_t i, int dtype, float x) {
  if (dtype == MUON_BF16)
    static_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(x);
  else
    static_cast<float*>(base)[i] = x;
}

struct Elem {
  float w, g, m, v;
};

__device__ __forceinline__ void adamw_elem(const AdamWLaunch& p, float decay, Elem& e) {
  e.m = fmaf(p.beta1, e.m, p.omb1 * e.g);
  e.v = fmaf(p.beta2, e.v, p.omb2 * (e.g * e.g));
  const float u = (e.m * p.c1) / (sqrtf(e.v * p.c2) + p.eps);
  e.w = fmaf(-p.lr, u, e.w * decay);
}

__device__ __forceinline__ bool misaligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) != 0;
}

__global__ void __launch_bounds__(kThreads) k_adamw(const __grid_constant__ AdamWLaunch p) {
  const int64_t total = p.item_begin[p.n_groups];
  for (int64_t item = blockIdx.x; item < total; item += gridDim.x) {
    int gi = 0;
    while (gi + 1 < p.n_groups && item >= p.item_begin[gi + 1]) ++gi;
    const AdamWGroupArgs& G = p.g[gi];
    const int64_t local = item - p.item_begin[gi];
    const int64_t tensor = local / G.chunks_per_tensor;
    const int64_t chunk = local - tensor * G.chunks_per_tensor;
    void* w = G.w_ptrs[tensor];
    const void* g = G.g_ptrs[tensor];
    float* m = G.m_ptrs[tensor];
    float* v = G.v_ptrs[tensor];
    if (misaligned16(w) || misaligned16(g) || misaligned16(m) || misaligned16(v)) {
      if (threadIdx.x == 0 && chunk == 0 && p.flags != nullptr)
        atomicOr(p.flags, MUON_FLAG_MISALIGNED);
      continue;  // the tensor is left untouched
    }
    const float decay = (G.wd_mask == nullptr || G.wd_mask[tensor]) ? p.decay_on : 1.f;
    const int wesz = G.w_dtype == MUON_BF16 ? 2 : 4, gesz = G.g_dtype == MUON_BF16 ? 2 : 4;
    const int64_t c0 = chunk * kChunk;
    // full vectors: loads of both vectors first, then the arithmetic
    int64_t idx[kUnroll];
    bool full[kUnroll];
    float W[kUnroll][8], Gv[kUnroll][8], Mv[kUnroll][8], Vv[kUnroll][8];
#pragma unroll
    for (int r = 0; r < kUnroll; ++r) {
      idx[r] = c0 + (static_cast<int64_t>(r) * kThreads + threadIdx.x) * kVec;
      full[r] = idx[r] + kVec <= G.numel;
      if (full[r]) {
        ld8(static_cast<const char*>(w) + idx[r] * wesz, G.w_dtype, W[r]);
        ld8(static_cast<const char*>(g) + idx[r] * gesz, G.g_dtype, Gv[r]);
        ld8(m + idx[r], MUON_F32, Mv[r]);
        ld8(v + idx[r], MUON_F32, Vv[r]);
      }
    }
#pragma unroll
    for (int r = 0; r < kUnroll; ++r) {
      if (full[r]) {
#pragma unroll
        for (int k = 0; k < kVec; ++k) {
          Elem e{W[r][k], Gv[r][k], Mv[r][k], Vv[r][k]};
          adamw_elem(p, decay, e);
          W[r][k] = e.w; Mv[r][k] = e.m; Vv[r][k] = e.v;
        }
        st8(static_cast<char*>(w) + idx[r] * wesz, G.w_dtype, W[r]);
        st8(m + idx[r], MUON_F32, Mv[r]);
        st8(v + idx[r], MUON_F32, Vv[r]);
      } else if (idx[r] < G.numel) {
        // ragged tail of the tensor (numel % 8 elements)
        for (int64_t i = idx[r]; i < G.numel; ++i) {
          Elem e{ld1(w, i, G.w_dtype), ld1(g, i, G.g_dtype), m[i], v[i]};
          adamw_elem(p, decay, e);
          st1(w, i, G.w_dtype, e.w);
          m[i] = e.m;
          v[i] = e.v;
        }
      }
    }
  }
}

int64_t chunks(int64_t numel) { return numel <= 0 ? 0 : (numel + kChunk - 1) / kChunk; }

// Resident blocks of k_adamw on the current device (SMs x blocks per SM).
cudaError_t resident_blocks(int* out) {
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_adamw, kThreads, 0);
  if (e != cudaSuccess) return e;
  *out = sms * (per_sm > 0 ? per_sm : 1);
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_adamw(AdamWGroupArgs* groups, int n_groups, const AdamWScalars& s,
                         uint32_t* flags, cudaStream_t st) {
  int resident = 0;
  cudaError_t e0 = resident_blocks(&resident);
  if (e0 != cudaSuccess) return e0;
  for (int i = 0; i < n_groups; ++i) groups[i].chunks_per_tensor = chunks(groups[i].numel);
  for (int base = 0; base < n_groups; base += kAdamWMaxGroups) {
    AdamWLaunch p{};
    p.n_groups = n_groups - base < kAdamWMaxGroups ? n_groups - base : kAdamWMaxGroups;
    p.item_begin[0] = 0;
    double bytes = 0.0;
    for (int i = 0; i < p.n_groups; ++i) {
      p.g[i] = groups[base + i];
      p.item_begin[i + 1] = p.item_begin[i] + p.g[i].chunks_per_tensor * p.g[i].count;
      const double n = static_cast<double>(p.g[i].numel) * p.g[i].count;
      bytes += n * (2.0 * (p.g[i].w_dtype == MUON_BF16 ? 2 : 4) +
                    (p.g[i].g_dtype == MUON_BF16 ? 2 : 4) + 16.0);
    }
    const int64_t items = p.item_begin[p.n_groups];
    if (items == 0) continue;
    p.lr = s.lr; p.beta1 = s.beta1; p.omb1 = s.omb1; p.beta2 = s.beta2; p.omb2 = s.omb2;
    p.eps = s.eps; p.c1 = s.c1; p.c2 = s.c2; p.decay_on = s.decay_on;
    p.flags = flags;
    // persistent grid: every resident block (a multiple of the SM count)
    const int grid = static_cast<int>(items < resident ? items : resident);
    prof_begin(kKindAdamW, st);
    k_adamw<<<grid, kThreads, 0, st>>>(p);
    prof_end(kKindAdamW, st, 0.0, bytes);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace muon
