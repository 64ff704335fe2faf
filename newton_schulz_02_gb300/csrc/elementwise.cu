// HBM-bound passes of the Muon step (no tensor cores):
//
//  * k_prepare_*: momentum M_t = mu*M + G and look-ahead X = mu*M_t + G
//    ("Muon 优化器" Algorithm 1; the 'ema' variant of "RFC-0023" §方案 1), or a
//    plain load for newton_schulz_batched; writes X as two bf16 planes
//    (hi, and lo = the rounding residual) into the workspace in the wide
//    orientation (transposing tall matrices through shared memory) with zero
//    padding, and per-block partial sums of X^2 for the Frobenius norm of
//    "Muon 优化器" §2.  16-byte vector accesses.
//  * k_finalize_norm: deterministic per-matrix sum of the partials -> 1/||X||_F.
//  * k_apply_*: W <- W*(1 - lr*wd*mask) - lr*scale*O' (Algorithm 1), or a
//    plain store of O' for newton_schulz_batched.
//
// All reductions run in a fixed order that depends on the matrix shape only,
// so a matrix gives bit-identical results whatever batch it is part of.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace muon {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 64;  // transpose tile (tall matrices)

__device__ __forceinline__ bool misaligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) != 0;
}

// ---- 8-element vector I/O ---------------------------------------------------
__device__ __forceinline__ void load8(const void* base, int64_t off, int dtype, float (&v)[8]) {
  if (dtype == MUON_BF16) {
    const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + off);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(h[k]);
      v[2 * k] = f.x;
      v[2 * k + 1] = f.y;
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + off);
    const float4 a = p[0], b = p[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}

__device__ __forceinline__ void store8(void* base, int64_t off, int dtype, const float (&v)[8]) {
  if (dtype == MUON_BF16) {
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int k = 0; k < 4; ++k) h[k] = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + off) = u;
  } else {
    float4* p = reinterpret_cast<float4*>(static_cast<float*>(base) + off);
    p[0] = make_float4(v[0], v[1], v[2], v[3]);
    p[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
}

// hi = bf16(v), lo = bf16(v - hi): v to about 16 significant bits.
__device__ __forceinline__ void split_bf16x8(const float (&v)[8], uint4& hi, uint4& lo) {
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&hi);
  __nv_bfloat162* l = reinterpret_cast<__nv_bfloat162*>(&lo);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    h[k] = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
    const float2 f = __bfloat1622float2(h[k]);
    l[k] = __floats2bfloat162_rn(v[2 * k] - f.x, v[2 * k + 1] - f.y);
  }
}

__device__ __forceinline__ void unpack_bf16x8(const uint4& u, float (&v)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = __bfloat1622float2(h[k]);
    v[2 * k] = f.x;
    v[2 * k + 1] = f.y;
  }
}

// Block-wide sum in a fixed order (warp shuffle tree, then warp 0).
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = v;
  __syncthreads();
  float s = 0.f;
  if (w == 0) {
    s = (l < (kThreads / 32)) ? red[l] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  }
  return s;  // valid in thread 0
}

// Momentum / look-ahead / load of 8 consecutive elements at `off`.
__device__ __forceinline__ void prepare8(const PrepareArgs& p, const void* g, float* m,
                                         int64_t off, float (&x)[8]) {
  float gv[8];
  load8(g, off, p.g_dtype, gv);
  if (p.mode == kPrepLoad) {
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = gv[k];
    return;
  }
  float mv[8];
  load8(m, off, MUON_F32, mv);
  if (p.mode == kPrepMomentumSgd) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float mt = fmaf(p.mu, mv[k], gv[k]);  // one rounding: M_t = mu*M + G
      mv[k] = mt;
      x[k] = p.nesterov ? fmaf(p.mu, mt, gv[k]) : mt;
    }
  } else {  // 'ema': exact products in fp64, one rounding to fp32
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float mt = static_cast<float>(fma(static_cast<double>(p.mu),
                                              static_cast<double>(mv[k]),
                                              p.ema_omb * static_cast<double>(gv[k])));
      mv[k] = mt;
      x[k] = fmaf(p.c_mom, mt, p.c_grad * gv[k]);
    }
  }
  store8(m, off, MUON_F32, mv);
}

struct MatrixPtrs {
  const void* g;
  float* m;
  bool skip;
};

__device__ __forceinline__ MatrixPtrs matrix_ptrs(const PrepareArgs& p, int b) {
  MatrixPtrs r;
  const int esz = p.g_dtype == MUON_BF16 ? 2 : 4;
  r.g = p.g_ptrs ? p.g_ptrs[b]
                 : static_cast<const void*>(static_cast<const char*>(p.g_base) +
                                            static_cast<int64_t>(b) * p.batch_stride * esz);
  r.m = (p.mode == kPrepLoad) ? nullptr : p.m_ptrs[b];
  bool bad = misaligned16(r.g) || (r.m && misaligned16(r.m));
  if (p.w_ptrs) bad = bad || misaligned16(p.w_ptrs[b]);
  r.skip = bad;
  return r;
}

// ---- pass 1, wide (rows <= cols): X_ws[i][j] = X[i][j] -----------------------
__global__ void __launch_bounds__(kThreads) k_prepare_wide(PrepareArgs p) {
  __shared__ float red[kThreads / 32];
  const int b = blockIdx.y;
  const MatrixPtrs mp = matrix_ptrs(p, b);
  if (mp.skip && blockIdx.x == 0 && threadIdx.x == 0) {
    p.skip[b] = 1;
    atomicOr(p.status, kFlagMisaligned);
  }
  const int64_t vpr = p.m_pad / 8;
  const int64_t total = static_cast<int64_t>(p.n_pad) * vpr;
  __nv_bfloat16* X = p.X + static_cast<int64_t>(b) * p.n_pad * p.m_pad;
  float acc = 0.f;
  for (int64_t v = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; v < total;
       v += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int i = static_cast<int>(v / vpr);
    const int j = static_cast<int>(v - static_cast<int64_t>(i) * vpr) * 8;
    float x[8];
    if (!mp.skip && i < p.rows && j < p.cols) {
      prepare8(p, mp.g, mp.m, static_cast<int64_t>(i) * p.row_stride + j, x);
#pragma unroll
      for (int k = 0; k < 8; ++k) acc = fmaf(x[k], x[k], acc);
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) x[k] = 0.f;
    }
    uint4 hi, lo;
    split_bf16x8(x, hi, lo);
    const int64_t o = static_cast<int64_t>(i) * p.m_pad + j;
    *reinterpret_cast<uint4*>(X + o) = hi;
    *reinterpret_cast<uint4*>(X + p.x_lo_off + o) = lo;
  }
  const float s = block_sum(acc, red);
  if (threadIdx.x == 0) p.partials[static_cast<int64_t>(b) * p.parts_stride + blockIdx.x] = s;
}

// ---- pass 1, tall (rows > cols): X_ws[j][i] = X[i][j] via 64x64 smem tiles ---
__global__ void __launch_bounds__(kThreads) k_prepare_tall(PrepareArgs p) {
  __shared__ float red[kThreads / 32];
  __shared__ float tile[kTile][kTile + 1];
  const int b = blockIdx.y;
  const MatrixPtrs mp = matrix_ptrs(p, b);
  if (mp.skip && blockIdx.x == 0 && threadIdx.x == 0) {
    p.skip[b] = 1;
    atomicOr(p.status, kFlagMisaligned);
  }
  // source tiles: rows (m dimension) x cols (n dimension)
  const int tiles_i = p.m_pad / kTile, tiles_j = p.n_pad / kTile;
  const int n_tiles = tiles_i * tiles_j;
  __nv_bfloat16* X = p.X + static_cast<int64_t>(b) * p.n_pad * p.m_pad;
  float acc = 0.f;
  for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
    const int i0 = (t / tiles_j) * kTile, j0 = (t % tiles_j) * kTile;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int q = threadIdx.x + k * kThreads;
      const int r = q >> 3, c8 = (q & 7) * 8;
      const int i = i0 + r, j = j0 + c8;
      float x[8];
      if (!mp.skip && i < p.rows && j < p.cols) {
        prepare8(p, mp.g, mp.m, static_cast<int64_t>(i) * p.row_stride + j, x);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(x[e], x[e], acc);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) tile[r][c8 + e] = x[e];
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int q = threadIdx.x + k * kThreads;
      const int jj = q >> 3, ii8 = (q & 7) * 8;
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = tile[ii8 + e][jj];
      uint4 hi, lo;
      split_bf16x8(v, hi, lo);
      const int64_t o = static_cast<int64_t>(j0 + jj) * p.m_pad + i0 + ii8;
      *reinterpret_cast<uint4*>(X + o) = hi;
      *reinterpret_cast<uint4*>(X + p.x_lo_off + o) = lo;
    }
    __syncthreads();
  }
  const float s = block_sum(acc, red);
  if (threadIdx.x == 0) p.partials[static_cast<int64_t>(b) * p.parts_stride + blockIdx.x] = s;
}

// ---- per-matrix norm ------------------------------------------------------------
// One warp per matrix: lane l adds partials l, l + 32, ... in order (double),
// then the lanes' sums meet in a fixed shuffle tree: a fixed order that
// depends on the partial count alone.
__global__ void __launch_bounds__(kThreads) k_finalize_norm(FinalizeArgs p) {
  griddep_wait();  // the partials come from the prepare pass
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int b = static_cast<int>((static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
  if (b >= p.batch) return;  // whole warps
  if (lane == 0 && p.gp_ctr != nullptr) p.gp_ctr[b] = 0;
  int seg = 0;
  while (seg + 1 < p.nseg && b >= p.seg_begin[seg + 1]) ++seg;
  const int parts = p.seg_parts[seg];
  const float* pp = p.partials + static_cast<int64_t>(b) * p.parts_stride;
  double s = 0.0;
  for (int k = lane; k < parts; k += 32) s += static_cast<double>(pp[k]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_down_sync(0xffffffffu, s, off);
  if (lane != 0) return;
  if (!isfinite(s)) atomicOr(p.status, kFlagNonFinite);
  float inv;
  if (p.skip[b]) {
    inv = 0.f;
  } else if (!p.normalize) {
    inv = 1.f;
  } else {
    inv = (s > 0.0) ? static_cast<float>(1.0 / sqrt(s)) : 0.f;
  }
  p.inv_s[b] = inv;
}

// ---- last pass, wide --------------------------------------------------------------
__device__ __forceinline__ void apply8(const ApplyArgs& p, int b, void* wbase, int64_t woff,
                                       const float (&o_in)[8]) {
  float o[8];
  const float os = p.oscale ? p.oscale[b] : 1.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) o[k] = o_in[k] * os;
  if (p.mode == 0) {
    const float decay = (p.wd_mask == nullptr || p.wd_mask[b]) ? p.decay_on : 1.f;
    float w[8];
    load8(wbase, woff, p.w_dtype, w);
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = fmaf(-p.lr_scale, o[k], w[k] * decay);
    store8(wbase, woff, p.w_dtype, w);
  } else {
    store8(wbase, woff, p.w_dtype, o);
  }
}

__device__ __forceinline__ void* apply_base(const ApplyArgs& p, int b) {
  if (p.mode == 0) return p.w_ptrs[b];
  const int esz = p.w_dtype == MUON_BF16 ? 2 : 4;
  return static_cast<char*>(p.out_base) + static_cast<int64_t>(b) * p.rows * p.cols * esz;
}

__global__ void __launch_bounds__(kThreads) k_apply_wide(ApplyArgs p) {
  griddep_wait();  // launched as a programmatic dependent of the last GEMM
  const int b = blockIdx.y;
  if (p.skip[b]) return;
  void* wbase = apply_base(p, b);
  const int64_t ld = p.mode == 0 ? p.row_stride : p.cols;
  const int64_t vpr = p.cols / 8;
  const int64_t total = static_cast<int64_t>(p.rows) * vpr;
  const __nv_bfloat16* X = p.X + static_cast<int64_t>(b) * p.n_pad * p.m_pad;
  for (int64_t v = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; v < total;
       v += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int i = static_cast<int>(v / vpr);
    const int j = static_cast<int>(v - static_cast<int64_t>(i) * vpr) * 8;
    const int64_t xo = static_cast<int64_t>(i) * p.m_pad + j;
    float o[8], ol[8];
    unpack_bf16x8(*reinterpret_cast<const uint4*>(X + xo), o);
    if (p.has_lo) {
      unpack_bf16x8(*reinterpret_cast<const uint4*>(X + p.x_lo_off + xo), ol);
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] += ol[e];
    }
    apply8(p, b, wbase, static_cast<int64_t>(i) * ld + j, o);
  }
}

// ---- last pass, tall: W[i][j] from X_ws[j][i] ----------------------------------------
__global__ void __launch_bounds__(kThreads) k_apply_tall(ApplyArgs p) {
  __shared__ float tile[kTile][kTile + 1];
  griddep_wait();  // launched as a programmatic dependent of the last GEMM
  const int b = blockIdx.y;
  if (p.skip[b]) return;
  void* wbase = apply_base(p, b);
  const int64_t ld = p.mode == 0 ? p.row_stride : p.cols;
  const int tiles_i = (p.rows + kTile - 1) / kTile, tiles_j = (p.cols + kTile - 1) / kTile;
  const int n_tiles = tiles_i * tiles_j;
  const __nv_bfloat16* X = p.X + static_cast<int64_t>(b) * p.n_pad * p.m_pad;
  for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
    const int i0 = (t / tiles_j) * kTile, j0 = (t % tiles_j) * kTile;
    // workspace rows j0.., columns i0..  (inside the padded workspace)
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int q = threadIdx.x + k * kThreads;
      const int jj = q >> 3, ii8 = (q & 7) * 8;
      const int64_t xo = static_cast<int64_t>(j0 + jj) * p.m_pad + i0 + ii8;
      float v[8], vl[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      unpack_bf16x8(*reinterpret_cast<const uint4*>(X + xo), v);
      if (p.has_lo) unpack_bf16x8(*reinterpret_cast<const uint4*>(X + p.x_lo_off + xo), vl);
#pragma unroll
      for (int e = 0; e < 8; ++e) tile[jj][ii8 + e] = v[e] + vl[e];
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int q = threadIdx.x + k * kThreads;
      const int r = q >> 3, c8 = (q & 7) * 8;
      const int i = i0 + r, j = j0 + c8;
      if (i < p.rows && j < p.cols) {
        float o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = tile[c8 + e][r];
        apply8(p, b, wbase, static_cast<int64_t>(i) * ld + j, o);
      }
    }
    __syncthreads();
  }
}

// ---- bounded-wait failure-path check -----------------------------------------------
__global__ void k_wait_timeout_check(uint32_t* status, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // Nobody arrives on `bar`: phase 0 never completes and the wait runs out.
    (void)mbar_wait_bounded(&bar, 0, &abort_flag, status, timeout_ns);
  }
  __syncthreads();
}

// Holds an SM for `ns` nanoseconds by the global timer, then exits: every
// block takes the dynamic shared memory it is launched with, so that no
// other large-shared-memory block fits beside it.
__global__ void k_occupy(uint64_t ns) {
  extern __shared__ uint8_t hold[];
  if (threadIdx.x == 0) {
    hold[0] = 0;
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < ns) __nanosleep(1000);
  }
}

}  // namespace

// Blocks per matrix: a function of the shape only (determinism across batch sizes).
int prepare_parts(int rows, int cols, int n_pad, int m_pad) {
  if (rows <= cols) {
    const int64_t vecs = static_cast<int64_t>(n_pad) * m_pad / 8;
    const int64_t want = (vecs + kThreads * 4 - 1) / (kThreads * 4);
    return static_cast<int>(want < 1 ? 1 : (want > 256 ? 256 : want));
  }
  const int64_t tiles = static_cast<int64_t>(m_pad / kTile) * (n_pad / kTile);
  return static_cast<int>(tiles > 256 ? 256 : tiles);
}

int apply_parts(int rows, int cols) {
  const int64_t vecs = static_cast<int64_t>(rows) * cols / 8;
  const int64_t want = (vecs + kThreads * 4 - 1) / (kThreads * 4);
  return static_cast<int>(want < 1 ? 1 : (want > 256 ? 256 : want));
}

cudaError_t launch_prepare(const PrepareArgs& a, cudaStream_t st) {
  dim3 grid(a.parts, a.batch);
  // algorithmic bytes: read G, read + write M (momentum modes), write X (hi + lo planes)
  const double elems = static_cast<double>(a.batch) * a.rows * a.cols;
  const double per = (a.g_dtype == MUON_BF16 ? 2.0 : 4.0) + (a.mode == kPrepLoad ? 0.0 : 8.0) + 4.0;
  prof_begin(kKindPrepare, st);
  if (a.tall)
    k_prepare_tall<<<grid, kThreads, 0, st>>>(a);
  else
    k_prepare_wide<<<grid, kThreads, 0, st>>>(a);
  prof_end(kKindPrepare, st, 0.0, elems * per);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const FinalizeArgs& a, cudaStream_t st) {
  // a programmatic dependent of the prepare pass (it waits for its partials)
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  const int64_t threads = static_cast<int64_t>(a.batch) * 32;
  cfg.gridDim = dim3(static_cast<unsigned>((threads + kThreads - 1) / kThreads));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_begin(kKindFinalize, st);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, k_finalize_norm, a);
  prof_end(kKindFinalize, st, 0.0, static_cast<double>(a.batch) * (a.parts_stride * 4.0 + 4.0));
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_apply(const ApplyArgs& a, cudaStream_t st) {
  dim3 grid(a.parts, a.batch);
  // algorithmic bytes: read O' (hi, and lo when present); read + write W (mode 0) or write out
  const double elems = static_cast<double>(a.batch) * a.rows * a.cols;
  const double wsz = a.w_dtype == MUON_BF16 ? 2.0 : 4.0;
  const double per = (a.has_lo ? 4.0 : 2.0) + (a.mode == 0 ? 2.0 * wsz : wsz);
  // programmatic dependent of the previous kernel (the last Newton–Schulz
  // GEMM, a persistent grid whose CTAs are all resident)
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_begin(kKindApply, st);
  const cudaError_t e = a.tall ? cudaLaunchKernelEx(&cfg, k_apply_tall, a)
                               : cudaLaunchKernelEx(&cfg, k_apply_wide, a);
  prof_end(kKindApply, st, 0.0, elems * per);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_occupy(int blocks, size_t smem_bytes, uint64_t ns, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(k_occupy, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem_bytes));
  if (e != cudaSuccess) return e;
  k_occupy<<<blocks, 32, smem_bytes, st>>>(ns);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout_check(uint32_t* status, uint64_t timeout_ns, cudaStream_t st) {
  prof_begin(kKindTimeoutCheck, st);
  k_wait_timeout_check<<<1, 32, 0, st>>>(status, timeout_ns);
  prof_end(kKindTimeoutCheck, st, 0.0, 0.0);
  return cudaGetLastError();
}

}  // namespace muon
