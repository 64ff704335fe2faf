// C ABI of the batched Muon step (declared in include/muon.h).
//
// Host side only: argument validation (everything the host can check is
// checked before the first enqueue), shape grouping, workspace layout, and
// the per-group launch sequence
//   prepare (momentum / look-ahead / X -> workspace, partial sums of X^2)
//   -> finalize (1/||X||_F per matrix)
//   -> Newton–Schulz chain (tcgen05 GEMMs)
//   -> apply (scale, decoupled weight decay, write W) or store O'.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <tuple>
#include <vector>

#include "internal.h"

namespace {

using namespace muon;

std::atomic<uint64_t> g_timeout_ns{2000000000ull};

const muon_ns_stage_t kHybridStages[2] = {
    {8, 3.4445f, -4.7750f, 2.0315f},  // "Muon 优化器" §2, fast stage
    {2, 2.0f, -1.5f, 0.5f},           // stable stage
};

constexpr int kMaxDim = 1 << 20;
constexpr size_t kHeaderBytes = 256;  // status word + reserved

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_dtype(int d) { return d == MUON_BF16 || d == MUON_F32; }

int dsize(int d) { return d == MUON_BF16 ? 2 : 4; }

struct Layout {
  int n_pad = 0, m_pad = 0, parts = 0;
  int64_t lo_off = 0;     // elements from an iterate's hi plane to its lo plane
  int64_t sq_lo_off = 0;  // split-bf16: from S's (P's) hi plane to its lo plane
  size_t x0 = 0, x1 = 0, a = 0, b = 0, pdiag = 0, partials = 0, inv_s = 0, skip = 0, total = 0;
  size_t kslices = 0;     // split-K Gram slices (fp32), when gram_ksplit(...) > 1
  size_t gp_ctr = 0;      // [batch] int: Gram arrivals of the fused Gram + polynomial launches
  size_t gp_log = 0;      // ticket counters and log of those launches (gp_log_bytes; 0 = none)
  size_t gp_log_bytes = 0;
  int ksplit = 1;
};

int wide_n(const muon_view_t& v) { return v.rows < v.cols ? v.rows : v.cols; }
int wide_m(const muon_view_t& v) { return v.rows < v.cols ? v.cols : v.rows; }

// Workspace of one Newton–Schulz chain over `batch` matrices of padded wide
// shape n_pad x m_pad whose prepare passes write up to `parts` partial sums
// per matrix.
Layout layout_for(int batch, int n_pad, int m_pad, int parts, bool x3) {
  Layout L;
  L.n_pad = n_pad;
  L.m_pad = m_pad;
  L.parts = parts;
  const size_t xb = static_cast<size_t>(batch) * L.n_pad * L.m_pad * 2;
  const size_t sb = static_cast<size_t>(batch) * L.n_pad * L.n_pad * 2;
  L.lo_off = static_cast<int64_t>(align256(xb) / 2);
  size_t off = kHeaderBytes;
  // each iterate: hi plane, then lo plane (lo_off = batch*n_pad*m_pad elements)
  L.x0 = off; off += 2 * align256(xb);
  L.x1 = off; off += 2 * align256(xb);
  // S and P: hi plane (and, in the split-bf16 precision, a lo plane after it)
  L.sq_lo_off = static_cast<int64_t>(align256(sb) / 2);
  L.a = off; off += (x3 ? 2 : 1) * align256(sb);
  L.b = off; off += (x3 ? 2 : 1) * align256(sb);
  L.pdiag = off; off += align256(static_cast<size_t>(batch) * L.n_pad * 4);
  L.partials = off; off += align256(static_cast<size_t>(batch) * L.parts * 4);
  L.inv_s = off; off += align256(static_cast<size_t>(batch) * 4);
  L.skip = off; off += align256(static_cast<size_t>(batch));
  L.gp_ctr = off; off += align256(static_cast<size_t>(batch) * 4);
  L.gp_log_bytes = gram_poly_log_ints(batch, n_pad, x3) * 4;
  L.gp_log = off; off += align256(L.gp_log_bytes);
  L.ksplit = gram_ksplit(n_pad, m_pad, x3);
  if (L.ksplit > 1) {
    L.kslices = off;
    off += align256(static_cast<size_t>(L.ksplit) * batch * L.n_pad * L.n_pad * 4);
  }
  L.total = off;
  return L;
}

Layout layout_for(int batch, const muon_view_t& v, bool x3) {
  const int n_pad = static_cast<int>(round_up(wide_n(v), kPad));
  const int m_pad = static_cast<int>(round_up(wide_m(v), kPad));
  return layout_for(batch, n_pad, m_pad, prepare_parts(v.rows, v.cols, n_pad, m_pad), x3);
}

// Groups of one muon_step_batched call, cut into Newton–Schulz chains.  With
// merging, groups of the same wide shape (n, m) -- either orientation, so a
// 14336 x 4096 weight and a 4096 x 14336 one share a chain -- go through one
// chain of at most kMaxMerge groups, in order of first appearance;
// otherwise every group has its own chain.
struct Chain {
  std::vector<int> members;  // group indices, in batch order
  int batch = 0, n = 0, m = 0, n_pad = 0, m_pad = 0, parts = 0;
};

std::vector<Chain> plan_chains(const muon_group_t* groups, int n_groups, bool merge) {
  std::vector<Chain> chains;
  for (int i = 0; i < n_groups; ++i) {
    const muon_view_t& v = groups[i].view;
    const int n = wide_n(v), m = wide_m(v);
    Chain* c = nullptr;
    if (merge)
      for (Chain& k : chains)
        if (k.n == n && k.m == m && static_cast<int>(k.members.size()) < kMaxMerge) {
          c = &k;
          break;
        }
    if (c == nullptr) {
      chains.emplace_back();
      c = &chains.back();
      c->n = n;
      c->m = m;
      c->n_pad = static_cast<int>(round_up(n, kPad));
      c->m_pad = static_cast<int>(round_up(m, kPad));
    }
    c->members.push_back(i);
    c->batch += groups[i].batch;
    const int parts = prepare_parts(v.rows, v.cols, c->n_pad, c->m_pad);
    if (parts > c->parts) c->parts = parts;
  }
  return chains;
}

muon_status_t check_view(const muon_view_t& v) {
  if (v.rows < 1 || v.cols < 1 || v.rows > kMaxDim || v.cols > kMaxDim) return MUON_ERR_INVALID_ARG;
  if (v.row_stride < v.cols) return MUON_ERR_INVALID_ARG;
  if (v.fan_out_axis != 0 && v.fan_out_axis != 1) return MUON_ERR_INVALID_ARG;
  if (v.cols % 8 != 0) return MUON_ERR_UNSUPPORTED;
  if (v.row_stride % 8 != 0) return MUON_ERR_MISALIGNED;
  return MUON_OK;
}

muon_status_t expand_schedule(const muon_ns_schedule_t* s, std::vector<float>* coeffs,
                              int* normalize, bool* x3, bool* merge = nullptr) {
  muon_ns_schedule_t def;
  if (s == nullptr) {
    muon_ns_hybrid_schedule(&def);
    s = &def;
  }
  if (s->prec == MUON_NS_TF32) return MUON_ERR_UNSUPPORTED;
  if (s->prec != MUON_NS_BF16 && s->prec != MUON_NS_BF16X3) return MUON_ERR_INVALID_ARG;
  if (s->n_stages < 0 || (s->n_stages > 0 && s->stages == nullptr)) return MUON_ERR_INVALID_ARG;
  if (s->normalize != 0 && s->normalize != 1) return MUON_ERR_INVALID_ARG;
  if (s->merge_groups != 0 && s->merge_groups != 1) return MUON_ERR_INVALID_ARG;
  coeffs->clear();
  for (int i = 0; i < s->n_stages; ++i) {
    const muon_ns_stage_t& st = s->stages[i];
    if (st.steps < 0 || st.steps > 1000) return MUON_ERR_INVALID_ARG;
    if (!std::isfinite(st.a) || !std::isfinite(st.b) || !std::isfinite(st.c))
      return MUON_ERR_INVALID_ARG;
    for (int k = 0; k < st.steps; ++k) {
      coeffs->push_back(st.a);
      coeffs->push_back(st.b);
      coeffs->push_back(st.c);
    }
  }
  *normalize = s->normalize;
  *x3 = (s->prec == MUON_NS_BF16X3);
  if (merge != nullptr) *merge = (s->merge_groups == 1);
  return MUON_OK;
}

// Update scale (host, double): "Muon 优化器" Algorithm 1 (spectral) and
// "Scaling for MuP over Muon optimizer" (unit_rms_norm).
double update_scale(const muon_view_t& v, muon_scale_mode_t mode, float gamma) {
  const double r = v.rows, c = v.cols;
  switch (mode) {
    case MUON_SCALE_SPECTRAL: return std::sqrt(r > c ? r : c) * static_cast<double>(gamma);
    case MUON_SCALE_UNIT_RMS_NORM: {
      const double fan_out = v.fan_out_axis == 0 ? r : c;
      const double fan_in = v.fan_out_axis == 0 ? c : r;
      return std::sqrt(fan_out / fan_in);
    }
    default: return 1.0;
  }
}

muon_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MUON_OK : MUON_ERR_CUDA; }

// One segment of a chain: a group's matrices [begin, begin + batch) and the
// arguments of its last pass (W update or dense output).
struct Segment {
  int begin = 0, batch = 0, parts = 0;
  muon_view_t view{};
  ApplyArgs ap{};
};

// Shared tail of both entry points: norm, NS chain, last pass, over the
// chain's segments (each already prepared into its slice of the workspace).
muon_status_t run_chain_tail(const Layout& L, char* ws, int batch, int n, int m,
                             const std::vector<Segment>& segs, const std::vector<float>& coeffs,
                             int normalize, bool x3, cudaStream_t st) {
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  FinalizeArgs fa{};
  fa.batch = batch;
  fa.parts_stride = L.parts;
  fa.nseg = static_cast<int>(segs.size());
  for (size_t k = 0; k < segs.size(); ++k) {
    fa.seg_begin[k] = segs[k].begin;
    fa.seg_parts[k] = segs[k].parts;
  }
  fa.partials = reinterpret_cast<const float*>(ws + L.partials);
  fa.skip = reinterpret_cast<const uint8_t*>(ws + L.skip);
  fa.inv_s = reinterpret_cast<float*>(ws + L.inv_s);
  fa.normalize = normalize;
  fa.status = status;
  fa.gp_ctr = reinterpret_cast<int*>(ws + L.gp_ctr);
  if (L.gp_log_bytes > 0 && cudaMemsetAsync(ws + L.gp_log, 0, L.gp_log_bytes, st) != cudaSuccess)
    return MUON_ERR_CUDA;
  cudaError_t e = launch_finalize(fa, st);
  if (e != cudaSuccess) return MUON_ERR_CUDA;

  const int iters = static_cast<int>(coeffs.size() / 3);
  NsChainArgs na{};
  na.batch = batch;
  na.n_pad = L.n_pad;
  na.m_pad = L.m_pad;
  na.n = n;
  na.m = m;
  na.X0 = reinterpret_cast<__nv_bfloat16*>(ws + L.x0);
  na.X1 = reinterpret_cast<__nv_bfloat16*>(ws + L.x1);
  na.lo_off = L.lo_off;
  na.A = reinterpret_cast<__nv_bfloat16*>(ws + L.a);
  na.B = reinterpret_cast<__nv_bfloat16*>(ws + L.b);
  na.pdiag = reinterpret_cast<float*>(ws + L.pdiag);
  na.inv_s = normalize ? reinterpret_cast<const float*>(ws + L.inv_s) : nullptr;
  na.coeffs = coeffs.data();
  na.iters = iters;
  na.status = status;
  na.timeout_ns = g_timeout_ns.load();
  na.x3 = x3 ? 1 : 0;
  na.sq_lo_off = L.sq_lo_off;
  na.partial = L.ksplit > 1 ? reinterpret_cast<float*>(ws + L.kslices) : nullptr;
  na.gp_ctr = reinterpret_cast<int*>(ws + L.gp_ctr);
  if (L.gp_log_bytes > 0) {
    na.gp_tick = reinterpret_cast<int*>(ws + L.gp_log);
    na.gp_log = na.gp_tick + kGpMaxLaunches;
  }
  const bool fused = ns_final_fused(iters, x3);
  if (fused) {
    // the last update's epilogue writes W (or the output) from its fp32 result
    FinalStore& f = na.fin;
    f.mode = segs[0].ap.mode == 0 ? 1 : 2;
    f.nseg = static_cast<int>(segs.size());
    f.skip = reinterpret_cast<const uint8_t*>(ws + L.skip);
    for (size_t k = 0; k < segs.size(); ++k) {
      const ApplyArgs& ap = segs[k].ap;
      FinalSeg& g = f.seg[k];
      g.begin = segs[k].begin;
      g.rows = segs[k].view.rows;
      g.cols = segs[k].view.cols;
      g.tall = segs[k].view.rows > segs[k].view.cols;
      g.dtype = ap.w_dtype;
      g.w_ptrs = ap.w_ptrs;
      g.w_ld = ap.row_stride;
      g.out_base = ap.out_base;
      g.wd_mask = ap.wd_mask;
      g.decay_on = ap.decay_on;
      g.lr_scale = ap.lr_scale;
    }
  }
  e = run_ns_chain(na, st);
  if (e == cudaErrorNotSupported) return MUON_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return MUON_ERR_CUDA;
  if (fused) return MUON_OK;

  for (const Segment& sg : segs) {
    ApplyArgs ap = sg.ap;
    const int64_t off = static_cast<int64_t>(sg.begin);
    ap.X = ((iters % 2 == 0) ? na.X0 : na.X1) + off * L.n_pad * L.m_pad;
    ap.x_lo_off = L.lo_off;
    ap.has_lo = ns_final_has_lo(iters, x3) ? 1 : 0;
    ap.n_pad = L.n_pad;
    ap.m_pad = L.m_pad;
    ap.tall = sg.view.rows > sg.view.cols;
    ap.parts = apply_parts(sg.view.rows, sg.view.cols);
    ap.skip = reinterpret_cast<const uint8_t*>(ws + L.skip) + off;
    ap.oscale = (iters == 0 && normalize) ? reinterpret_cast<const float*>(ws + L.inv_s) + off
                                          : nullptr;
    const muon_status_t r = cuda_status(launch_apply(ap, st));
    if (r != MUON_OK) return r;
  }
  return MUON_OK;
}

size_t step_workspace_bytes(const muon_group_t* groups, int n_groups, bool merge, bool x3) {
  size_t need = kHeaderBytes;
  for (const Chain& c : plan_chains(groups, n_groups, merge)) {
    const Layout L = layout_for(c.batch, c.n_pad, c.m_pad, c.parts, x3);
    if (L.total > need) need = L.total;
  }
  return need;
}

muon_status_t check_workspace(const void* ws, size_t bytes, size_t need) {
  if (ws == nullptr) return MUON_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MUON_ERR_MISALIGNED;
  if (bytes < need) return MUON_ERR_WORKSPACE_TOO_SMALL;
  return MUON_OK;
}

}  // namespace

extern "C" {

muon_status_t muon_ns_hybrid_schedule(muon_ns_schedule_t* out) {
  if (out == nullptr) return MUON_ERR_INVALID_ARG;
  out->stages = kHybridStages;
  out->n_stages = 2;
  out->normalize = 1;
  out->merge_groups = 0;
  out->prec = MUON_NS_BF16;
  return MUON_OK;
}

muon_status_t muon_group_by_shape(const muon_tensor_desc_t* t, int n, int max_batch,
                                  int* group_of_tensor, int* n_groups) {
  if (n < 0 || max_batch < 0 || n_groups == nullptr) return MUON_ERR_INVALID_ARG;
  if (n > 0 && (t == nullptr || group_of_tensor == nullptr)) return MUON_ERR_INVALID_ARG;
  using Key = std::tuple<int, int, int64_t, int, int, int>;
  std::vector<Key> order;
  std::map<Key, std::vector<int>> members;
  for (int i = 0; i < n; ++i) {
    const Key k{t[i].rows, t[i].cols, t[i].row_stride, static_cast<int>(t[i].w_dtype),
                static_cast<int>(t[i].g_dtype), t[i].fan_out_axis};
    auto it = members.find(k);
    if (it == members.end()) {
      order.push_back(k);
      members[k].push_back(i);
    } else {
      it->second.push_back(i);
    }
  }
  int g = 0;
  for (const Key& k : order) {
    const std::vector<int>& idx = members[k];
    const size_t step = max_batch == 0 ? idx.size() : static_cast<size_t>(max_batch);
    for (size_t s = 0; s < idx.size(); s += step) {
      for (size_t j = s; j < idx.size() && j < s + step; ++j) group_of_tensor[idx[j]] = g;
      ++g;
    }
  }
  *n_groups = g;
  return MUON_OK;
}

muon_status_t muon_step_workspace_size(const muon_group_t* groups, int n_groups,
                                       const muon_ns_schedule_t* schedule, size_t* bytes) {
  if (bytes == nullptr || n_groups < 0 || (n_groups > 0 && groups == nullptr))
    return MUON_ERR_INVALID_ARG;
  std::vector<float> coeffs;
  int normalize = 1;
  bool x3 = false, merge = false;
  muon_status_t s = expand_schedule(schedule, &coeffs, &normalize, &x3, &merge);
  if (s != MUON_OK) return s;
  for (int i = 0; i < n_groups; ++i) {
    if (groups[i].batch < 1) return MUON_ERR_INVALID_ARG;
    s = check_view(groups[i].view);
    if (s != MUON_OK) return s;
  }
  *bytes = step_workspace_bytes(groups, n_groups, merge, x3);
  return MUON_OK;
}

muon_status_t muon_step_batched(const muon_group_t* groups, int n_groups,
                                const muon_hparams_t* hp, const muon_ns_schedule_t* schedule,
                                void* workspace, size_t workspace_bytes, muon_stream_t stream) {
  if (hp == nullptr || n_groups < 0 || (n_groups > 0 && groups == nullptr))
    return MUON_ERR_INVALID_ARG;
  if (!std::isfinite(hp->mu) || !std::isfinite(hp->lr) || !std::isfinite(hp->weight_decay) ||
      !std::isfinite(hp->gamma))
    return MUON_ERR_INVALID_ARG;
  if (hp->style != MUON_NESTEROV_SGD && hp->style != MUON_NESTEROV_EMA) return MUON_ERR_INVALID_ARG;
  if (hp->nesterov != 0 && hp->nesterov != 1) return MUON_ERR_INVALID_ARG;
  if (hp->scale_mode != MUON_SCALE_SPECTRAL && hp->scale_mode != MUON_SCALE_UNIT_RMS_NORM &&
      hp->scale_mode != MUON_SCALE_NONE)
    return MUON_ERR_INVALID_ARG;
  if (hp->style == MUON_NESTEROV_EMA && (hp->t < 1 || hp->mu >= 1.f || hp->mu < 0.f))
    return MUON_ERR_INVALID_ARG;
  std::vector<float> coeffs;
  int normalize = 1;
  bool x3 = false, merge = false;
  muon_status_t s = expand_schedule(schedule, &coeffs, &normalize, &x3, &merge);
  if (s != MUON_OK) return s;
  for (int i = 0; i < n_groups; ++i) {
    const muon_group_t& g = groups[i];
    if (g.batch < 1 || g.w_ptrs == nullptr || g.g_ptrs == nullptr || g.m_ptrs == nullptr)
      return MUON_ERR_INVALID_ARG;
    if (!valid_dtype(g.w_dtype) || !valid_dtype(g.g_dtype)) return MUON_ERR_INVALID_ARG;
    s = check_view(g.view);
    if (s != MUON_OK) return s;
  }
  size_t need = 0;
  s = muon_step_workspace_size(groups, n_groups, schedule, &need);
  if (s != MUON_OK) return s;
  s = check_workspace(workspace, workspace_bytes, need);
  if (s != MUON_OK) return s;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  if (cudaMemsetAsync(ws, 0, kHeaderBytes, st) != cudaSuccess) return MUON_ERR_CUDA;

  // 'ema' look-ahead coefficients, from the fp32 beta, in double.
  const double beta = hp->mu;
  double c_mom = 0.0, c_grad = 0.0;
  if (hp->style == MUON_NESTEROV_EMA) {
    const double t = static_cast<double>(hp->t);
    if (hp->nesterov) {
      c_mom = beta / (1.0 - std::pow(beta, t + 1.0));
      c_grad = (1.0 - beta) / (1.0 - std::pow(beta, t));
    } else {
      c_mom = 1.0 / (1.0 - std::pow(beta, t));
    }
  }

  const float decay_on = static_cast<float>(1.0 - static_cast<double>(hp->lr) * hp->weight_decay);
  for (const Chain& c : plan_chains(groups, n_groups, merge)) {
    const Layout L = layout_for(c.batch, c.n_pad, c.m_pad, c.parts, x3);
    if (cudaMemsetAsync(ws + L.skip, 0, static_cast<size_t>(c.batch), st) != cudaSuccess)
      return MUON_ERR_CUDA;
    std::vector<Segment> segs;
    int begin = 0;
    for (int gi : c.members) {
      const muon_group_t& g = groups[gi];
      const int64_t off = begin;
      PrepareArgs pa{};
      pa.batch = g.batch;
      pa.rows = g.view.rows;
      pa.cols = g.view.cols;
      pa.row_stride = g.view.row_stride;
      pa.g_dtype = g.g_dtype;
      pa.g_ptrs = g.g_ptrs;
      pa.m_ptrs = g.m_ptrs;
      pa.w_ptrs = g.w_ptrs;
      pa.mode = hp->style == MUON_NESTEROV_SGD ? kPrepMomentumSgd : kPrepMomentumEma;
      pa.nesterov = hp->nesterov;
      pa.mu = hp->mu;
      pa.ema_omb = 1.0 - beta;
      pa.c_mom = static_cast<float>(c_mom);
      pa.c_grad = static_cast<float>(c_grad);
      pa.X = reinterpret_cast<__nv_bfloat16*>(ws + L.x0) + off * L.n_pad * L.m_pad;
      pa.x_lo_off = L.lo_off;
      pa.n_pad = L.n_pad;
      pa.m_pad = L.m_pad;
      pa.tall = g.view.rows > g.view.cols;
      pa.parts = prepare_parts(g.view.rows, g.view.cols, L.n_pad, L.m_pad);
      pa.parts_stride = L.parts;
      pa.partials = reinterpret_cast<float*>(ws + L.partials) + off * L.parts;
      pa.skip = reinterpret_cast<uint8_t*>(ws + L.skip) + off;
      pa.status = reinterpret_cast<uint32_t*>(ws);
      if (launch_prepare(pa, st) != cudaSuccess) return MUON_ERR_CUDA;

      Segment sg;
      sg.begin = begin;
      sg.batch = g.batch;
      sg.parts = pa.parts;
      sg.view = g.view;
      ApplyArgs& ap = sg.ap;
      ap.batch = g.batch;
      ap.rows = g.view.rows;
      ap.cols = g.view.cols;
      ap.row_stride = g.view.row_stride;
      ap.mode = 0;
      ap.w_dtype = g.w_dtype;
      ap.w_ptrs = g.w_ptrs;
      ap.wd_mask = g.wd_mask;
      ap.decay_on = decay_on;
      ap.lr_scale = static_cast<float>(static_cast<double>(hp->lr) *
                                       update_scale(g.view, hp->scale_mode, hp->gamma));
      segs.push_back(sg);
      begin += g.batch;
    }
    s = run_chain_tail(L, ws, c.batch, c.n, c.m, segs, coeffs, normalize, x3, st);
    if (s != MUON_OK) return s;
  }
  return MUON_OK;
}

muon_status_t newton_schulz_workspace_size(const muon_view_t* view, int batch,
                                           const muon_ns_schedule_t* schedule, size_t* bytes) {
  if (view == nullptr || bytes == nullptr || batch < 1) return MUON_ERR_INVALID_ARG;
  muon_status_t s = check_view(*view);
  if (s != MUON_OK) return s;
  std::vector<float> coeffs;
  int normalize = 1;
  bool x3 = false;
  s = expand_schedule(schedule, &coeffs, &normalize, &x3);
  if (s != MUON_OK) return s;
  *bytes = layout_for(batch, *view, x3).total;
  return MUON_OK;
}

muon_status_t newton_schulz_batched(const void* x, muon_dtype_t xdt, const muon_view_t* view,
                                    int batch, void* out, muon_dtype_t odt,
                                    const muon_ns_schedule_t* schedule, void* workspace,
                                    size_t workspace_bytes, muon_stream_t stream) {
  if (x == nullptr || out == nullptr || view == nullptr || batch < 1) return MUON_ERR_INVALID_ARG;
  if (!valid_dtype(xdt) || !valid_dtype(odt)) return MUON_ERR_INVALID_ARG;
  muon_status_t s = check_view(*view);
  if (s != MUON_OK) return s;
  if (batch > 1 && view->batch_stride < 0) return MUON_ERR_INVALID_ARG;
  if (view->batch_stride % 8 != 0) return MUON_ERR_MISALIGNED;
  if (!aligned16(x) || !aligned16(out)) return MUON_ERR_MISALIGNED;
  // x and out must not overlap
  {
    const char* xb = static_cast<const char*>(x);
    const char* xe = xb + (static_cast<int64_t>(batch - 1) * view->batch_stride +
                           static_cast<int64_t>(view->rows - 1) * view->row_stride + view->cols) *
                              dsize(xdt);
    const char* ob = static_cast<const char*>(out);
    const char* oe = ob + static_cast<int64_t>(batch) * view->rows * view->cols * dsize(odt);
    if (xb < oe && ob < xe) return MUON_ERR_INVALID_ARG;
  }
  std::vector<float> coeffs;
  int normalize = 1;
  bool x3 = false;
  s = expand_schedule(schedule, &coeffs, &normalize, &x3);
  if (s != MUON_OK) return s;
  const Layout L = layout_for(batch, *view, x3);
  s = check_workspace(workspace, workspace_bytes, L.total);
  if (s != MUON_OK) return s;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  if (cudaMemsetAsync(ws, 0, kHeaderBytes, st) != cudaSuccess) return MUON_ERR_CUDA;
  if (cudaMemsetAsync(ws + L.skip, 0, static_cast<size_t>(batch), st) != cudaSuccess)
    return MUON_ERR_CUDA;

  PrepareArgs pa{};
  pa.batch = batch;
  pa.rows = view->rows;
  pa.cols = view->cols;
  pa.row_stride = view->row_stride;
  pa.batch_stride = view->batch_stride;
  pa.g_dtype = xdt;
  pa.g_base = x;
  pa.mode = kPrepLoad;
  pa.X = reinterpret_cast<__nv_bfloat16*>(ws + L.x0);
  pa.x_lo_off = L.lo_off;
  pa.n_pad = L.n_pad;
  pa.m_pad = L.m_pad;
  pa.tall = view->rows > view->cols;
  pa.parts = L.parts;
  pa.parts_stride = L.parts;
  pa.partials = reinterpret_cast<float*>(ws + L.partials);
  pa.skip = reinterpret_cast<uint8_t*>(ws + L.skip);
  pa.status = reinterpret_cast<uint32_t*>(ws);
  if (launch_prepare(pa, st) != cudaSuccess) return MUON_ERR_CUDA;

  Segment sg;
  sg.begin = 0;
  sg.batch = batch;
  sg.parts = L.parts;
  sg.view = *view;
  sg.ap.batch = batch;
  sg.ap.rows = view->rows;
  sg.ap.cols = view->cols;
  sg.ap.mode = 1;
  sg.ap.w_dtype = odt;
  sg.ap.out_base = out;
  return run_chain_tail(L, ws, batch, wide_n(*view), wide_m(*view), {sg}, coeffs, normalize, x3,
                        st);
}

muon_status_t muon_get_status(const void* workspace, muon_stream_t stream, uint32_t* flags) {
  if (workspace == nullptr || flags == nullptr) return MUON_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MUON_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MUON_ERR_CUDA;
  *flags = v;
  return (v & MUON_FLAG_TIMEOUT) ? MUON_ERR_TIMEOUT : MUON_OK;
}

muon_status_t muon_set_wait_timeout_ns(uint64_t ns) {
  if (ns == 0) return MUON_ERR_INVALID_ARG;
  g_timeout_ns.store(ns);
  return MUON_OK;
}

muon_status_t muon_check_wait_timeout(void* workspace, size_t workspace_bytes,
                                      uint64_t timeout_ns, muon_stream_t stream) {
  muon_status_t s = check_workspace(workspace, workspace_bytes, kHeaderBytes);
  if (s != MUON_OK) return s;
  if (timeout_ns == 0 || timeout_ns > 10000000000ull) return MUON_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace, 0, kHeaderBytes, st) != cudaSuccess) return MUON_ERR_CUDA;
  return cuda_status(
      launch_wait_timeout_check(static_cast<uint32_t*>(workspace), timeout_ns, st));
}

muon_status_t muon_occupy_sms(int blocks, size_t smem_bytes, uint64_t ns, muon_stream_t stream) {
  if (blocks < 1 || blocks > 4096 || smem_bytes > (size_t{227} << 10) || ns == 0 ||
      ns > 1000000000ull)
    return MUON_ERR_INVALID_ARG;
  return cuda_status(launch_occupy(blocks, smem_bytes, ns, reinterpret_cast<cudaStream_t>(stream)));
}

muon_status_t muon_adamw_step(const muon_adamw_group_t* groups, int n_groups,
                              const muon_adamw_hparams_t* hp, uint32_t* device_flags,
                              muon_stream_t stream) {
  if (hp == nullptr || n_groups < 0 || (n_groups > 0 && groups == nullptr))
    return MUON_ERR_INVALID_ARG;
  if (hp->t < 1 || !(hp->beta1 >= 0.f && hp->beta1 < 1.f) || !(hp->beta2 >= 0.f && hp->beta2 < 1.f))
    return MUON_ERR_INVALID_ARG;
  if (!(hp->eps >= 0.f) || !std::isfinite(hp->eps) || !std::isfinite(hp->lr) ||
      !std::isfinite(hp->weight_decay))
    return MUON_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(device_flags) & 3u) != 0) return MUON_ERR_MISALIGNED;
  std::vector<AdamWGroupArgs> args;
  args.reserve(static_cast<size_t>(n_groups));
  for (int i = 0; i < n_groups; ++i) {
    const muon_adamw_group_t& g = groups[i];
    if (g.count < 0 || g.numel < 0) return MUON_ERR_INVALID_ARG;
    if (!valid_dtype(g.w_dtype) || !valid_dtype(g.g_dtype)) return MUON_ERR_INVALID_ARG;
    if (g.count == 0 || g.numel == 0) continue;
    if (g.w_ptrs == nullptr || g.g_ptrs == nullptr || g.m_ptrs == nullptr || g.v_ptrs == nullptr)
      return MUON_ERR_INVALID_ARG;
    AdamWGroupArgs a{};
    a.count = g.count;
    a.numel = g.numel;
    a.w_dtype = g.w_dtype;
    a.g_dtype = g.g_dtype;
    a.w_ptrs = g.w_ptrs;
    a.g_ptrs = g.g_ptrs;
    a.m_ptrs = g.m_ptrs;
    a.v_ptrs = g.v_ptrs;
    a.wd_mask = g.wd_mask;
    args.push_back(a);
  }
  if (args.empty()) return MUON_OK;
  // bias corrections and coefficients in double from the fp32 values given
  const double b1 = hp->beta1, b2 = hp->beta2, t = static_cast<double>(hp->t);
  AdamWScalars sc{};
  sc.lr = hp->lr;
  sc.beta1 = hp->beta1;
  sc.beta2 = hp->beta2;
  sc.omb1 = static_cast<float>(1.0 - b1);
  sc.omb2 = static_cast<float>(1.0 - b2);
  sc.eps = hp->eps;
  sc.c1 = static_cast<float>(1.0 / (1.0 - std::pow(b1, t)));
  sc.c2 = static_cast<float>(1.0 / (1.0 - std::pow(b2, t)));
  sc.decay_on = static_cast<float>(1.0 - static_cast<double>(hp->lr) * hp->weight_decay);
  return cuda_status(launch_adamw(args.data(), static_cast<int>(args.size()), sc, device_flags,
                                  reinterpret_cast<cudaStream_t>(stream)));
}

const char* muon_status_string(muon_status_t s) {
  switch (s) {
    case MUON_OK: return "MUON_OK";
    case MUON_ERR_INVALID_ARG: return "MUON_ERR_INVALID_ARG";
    case MUON_ERR_MISALIGNED: return "MUON_ERR_MISALIGNED";
    case MUON_ERR_UNSUPPORTED: return "MUON_ERR_UNSUPPORTED";
    case MUON_ERR_WORKSPACE_TOO_SMALL: return "MUON_ERR_WORKSPACE_TOO_SMALL";
    case MUON_ERR_CUDA: return "MUON_ERR_CUDA";
    case MUON_ERR_TIMEOUT: return "MUON_ERR_TIMEOUT";
  }
  return "MUON_ERR_UNKNOWN";
}

}  // extern "C"
