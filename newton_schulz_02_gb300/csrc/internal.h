// Internal interface between the C-ABI layer (muon_api.cu) and the kernels.
// Not installed; the public interface is include/muon.h.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/muon.h"

namespace muon {

constexpr uint32_t kFlagNonFinite = MUON_FLAG_NONFINITE;
constexpr uint32_t kFlagTimeout = MUON_FLAG_TIMEOUT;
constexpr uint32_t kFlagMisaligned = MUON_FLAG_MISALIGNED;

// Newton–Schulz work is done on the "wide" orientation n x m (n = min(rows,
// cols), m = max), zero-padded to multiples of kPad in both dimensions so the
// tensor-core kernels only ever see whole tiles.  Zero padding is exact: the
// padded rows/columns of X, X X^T and of every later iterate stay zero.
constexpr int kPad = 128;

inline int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

enum PrepMode : int { kPrepMomentumSgd = 0, kPrepMomentumEma = 1, kPrepLoad = 2 };

// The Newton–Schulz iterate is kept as two bf16 planes, X = hi + lo, with
// lo = bf16(x - hi) the rounding residual: the tensor cores read hi only,
// while the a*X term of every update uses hi + lo (about 16 significant
// bits).  The lo plane of an iterate sits lo_off elements after its hi plane.
//
// Pass 1: momentum (+ look-ahead) or a plain load, writing the iterate X
// (hi and lo planes) into the workspace (wide orientation, padded) and
// per-block partial sums of X^2 (fp32, from the fp32 value before rounding).
struct PrepareArgs {
  int batch, rows, cols;
  int64_t row_stride;    // elements, of G, M and W
  int64_t batch_stride;  // elements, used when g_ptrs == nullptr
  int g_dtype;           // muon_dtype_t of the input (G, or X for newton_schulz_batched)
  const void* const* g_ptrs;  // device array, or nullptr
  const void* g_base;         // used when g_ptrs == nullptr
  float* const* m_ptrs;       // momentum buffers (modes 0 and 1)
  void* const* w_ptrs;        // only checked for alignment (may be nullptr)
  int mode;
  int nesterov;
  float mu;            // sgd: mu; ema: beta
  double ema_omb;      // ema: 1 - beta (exact, from the fp32 beta)
  float c_mom, c_grad;  // ema look-ahead: X = c_mom*buf + c_grad*g
  __nv_bfloat16* X;     // hi plane [batch][n_pad][m_pad]; lo plane at X + x_lo_off
  int64_t x_lo_off;
  int n_pad, m_pad;
  int tall;             // rows > cols: X holds the transpose
  int parts;            // blocks per matrix (partials per matrix)
  int parts_stride;     // partials between consecutive matrices (>= parts)
  float* partials;      // [batch][parts_stride]
  uint8_t* skip;        // [batch], set to 1 for a matrix with a misaligned pointer
  uint32_t* status;
};

// Groups of matrices that share one Newton–Schulz chain (same wide shape,
// either orientation) go through it as one batch of at most kMaxMerge
// segments.
constexpr int kMaxMerge = 4;

struct FinalizeArgs {
  int batch, parts_stride;
  int nseg;
  int seg_begin[kMaxMerge];   // first matrix of each segment
  int seg_parts[kMaxMerge];   // partials per matrix in each segment
  const float* partials;      // [batch][parts_stride]
  const uint8_t* skip;
  float* inv_s;  // [batch]: 1/||X||_F (0 for a zero or skipped matrix); 1 if !normalize
  int normalize;
  uint32_t* status;
  int* gp_ctr;  // [batch] Gram arrival counters of the fused Gram + polynomial launches, zeroed here
};

// Last pass: W <- W*decay - lr_scale*O'  (mode 0), or out <- O' (mode 1).
struct ApplyArgs {
  int batch, rows, cols;
  int64_t row_stride;        // W (mode 0)
  int mode;
  int w_dtype;               // W dtype (mode 0) / out dtype (mode 1)
  void* const* w_ptrs;       // mode 0
  void* out_base;            // mode 1: dense [batch][rows][cols]
  const uint8_t* wd_mask;    // mode 0, may be nullptr
  float decay_on;            // 1 - lr*wd
  float lr_scale;            // lr * scale
  const __nv_bfloat16* X;    // final iterate, hi plane [batch][n_pad][m_pad]
  int64_t x_lo_off;          // lo plane at X + x_lo_off
  int has_lo;                // 0: the final iterate is the hi plane alone
  int n_pad, m_pad, tall;
  int parts;
  const uint8_t* skip;
  const float* oscale;       // per-matrix factor on O' (zero-iteration schedules), or nullptr
};

// Last-iteration store fused into the update epilogue: mode 1 applies
// W <- W*(1 - lr*wd*mask) - lr*scale*O' (muon_step_batched), mode 2 writes O'
// into a dense output (newton_schulz_batched); mode 0 keeps the iterate in the
// workspace for a separate last pass.  One segment per group of the chain's
// batch (matrices seg[s].begin .. seg[s+1].begin - 1).
struct FinalSeg {
  int begin;                 // first matrix of the segment in the chain's batch
  int rows, cols;            // W / output shape in its own orientation
  int tall;                  // rows > cols: the wide element (i, j) is W[j][i]
  int dtype;                 // W dtype (mode 1) or output dtype (mode 2)
  void* const* w_ptrs;       // mode 1: device array of W pointers (segment-local index)
  int64_t w_ld;              // mode 1: W row stride (elements)
  void* out_base;            // mode 2: dense [segment batch][rows][cols]
  const uint8_t* wd_mask;    // mode 1: decay mask (segment-local), or nullptr (all on)
  float decay_on;            // 1 - lr*wd
  float lr_scale;            // lr * scale
};

struct FinalStore {
  int mode;
  int nseg;
  const uint8_t* skip;       // [chain batch]: matrices to leave untouched
  FinalSeg seg[kMaxMerge];
};

struct NsChainArgs {
  int batch, n_pad, m_pad;
  int n, m;             // unpadded sizes (algorithmic flop counts)
  __nv_bfloat16* X0;    // hi planes; lo planes at X0 + lo_off, X1 + lo_off
  __nv_bfloat16* X1;
  int64_t lo_off;
  __nv_bfloat16* A;
  __nv_bfloat16* B;
  float* pdiag;         // [batch][n_pad] fp32 residual of P's diagonal
  const float* inv_s;   // folded into the first iteration; nullptr = no normalisation
  const float* coeffs;  // host [iters][3]
  int iters;
  int x3;               // split-bf16 precision: S and P carry lo planes at +sq_lo_off
  int64_t sq_lo_off;
  FinalStore fin;       // fused into the last iteration when fin.mode != 0
  float* partial;       // split-K Gram slices, gram_ksplit(...) * batch * n_pad^2 fp32, or nullptr
  int* gp_ctr;          // [batch] counters for the fused Gram + polynomial launches (zero on
                        // entry), or nullptr
  int* gp_tick;         // [kGpMaxLaunches] ticket counters of those launches, then (at
  int* gp_log;          // gp_log) their ticket log; both zero on entry, or nullptr
  uint32_t* status;
  uint64_t timeout_ns;
};

// Kernel kinds for launch counting and event timing (prof.cu).
enum KernelKind : int {
  kKindPrepare = 0,
  kKindFinalize,
  kKindGram,
  kKindPoly,
  kKindUpdate,
  kKindApply,
  kKindTimeoutCheck,
  kKindAdamW,
  kKindGramPoly,
  kKindChain,
  kKindCount
};
void prof_begin(KernelKind k, cudaStream_t st);
void prof_end(KernelKind k, cudaStream_t st, double alg_flops, double alg_bytes);

int prepare_parts(int rows, int cols, int n_pad, int m_pad);
int apply_parts(int rows, int cols);

cudaError_t launch_prepare(const PrepareArgs& a, cudaStream_t st);
cudaError_t launch_finalize(const FinalizeArgs& a, cudaStream_t st);
cudaError_t launch_apply(const ApplyArgs& a, cudaStream_t st);
// ---- AdamW partition (adamw.cu) ----
constexpr int kAdamWMaxGroups = 16;  // groups per launch (kernel-parameter table)

struct AdamWGroupArgs {
  int count;                 // tensors in the group
  int64_t numel;             // elements per tensor
  int64_t chunks_per_tensor; // filled by launch_adamw
  int w_dtype, g_dtype;
  void* const* w_ptrs;       // device arrays [count] of device pointers
  const void* const* g_ptrs;
  float* const* m_ptrs;
  float* const* v_ptrs;
  const uint8_t* wd_mask;    // device [count] or nullptr (all on)
};

struct AdamWScalars {
  float lr, beta1, omb1, beta2, omb2, eps;
  float c1, c2;              // 1/(1 - beta1^t), 1/(1 - beta2^t)
  float decay_on;            // 1 - lr*wd
};

cudaError_t launch_adamw(AdamWGroupArgs* groups, int n_groups, const AdamWScalars& s,
                         uint32_t* flags, cudaStream_t st);

cudaError_t launch_wait_timeout_check(uint32_t* status, uint64_t timeout_ns, cudaStream_t st);
cudaError_t launch_occupy(int blocks, size_t smem_bytes, uint64_t ns, cudaStream_t st);

// Whether the chain's last iterate (after `iters` iterations) carries a lo plane.
bool ns_final_has_lo(int iters, bool x3);

// Whether the last iteration's update can write W (or the output) itself
// (NsChainArgs::fin); otherwise the iterate stays in the workspace for the
// separate last pass.
bool ns_final_fused(int iters, bool x3);

// K-slices of the Gram of a chain of padded wide shape n_pad x m_pad (1 =
// unsplit); a function of the shape alone, so that a matrix's result does not
// depend on the batch it is in.
int gram_ksplit(int n_pad, int m_pad, bool x3);

// Fused Gram + polynomial launches (bf16 precision, n_pad a multiple of 256)
// hand their work units out by tickets: per chain at most kGpMaxLaunches of
// them (later iterations launch the Gram and the polynomial separately), each
// with at most kGpMaxClusters CTA pairs.
constexpr int kGpMaxLaunches = 64;
constexpr int kGpMaxClusters = 128;

// Ints of workspace the ticket counters and log of a chain take (0 where the
// chain never fuses): kGpMaxLaunches counters, then kGpMaxClusters rows of
// (tickets of one launch + 2) entries.  Zeroed once per chain.
size_t gram_poly_log_ints(int batch, int n_pad, bool x3);

// Runs the whole chain; the final iterate is left in X0 if the number of
// iterations is even, else in X1.  Returns cudaErrorNotSupported when the
// driver entry point for tensor maps is missing.
cudaError_t run_ns_chain(const NsChainArgs& a, cudaStream_t st);

}  // namespace muon
