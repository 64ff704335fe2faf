/*
 * muon.h — C ABI of the GB300 (sm_103a) batched Muon optimizer step.
 *
 * The step, per 2-D weight matrix W (rows x cols), as stated by Algorithm 1 of
 * "Muon 优化器" (DeepSeek-V4 tech notes, §1 "Muon 一步在做什么"):
 *
 *   M_t  = mu * M_{t-1} + G_t                         momentum
 *   X    = mu * M_t + G_t                             Nesterov look-ahead
 *   O'   = HybridNewtonSchulz(X)                      §2 of the same page
 *   O    = O' * scale                                 spectral / unit_rms_norm
 *   W_t  = W_{t-1} * (1 - lr * wd * mask) - lr * O    decoupled weight decay
 *
 * HybridNewtonSchulz normalises X by its Frobenius norm (a zero X stays zero)
 * and repeats X <- a X + b (X X^T) X + c (X X^T)^2 X, eight times with
 * (3.4445, -4.7750, 2.0315) and twice with (2.0, -1.5, 0.5) ("Muon 优化器" §2).
 * The 'ema' momentum style and bias correction follow "RFC-0023: 对齐 MaxText
 * Muon 优化器实现与 Megatron-LM 完整行为" §方案 1; the per-tensor decay mask
 * §方案 2; the spectral scale sqrt(max(fan_in, fan_out)) * gamma §方案 3;
 * batching of same-shape matrices and split_head sub-matrices §方案 4 and
 * §背景; the 'unit_rms_norm' scale sqrt(fan_out / fan_in) comes from
 * "Scaling for MuP over Muon optimizer" (Megatron-LM PR #3715).
 *
 * Conventions shared by every entry point:
 *  - The caller owns all memory.  W and M are updated in place.  The library
 *    allocates nothing on the device: scratch is a caller workspace whose size
 *    the *_workspace_size queries return.  The workspace must be 256-byte
 *    aligned and must not be shared by calls that may overlap on the GPU.
 *  - Calls are stream-ordered and asynchronous.  Every argument the host can
 *    check is checked before anything is enqueued; on error nothing is
 *    enqueued and no memory is touched.
 *  - Conditions only the device can see (a non-finite Frobenius norm, a
 *    misaligned pointer inside a device pointer array, a device wait that
 *    ran out) set bits of a status word kept in the workspace; read it with
 *    muon_get_status.  Each call clears the word when it starts.
 *  - Matrices are row-major with unit column stride.  cols and row_stride
 *    must be multiples of 8 elements and every data pointer 16-byte aligned
 *    (MUON_ERR_MISALIGNED / MUON_ERR_UNSUPPORTED otherwise).  There is no
 *    slow path and no CPU fallback.
 *  - A stream argument is a cudaStream_t (NULL = the legacy default stream).
 */
#ifndef MUON_GB300_H_
#define MUON_GB300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* muon_stream_t; /* identical to cudaStream_t */

typedef enum {
  MUON_OK = 0,
  MUON_ERR_INVALID_ARG = 1,        /* NULL where a pointer is required, bad size, bad enum */
  MUON_ERR_MISALIGNED = 2,         /* pointer not 16 B (workspace: 256 B) aligned, stride not a multiple of 8 */
  MUON_ERR_UNSUPPORTED = 3,        /* valid request the library does not implement (e.g. TF32 NS, cols % 8) */
  MUON_ERR_WORKSPACE_TOO_SMALL = 4,
  MUON_ERR_CUDA = 5,               /* a CUDA runtime call failed (no device, launch failure, ...) */
  MUON_ERR_TIMEOUT = 6             /* returned by muon_get_status when a device wait ran out */
} muon_status_t;

/* Bits of the device status word (muon_get_status). */
#define MUON_FLAG_NONFINITE 0x1u   /* some matrix had a non-finite Frobenius norm */
#define MUON_FLAG_TIMEOUT 0x2u     /* a bounded device wait ran out; results are invalid */
#define MUON_FLAG_MISALIGNED 0x4u  /* a pointer in a device pointer array was not 16 B aligned;
                                      that matrix was left untouched */

typedef enum { MUON_BF16 = 0, MUON_F32 = 1 } muon_dtype_t;

/* 'sgd': buf = mu*buf + g, look-ahead mu*buf + g (no bias correction).
 * 'ema': buf = mu*buf + (1-mu)*g, look-ahead mu*bc(buf,t+1) + (1-mu)*bc(g,t)
 *        with bc(x,k) = x/(1-mu^k).  ("RFC-0023" §方案 1) */
typedef enum { MUON_NESTEROV_SGD = 0, MUON_NESTEROV_EMA = 1 } muon_nesterov_style_t;

/* spectral: sqrt(max(rows, cols)) * gamma  ("Muon 优化器" Algorithm 1)
 * unit_rms_norm: sqrt(fan_out / fan_in), no gamma ("Scaling for MuP over Muon optimizer")
 * none: 1 */
typedef enum {
  MUON_SCALE_SPECTRAL = 0,
  MUON_SCALE_UNIT_RMS_NORM = 1,
  MUON_SCALE_NONE = 2
} muon_scale_mode_t;

/* Precision of the Newton–Schulz chain (the pages fix none; "RFC-0023" §风险
 * contrasts the float64 reference with bf16).  Every kind uses bf16
 * tensor-core operands with fp32 accumulation and fp32 epilogues.
 *  MUON_NS_BF16:   X X^T and the polynomial stored in bf16 (the polynomial's
 *                  diagonal keeps an fp32 residual), the iterate as bf16 plus
 *                  its bf16 rounding residual in the first iterations;
 *                  relative error about 5e-3 against float64.
 *  MUON_NS_BF16X3: split-bf16: X, X X^T and the polynomial all stored as
 *                  hi + lo bf16 planes (about 16 significant bits), every
 *                  product the three-term sum A_hi B_hi + A_hi B_lo + A_lo B_hi;
 *                  relative error about 1e-5 for three times the tensor-core
 *                  work and twice the workspace for X X^T and the polynomial.
 *  MUON_NS_TF32:   reserved (returns MUON_ERR_UNSUPPORTED): one-pass TF32
 *                  products, emulated, miss a 1e-3 relative bound on
 *                  gradients with a low-rank spike. */
typedef enum { MUON_NS_BF16 = 0, MUON_NS_TF32 = 1, MUON_NS_BF16X3 = 2 } muon_ns_precision_t;

/* `steps` iterations of X <- a X + b (X X^T) X + c (X X^T)^2 X. */
typedef struct {
  int steps;
  float a, b, c;
} muon_ns_stage_t;

/* stages: host array of n_stages entries (read during the call only).
 * normalize: 1 = divide by the Frobenius norm first (the page's behaviour),
 *            0 = iterate the input as is.
 * merge_groups (muon_step_batched / muon_step_workspace_size only):
 *            1 = groups whose matrices have the same wide shape (min and max
 *            of rows, cols), in either orientation, share one Newton–Schulz
 *            chain of up to 4 groups (a 14336 x 4096 weight group and a
 *            4096 x 14336 one run as one batch: fewer launches, fuller
 *            waves; results are bit-identical to unmerged, the workspace is
 *            sized for the merged batches); 0 = one chain per group. */
typedef struct {
  const muon_ns_stage_t* stages;
  int n_stages;
  int normalize;
  muon_ns_precision_t prec;
  int merge_groups;
} muon_ns_schedule_t;

/* A matrix view in elements.  rows x cols, row-major, unit column stride.
 * row_stride >= cols, multiple of 8.  batch_stride: elements between
 * consecutive matrices (newton_schulz_batched only; ignored by groups, which
 * carry one pointer per matrix).  fan_out_axis: 0 = rows hold fan_out
 * (PyTorch [out, in]); 1 = cols hold fan_out (MaxText [in, out], and the
 * split_head sub-matrices [embed, head_dim]); used by unit_rms_norm only. */
typedef struct {
  int rows, cols;
  int64_t row_stride;
  int64_t batch_stride;
  int fan_out_axis;
} muon_view_t;

/* One batched group of same-shape matrices ("RFC-0023" §方案 4).
 * w_ptrs, g_ptrs, m_ptrs: DEVICE arrays of `batch` DEVICE pointers.  Matrix i
 * of the group is W = w_ptrs[i], G = g_ptrs[i], M = m_ptrs[i], all with
 * `view` (same row_stride).  W is w_dtype, G is g_dtype, M is fp32.
 * A split_head weight [embed, heads*head_dim] is one group of `heads`
 * matrices embed x head_dim with row_stride = heads*head_dim and pointers
 * base + h*head_dim (the heads form the batch; fan_out = head_dim).
 * wd_mask: DEVICE array [batch] of 0/1 (1 = apply weight decay); NULL = all on. */
typedef struct {
  int batch;
  muon_view_t view;
  muon_dtype_t w_dtype, g_dtype;
  void* const* w_ptrs;
  const void* const* g_ptrs;
  float* const* m_ptrs;
  const uint8_t* wd_mask;
} muon_group_t;

/* mu: momentum coefficient (beta for 'ema').  nesterov: 1 = look-ahead
 * (default), 0 = orthogonalise the (bias-corrected, for 'ema') buffer.
 * t: steps taken including this one (>= 1), used by 'ema' only.
 * Defaults from "Muon 优化器" §3: mu 0.95, gamma 0.18, weight_decay 0.1;
 * lr 2.7e-4 in §2's routine. */
typedef struct {
  float mu;
  int nesterov;
  muon_nesterov_style_t style;
  int64_t t;
  muon_scale_mode_t scale_mode;
  float gamma, lr, weight_decay;
} muon_hparams_t;

/* Grouping key of one tensor: tensors group together iff every field is equal. */
typedef struct {
  int rows, cols;
  int64_t row_stride;
  muon_dtype_t w_dtype, g_dtype;
  int fan_out_axis;
} muon_tensor_desc_t;

/* Fill `out` with the hybrid 8 x (3.4445, -4.7750, 2.0315) + 2 x (2.0, -1.5, 0.5)
 * schedule of "Muon 优化器" §2 (normalize = 1, bf16).  The stage array is static. */
muon_status_t muon_ns_hybrid_schedule(muon_ns_schedule_t* out);

/* Host only, pure.  Assign each of the n tensors a group: tensors with equal
 * descriptors share a group, groups are numbered in order of first
 * appearance, each group's members are taken in tensor order and cut into
 * chunks of at most max_batch (0 = no limit), each chunk its own group
 * ("RFC-0023" §方案 4, chunking by the batch-update size).
 * group_of_tensor: host array [n] (output).  n_groups: output. */
muon_status_t muon_group_by_shape(const muon_tensor_desc_t* tensors, int n, int max_batch,
                                  int* group_of_tensor, int* n_groups);

/* Bytes of workspace muon_step_batched needs for these groups and schedule
 * (NULL schedule = hybrid).  Host only. */
muon_status_t muon_step_workspace_size(const muon_group_t* groups, int n_groups,
                                       const muon_ns_schedule_t* schedule, size_t* bytes);

/* One Muon step for every matrix of every group, in group order, on `stream`.
 * groups: host array [n_groups].  hparams: host.  schedule: host, NULL = hybrid.
 * workspace: device, >= muon_step_workspace_size bytes, 256 B aligned.
 * Updates M and W in place.  Returns before the GPU work completes. */
muon_status_t muon_step_batched(const muon_group_t* groups, int n_groups,
                                const muon_hparams_t* hparams,
                                const muon_ns_schedule_t* schedule, void* workspace,
                                size_t workspace_bytes, muon_stream_t stream);

/* Bytes of workspace newton_schulz_batched needs.  Host only. */
muon_status_t newton_schulz_workspace_size(const muon_view_t* view, int batch,
                                           const muon_ns_schedule_t* schedule, size_t* bytes);

/* O' = HybridNewtonSchulz(X) for `batch` matrices ("Muon 优化器" §2).
 * x: device, matrix i at x + i*view->batch_stride elements, dtype xdt, view.
 * out: device, dense [batch, rows, cols] row-major of dtype odt (written, in
 * the input's orientation).  x and out must not overlap.  The chain runs in
 * the precision schedule->prec names; the last iterate (value + residual) is
 * rounded to odt. */
muon_status_t newton_schulz_batched(const void* x, muon_dtype_t xdt, const muon_view_t* view,
                                    int batch, void* out, muon_dtype_t odt,
                                    const muon_ns_schedule_t* schedule, void* workspace,
                                    size_t workspace_bytes, muon_stream_t stream);

/* Synchronise `stream`, then read the status word of `workspace` into
 * *device_flags (MUON_FLAG_*).  Returns MUON_ERR_TIMEOUT if the timeout bit
 * is set, MUON_ERR_CUDA if the stream reported an error, else MUON_OK. */
muon_status_t muon_get_status(const void* workspace, muon_stream_t stream,
                              uint32_t* device_flags);

/* Upper bound, in nanoseconds, for every bounded wait inside the library's
 * kernels (default 2e9).  A wait that runs out sets MUON_FLAG_TIMEOUT and the
 * kernel returns early.  Process-wide; takes effect for later launches. */
muon_status_t muon_set_wait_timeout_ns(uint64_t ns);

/* Failure-path check: launches one kernel whose bounded wait is never
 * satisfied (an mbarrier nobody arrives on), with `timeout_ns` as its limit,
 * so that the kernel gives up, sets MUON_FLAG_TIMEOUT in the workspace's
 * status word and returns.  Used to test the timeout path without hanging a
 * GPU.  workspace: >= 256 bytes, 256 B aligned. */
muon_status_t muon_check_wait_timeout(void* workspace, size_t workspace_bytes,
                                      uint64_t timeout_ns, muon_stream_t stream);

/* Co-scheduling check: launches `blocks` blocks of one warp, each holding
 * `smem_bytes` of dynamic shared memory (at most 227 KiB), that wait `ns`
 * nanoseconds by the GPU's global timer (at most 1 s) and exit.  Run on one
 * stream while a step runs on another, it keeps most SMs from the step's
 * kernels for a bounded time, the way concurrent work (a communication
 * kernel, another model's step) does in a shared job; used to test that the
 * step still completes within its bounded waits.  The pages have no
 * counterpart to it. */
muon_status_t muon_occupy_sms(int blocks, size_t smem_bytes, uint64_t ns, muon_stream_t stream);

/* Allocation-free variant of newton_schulz_batched.  The pages have no
 * counterpart to it; it exists for callers that cannot obtain a workspace
 * from cudaMalloc: code inside a framework whose caching allocator owns all
 * device memory (a raw cudaMalloc there fragments memory and escapes the
 * framework's accounting), and latency-critical loops that cannot pay the
 * implicit device synchronisation cudaMalloc / cudaFree may cause.
 *
 * Same arguments and results as newton_schulz_batched, without the
 * workspace: the scratch is a 32 MiB array inside the library's device image
 * (held by every GPU the library is loaded on until the process exits).  A
 * call whose workspace need (newton_schulz_workspace_size) exceeds 32 MiB
 * returns MUON_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.  The
 * call allocates no device memory.
 *
 * The first call in each CUDA context looks up the array's device address
 * in that context (cudaGetSymbolAddress, with the device current; kept for
 * later calls in the same context, keyed by the context's unique id, so a
 * context created after cudaDeviceReset gets a fresh lookup), so make that
 * first call before any stream capture.  All calls share the one array: each
 * call clears what must start at zero (status word, skip flags, hand-over
 * counters) and rewrites everything else it reads, so the previous call's
 * contents do not matter, but calls that may overlap on the GPU (different
 * streams, several host threads) race on it and must be serialised by the
 * caller.
 *
 * device_flags: NULL, or a caller-owned 4-byte-aligned device word that
 * receives this call's MUON_FLAG_* bits (stream-ordered copy at the end). */
muon_status_t newton_schulz_batched_noalloc(const void* x, muon_dtype_t xdt,
                                            const muon_view_t* view, int batch, void* out,
                                            muon_dtype_t odt, const muon_ns_schedule_t* schedule,
                                            uint32_t* device_flags, muon_stream_t stream);

/* ---- AdamW partition ------------------------------------------------------
 * The parameters that stay on AdamW next to Muon: embeddings, the output
 * head, norm scales and other non-matrix tensors ("Muon 优化器" §3, whose V4
 * settings are beta1 0.9, beta2 0.95, eps 1e-20, weight decay 0.1), with the
 * per-tensor decay mask of "RFC-0023" §方案 2.  Per element, in fp32:
 *
 *   m <- beta1*m + (1 - beta1)*g
 *   v <- beta2*v + (1 - beta2)*g^2
 *   u  = (m / (1 - beta1^t)) / (sqrt(v / (1 - beta2^t)) + eps)
 *   W <- W*(1 - lr*wd*mask) - lr*u
 *
 * (the pages name AdamW without writing it out: this is Adam with bias
 * correction and decoupled decay, eps outside the square root, the form of
 * optax's adamw and PyTorch's AdamW). */

/* `count` contiguous tensors of `numel` elements each (any shape).
 * w_ptrs, g_ptrs, m_ptrs, v_ptrs: DEVICE arrays of `count` DEVICE pointers,
 * each 16-byte aligned; W is w_dtype, G is g_dtype, m and v (first and second
 * moments) are fp32; W, m and v are updated in place.  numel need not be a
 * multiple of anything.  wd_mask: DEVICE [count] of 0/1 (1 = decay), NULL =
 * all on. */
typedef struct {
  int count;
  int64_t numel;
  muon_dtype_t w_dtype, g_dtype;
  void* const* w_ptrs;
  const void* const* g_ptrs;
  float* const* m_ptrs;
  float* const* v_ptrs;
  const uint8_t* wd_mask;
} muon_adamw_group_t;

/* t: steps taken including this one (>= 1).  0 <= beta1, beta2 < 1; eps >= 0. */
typedef struct {
  float lr, beta1, beta2, eps, weight_decay;
  int64_t t;
} muon_adamw_hparams_t;

/* One AdamW step for every tensor of every group, on `stream`, in one
 * kernel launch per 16 groups.  groups: host array [n_groups]; hparams: host.
 * Needs no workspace.  device_flags: NULL, or a caller-owned device word
 * (4-byte aligned) into which the kernel ORs MUON_FLAG_MISALIGNED when a
 * pointer in a pointer array is not 16-byte aligned (that tensor is left
 * untouched); the caller clears it.  Returns before the GPU work completes. */
muon_status_t muon_adamw_step(const muon_adamw_group_t* groups, int n_groups,
                              const muon_adamw_hparams_t* hparams, uint32_t* device_flags,
                              muon_stream_t stream);

/* Per-kernel statistics since the last muon_profile_reset.  Launches are
 * always counted.  With profiling on, the library records a CUDA event pair
 * on the launching stream around every kernel launch and total_ms sums their
 * elapsed times.  alg_flops / alg_bytes sum the algorithmic work of the
 * launches: Newton–Schulz GEMM flops counted on the unpadded shapes with the
 * symmetric Gram and polynomial products at half their dense count, and the
 * HBM bytes the elementwise passes must move. */
typedef struct {
  char name[32];
  uint64_t launches;
  double total_ms;
  double alg_flops;
  double alg_bytes;
} muon_kernel_stats_t;

/* Turn event timing of every launch on (1) or off (0).  Process-wide. */
muon_status_t muon_profile_enable(int on);

/* Clear all counters and timings (waits for pending events first). */
muon_status_t muon_profile_reset(void);

/* Copy up to `capacity` entries into `out` (host) and the number of kernel
 * kinds into *n.  Synchronises the events still pending. */
muon_status_t muon_profile_query(muon_kernel_stats_t* out, int capacity, int* n);

/* Static, human-readable name of a status code. */
const char* muon_status_string(muon_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* MUON_GB300_H_ */
