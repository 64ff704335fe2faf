// Newton–Schulz chain on 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// One iteration of "Muon 优化器" (DeepSeek-V4 tech notes) §2,
//     X <- a X + b (X X^T) X + c (X X^T)^2 X,
// runs as three batched GEMMs on the wide, zero-padded iterate X (n x m):
//
//   Gram    S = X X^T                      n x n, K = m  (symmetric: upper tiles + mirror)
//   Poly    P = b S + c S S + (a - 1) I    n x n, K = n  (symmetric: upper tiles + mirror)
//   Update  X' = X + P X                   n x m, K = n
//
// which is  a X + b S X + c S^2 X  exactly.  When c == 0 the Gram epilogue
// writes P = b S + (a - 1) I directly and the Poly GEMM is skipped.  P is
// stored in bf16 except for the rounding residual of its diagonal, kept in
// fp32 and added back in the update (the shifted diagonal is large and its
// bf16 rounding would otherwise swamp b S_ii when a is small).  The
// Frobenius normalisation is folded into the first iteration: with
// s = ||X||_F, S_0 = (X X^T)/s^2 and X_1 = (X + P_0 X)/s.
//
// Kernel shapes (one persistent CTA per SM).  Where tile rows come in pairs
// and BN = 256, k_ns_gemm2 runs each 256 x 256 tile on a CTA pair with
// pair-wide tcgen05 MMAs (cta_group::2, 10 warps); otherwise k_ns_gemm runs
// 128 x BN tiles per CTA (6 warps), and a Gram of a single 128 x 128 tile
// over a long K is split into K-slices whose fp32 sums k_gram_reduce adds in
// a fixed order.
// Roles:
//   warp 0      one thread issues TMA loads of A and B k-blocks into a
//               multi-stage shared-memory ring (128-byte swizzle);
//   warp 1      allocates TMEM and one thread issues tcgen05.mma
//               (bf16 -> fp32) into one of two TMEM accumulators,
//               committing to mbarriers;
//   the rest    epilogue (4 warps, or 8 in k_ns_gemm2: two per 32-lane TMEM
//               quarter): tcgen05.ld, fp32 epilogue math, 256-bit residual
//               loads, and bf16 stores -- in k_ns_gemm2 through per-warp
//               staging boxes and TMA stores, the transposed copy of
//               off-diagonal symmetric tiles included.
// The two accumulators let the epilogue of tile i overlap the MMAs of tile i+1.
// In the bf16 precision, where tile rows pair up, k_ns_gram_poly runs an
// iteration's Gram and polynomial as one launch (per-matrix hand-over through
// arrival counters) and k_ns_gemm2 the update.  Consecutive launches walk the
// batch in opposite directions, so that each starts on the matrices its
// predecessor wrote last; the update's tiles go in column bands.
//
// Precision.  Operands are bf16 with fp32 accumulation; S and P are stored
// as bf16; the iterate is stored as two bf16 planes X = hi + lo with
// lo = bf16(x - hi) for the first kLoIters iterations and as hi alone after
// that.  The exact X term of the update reads hi + lo; the product P X
// reads hi only, and the epilogue adds back the shift's share of the
// dropped P lo, (a - 1) lo, exactly in fp32.
// Why: when a few singular directions dominate the entries (a low-rank
// spike in the gradient), rounding X to bf16 puts noise the size of the
// large entries into the small directions, which the fast stage multiplies
// by a ~ 3.4 per step, so both the X term and, while those directions are
// still small, the product need the residual.  Writing the update as
// X + P X with the a - 1 shift inside P keeps the product's coefficient small
// on directions that have converged (a + b + c - 1: -0.30 in the fast stage,
// 0 in the stable stage), so dropping lo from the product costs little
// there; on the directions that are still small P is (a - 1) I plus terms
// of order sigma^2, so (a - 1) lo is nearly all of P lo, and it costs no
// tensor work.  (Written as a X + (b S + c S^2) X, converged directions would
// cancel 3.44 X against -2.74 X and amplify the dropped residual about
// ninefold.)  Reading lo in the product instead (a second K-loop over the lo
// plane) doubles the first updates' tensor work for a result no closer to
// float64 on the spiky, row-scaled and Gaussian sets (worst relative error
// 7.7e-3 against 5.5e-3 with the shift share; 4.3e-3 against 5.0e-3 on the
// Student-t set).
//
// Split-bf16 precision (kEpiX3, MUON_NS_BF16X3): S, P and X are all stored
// as hi + lo planes and every GEMM runs one K-loop over three plane pairs,
// A_hi B_hi + A_hi B_lo + A_lo B_hi, which keeps about 16 significant bits
// throughout.  With that precision the shift buys nothing and costs digits
// when a is small (X + (S^2 - I) X cancels for a = 0), so the update is
// evaluated as written, X' = a X + (b S + c S^2) X.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace muon {
namespace {

constexpr int kBM = 128;  // tile rows (TMEM lanes)
constexpr int kResidualIters = 0;  // iterations whose product also reads the lo plane
constexpr int kLoIters = 4;        // iterations that read the lo plane (the first kLoIters-1 write it)
#ifndef MUON_PDL
#define MUON_PDL 1
#endif
// Launch the GEMMs as programmatic dependents of the previous kernel: their
// set-up (barriers, TMEM allocation, descriptor prefetch) overlaps its tail,
// and griddepcontrol.wait holds every dependent read until it has finished.
constexpr bool kUsePdl = MUON_PDL != 0;
#ifndef MUON_TWO_SM
#define MUON_TWO_SM 1
#endif
constexpr bool kUseTwoSm = MUON_TWO_SM != 0;  // pair-wide MMA (k_ns_gemm2) where BN = 256
#ifndef MUON_FUSE_GRAM_POLY
#define MUON_FUSE_GRAM_POLY 1
#endif
// Gram and polynomial of an iteration in one launch (k_ns_gram_poly) where possible.
constexpr bool kFuseGramPoly = MUON_FUSE_GRAM_POLY != 0;
#ifndef MUON_CLUSTER_CHAIN
#define MUON_CLUSTER_CHAIN 1
#endif
// Iterates of one 128-row tile run the whole chain in one launch
// (k_ns_cluster_chain) where the GPU can hold its clusters.
constexpr bool kUseClusterChain = MUON_CLUSTER_CHAIN != 0;
constexpr int kBK = 64;   // k-block: 64 bf16 = one 128-byte swizzle row
constexpr int kBandTiles = 8;  // update (non-symmetric, paired) tiles: column band width
constexpr int kEpiWarps = 4;
constexpr int kGemmThreads = 64 + 32 * kEpiWarps;  // producer, MMA, 4 epilogue warps

// kEpiFinal: the update of the last iteration, whose epilogue writes W (or
// the output) instead of the iterate; it never carries a lo plane.
// kEpiX3 (or-ed into Gram / Poly / Update): the split-bf16 precision, in
// which S, P and X are all stored as hi + lo planes and every product is the
// three-term sum A_hi B_hi + A_hi B_lo + A_lo B_hi.
// kEpiTall (or-ed into kEpiFinal): some matrix of the chain keeps W (or its
// output) in the tall orientation, so the epilogue carries the turn-around
// path and its shared-memory buffers; without it the kernel serves wide W only.
enum Epi : int { kEpiGram = 0, kEpiPoly = 1, kEpiUpdate = 2, kEpiFinal = 3, kEpiX3 = 4, kEpiTall = 8 };
__host__ __device__ constexpr int epi_kind(int e) { return e & 3; }
__host__ __device__ constexpr bool epi_x3(int e) { return (e & kEpiX3) != 0; }
__host__ __device__ constexpr bool epi_tall(int e) { return (e & kEpiTall) != 0; }

template <int BN>
struct Cfg {
  static constexpr int kStages = (BN == 256) ? 4 : 6;
  static constexpr uint32_t kABytes = kBM * kBK * 2;
  static constexpr uint32_t kBBytes = BN * kBK * 2;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr uint32_t kTmemCols = 2 * BN;
  static constexpr size_t kSmemBytes = kStages * kStageBytes + 1024 /*align*/ + 256 /*barriers*/;
};

struct GemmParams {
  int M, N, K;
  int tiles_m, tiles_n, tiles_per_matrix, total_tiles;
  __nv_bfloat16* out;
  int64_t out_ld, out_bstride;
  const __nv_bfloat16* aux;
  int64_t aux_ld, aux_bstride;
  int64_t lo_off;  // lo planes of aux and out at +lo_off elements
  int lo_in, lo_out;  // update (any kind with kEpiX3): read aux's lo plane / write out's lo plane
  float ca, cb, cc;
  float cd;         // added on the diagonal (Gram when c == 0, Poly): a - 1
  float clo;        // update whose product reads X hi only: coefficient of the
                    // lo plane added in the epilogue (a - 1, the shift's share of P lo)
  int kplanes;      // K-loop over 1..3 operand planes; plane p reads A's lo plane
  int a_lo_mask;    // (tmA2) if bit p of a_lo_mask is set, else its hi plane
  int b_lo_mask;    // (tmA), and likewise B from tmB2 / tmB
  float* pdiag;     // Gram (c == 0) / Poly: fp32 rounding residual of P's diagonal, [batch][n]
  const float* pdiag_in;  // update: that residual, added back as d_row * X
  int64_t pdiag_bstride;
  const float* mscale;
  uint32_t* status;
  uint64_t timeout_ns;
  FinalStore fin;   // update, last iteration: fused scale / decay / store
  int reverse;      // walk the units from the last matrix to the first
  int ksplit;       // Gram split into ksplit K-slices (1-CTA kernel): unit t is slice
                    // t % ksplit of tile t / ksplit; 0 or 1 = whole K
  float* partial;   // split-K: fp32 [ksplit][batch][n][n] raw accumulators
};

// Tile t -> (matrix, tile row, tile column).  For symmetric outputs only the
// tiles on or above the diagonal of BN x BN super-blocks are enumerated.
template <int BN, bool SYM>
__device__ __forceinline__ void decode_tile(const GemmParams& p, int t, int& b, int& tm, int& tn) {
  b = t / p.tiles_per_matrix;
  int l = t - b * p.tiles_per_matrix;
  if (!SYM) {
    tm = l / p.tiles_n;
    tn = l - tm * p.tiles_n;
    return;
  }
  constexpr int R = BN / kBM;
  const int S = p.tiles_n;
  tn = 0;
  for (tm = 0; tm < p.tiles_m; ++tm) {
    const int cnt = S - tm / R;
    if (l < cnt) {
      tn = tm / R + l;
      return;
    }
    l -= cnt;
  }
}

// Work unit t -> (matrix, tile row, tile column).  With PAIR the unit is a
// pair of vertically adjacent tiles (tm = 2 pm + cluster rank) sharing the
// tile column; for symmetric outputs (BN = 256) a pair is one upper
// super-block row segment (pm = super-row).
template <int BN, bool SYM, bool PAIR>
__device__ __forceinline__ void decode_unit(const GemmParams& p, int t, uint32_t rank, int& b,
                                            int& tm, int& tn) {
  if (p.reverse) t = p.total_tiles - 1 - t;
  if (!PAIR) {
    decode_tile<BN, SYM>(p, t, b, tm, tn);
    return;
  }
  b = t / p.tiles_per_matrix;
  int l = t - b * p.tiles_per_matrix;
  int pm = 0;
  tn = 0;
  if (!SYM) {
    // Column bands of kBandTiles tile columns, tile rows inside a band: the
    // band's B columns (n x 2048 of X) and A (P, n x n) stay in L2 while
    // every tile row of the band reads them.  (Row-major over all tiles
    // streamed a 4096 x 14336 X once per tile row: 5x its size from DRAM.)
    const int rows = p.tiles_m >> 1;
    const int full = rows * kBandTiles;
    const int band = l / full;
    const int in = l - band * full;
    const int width = min(kBandTiles, p.tiles_n - band * kBandTiles);
    pm = in / width;
    tn = band * kBandTiles + (in - pm * width);
  } else {
    const int S = p.tiles_n;
    for (int sr = 0; sr < S; ++sr) {
      const int cnt = S - sr;
      if (l < cnt) {
        pm = sr;
        tn = sr + l;
        break;
      }
      l -= cnt;
    }
  }
  tm = 2 * pm + static_cast<int>(rank);
}

// A drain wait: ignores the abort flag, still bounded.
__device__ __forceinline__ void mbar_wait_drain(uint64_t* bar, uint32_t parity, uint32_t* status,
                                                uint64_t timeout_ns) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (global_timer_ns() - t0 > timeout_ns) {
      atomicOr(status, kFlagTimeout);
      return;
    }
  }
}

// 32 bf16 of one row (64 bytes, 64-byte aligned in the workspace) as two
// full-sector loads.
__device__ __forceinline__ void load_raw4(const __nv_bfloat16* src, uint4 (&u)[4]) {
  // from L2: in a fused Gram + polynomial launch another CTA wrote these lines
  ld_global_cg_v8(src, u[0], u[1]);
  ld_global_cg_v8(src + 16, u[2], u[3]);
}

__device__ __forceinline__ void unpack_raw4(const uint4 (&u)[4], float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u[q]);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(h[k]);
      v[q * 8 + 2 * k] = f.x;
      v[q * 8 + 2 * k + 1] = f.y;
    }
  }
}

// ---- last iteration: W <- W*decay - lr_scale*O' fused into the update ---------
// ("Muon 优化器" Algorithm 1, last line; the mask is RFC-0023 §方案 2).  The
// epilogue holds O' in fp32 for 32 consecutive wide-orientation elements
// (row, col0 .. col0+31) per lane.  W is read before the accumulator is
// ready: the tile's W lines are prefetched into L2 when the tile starts and
// each chunk's W is loaded into registers one chunk ahead, so the
// read-modify-write adds no HBM latency to the epilogue.  Padding rows and
// columns and skipped matrices are left alone.
struct FinTile {
  void* base;        // W (mode 1) or the matrix's dense output (mode 2); nullptr = skip
  int64_t ld;
  float decay, lr_scale;
  int n_real, m_real;
  bool tall, bf;     // W[j][i] holds wide element (i, j); bf16 storage
  bool v8;           // wide rows 32-byte aligned: 256-bit accesses
};

// Matrix b of the chain's batch: its segment's W (or output) and parameters.
__device__ __forceinline__ FinTile fin_tile(const FinalStore& f, int b) {
  int s = 0;
  while (s + 1 < f.nseg && b >= f.seg[s + 1].begin) ++s;
  const FinalSeg& g = f.seg[s];
  const int bl = b - g.begin;
  FinTile t;
  t.tall = g.tall != 0;
  t.bf = (g.dtype == MUON_BF16);
  t.n_real = t.tall ? g.cols : g.rows;
  t.m_real = t.tall ? g.rows : g.cols;
  const bool muon = (f.mode == 1);
  t.base = f.skip[b] ? nullptr
           : muon    ? g.w_ptrs[bl]
                     : static_cast<void*>(static_cast<char*>(g.out_base) +
                                          static_cast<int64_t>(bl) * g.rows * g.cols * (t.bf ? 2 : 4));
  t.ld = muon ? g.w_ld : g.cols;
  const int esz = t.bf ? 2 : 4;
  t.v8 = !t.tall && t.base != nullptr && (reinterpret_cast<uintptr_t>(t.base) & 31u) == 0 &&
         ((t.ld * esz) & 31) == 0;
  t.decay = (muon && (g.wd_mask == nullptr || g.wd_mask[bl])) ? g.decay_on : 1.f;
  t.lr_scale = g.lr_scale;
  return t;
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// L2 prefetch of the W the calling lane's chunks [c0, c0 + nch) will read.
__device__ __forceinline__ void fin_prefetch(const FinalStore& f, const FinTile& t, int row,
                                             int row0, int col_begin, int ncols, int lane) {
  if (t.base == nullptr || f.mode != 1) return;
  const int esz = t.bf ? 2 : 4;
  const char* base = static_cast<const char*>(t.base);
  if (!t.tall) {
    if (row >= t.n_real) return;
    const int c_end = min(col_begin + ncols, t.m_real);
    for (int j = col_begin; j < c_end; j += 128 / esz)
      prefetch_l2(base + (static_cast<int64_t>(row) * t.ld + j) * esz);
  } else {
    if (row0 >= t.n_real) return;
    // W[j][row0 .. row0+31]: one 64- or 128-byte segment per W row j
    for (int j = col_begin + lane; j < col_begin + ncols; j += 32)
      if (j < t.m_real) prefetch_l2(base + (static_cast<int64_t>(j) * t.ld + row0) * esz);
  }
}

// W of one chunk into registers (raw bits; bf16 wide packs two per word).
template <bool kTall>
__device__ __forceinline__ void fin_load(const FinalStore& f, const FinTile& t, int row, int row0,
                                         int col0, uint32_t (&w)[32]) {
  if (t.base == nullptr || f.mode != 1) return;
  const bool bf = t.bf;
  if (!kTall || !t.tall) {
    if (row >= t.n_real) return;
    // whole 32-byte sectors where the row allows (m_real is a multiple of 8)
    const int64_t roff = static_cast<int64_t>(row) * t.ld;
    if (t.v8 && col0 + 32 <= t.m_real) {
      if (bf) {
        const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(t.base) + roff + col0;
        uint4 a, b, c, d;
        ld_global_v8(src, a, b);
        ld_global_v8(src + 16, c, d);
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
        w[8] = c.x; w[9] = c.y; w[10] = c.z; w[11] = c.w; w[12] = d.x; w[13] = d.y; w[14] = d.z; w[15] = d.w;
      } else {
        const float* src = static_cast<const float*>(t.base) + roff + col0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint4 a, b;
          ld_global_v8(src + 8 * k, a, b);
          w[8 * k] = a.x; w[8 * k + 1] = a.y; w[8 * k + 2] = a.z; w[8 * k + 3] = a.w;
          w[8 * k + 4] = b.x; w[8 * k + 5] = b.y; w[8 * k + 6] = b.z; w[8 * k + 7] = b.w;
        }
      }
      return;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int j = col0 + 8 * k;
      if (j >= t.m_real) continue;  // m_real is a multiple of 8
      const int64_t off = roff + j;
      if (bf) {
        const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(t.base) + off);
        w[4 * k] = u.x; w[4 * k + 1] = u.y; w[4 * k + 2] = u.z; w[4 * k + 3] = u.w;
      } else {
        const uint4* q = reinterpret_cast<const uint4*>(static_cast<const float*>(t.base) + off);
        const uint4 u0 = q[0], u1 = q[1];
        w[8 * k] = u0.x; w[8 * k + 1] = u0.y; w[8 * k + 2] = u0.z; w[8 * k + 3] = u0.w;
        w[8 * k + 4] = u1.x; w[8 * k + 5] = u1.y; w[8 * k + 6] = u1.z; w[8 * k + 7] = u1.w;
      }
    }
  } else {
    // turned-around layout (see fin_store): half h of the chunk gives this
    // lane 16 consecutive elements of W row col0 + 16h + lane / 2, from
    // wide row row0 + 16 (lane & 1); bf16 packs two per word (words 8h..8h+7),
    // fp32 one (words 16h..16h+15)
    const int lane = row - row0;
    const int i0 = row0 + 16 * (lane & 1);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int j = col0 + 16 * h + (lane >> 1);
      if (j >= t.m_real) continue;
      const int64_t off = static_cast<int64_t>(j) * t.ld + i0;
      if (i0 + 16 <= t.n_real) {
        if (bf) {
          const uint4* q = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(t.base) + off);
          const uint4 a = q[0], b = q[1];
          w[8 * h] = a.x; w[8 * h + 1] = a.y; w[8 * h + 2] = a.z; w[8 * h + 3] = a.w;
          w[8 * h + 4] = b.x; w[8 * h + 5] = b.y; w[8 * h + 6] = b.z; w[8 * h + 7] = b.w;
        } else {
          const uint4* q = reinterpret_cast<const uint4*>(static_cast<const float*>(t.base) + off);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint4 a = q[k];
            w[16 * h + 4 * k] = a.x; w[16 * h + 4 * k + 1] = a.y;
            w[16 * h + 4 * k + 2] = a.z; w[16 * h + 4 * k + 3] = a.w;
          }
        }
      } else {
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          if (i0 + k >= t.n_real) continue;
          if (bf) {
            const uint32_t hb = *reinterpret_cast<const unsigned short*>(
                static_cast<const __nv_bfloat16*>(t.base) + off + k);
            w[8 * h + (k >> 1)] = (k & 1) ? ((w[8 * h + (k >> 1)] & 0xffffu) | (hb << 16))
                                          : ((w[8 * h + (k >> 1)] & 0xffff0000u) | hb);
          } else {
            w[16 * h + k] = *reinterpret_cast<const uint32_t*>(static_cast<const float*>(t.base) + off + k);
          }
        }
      }
    }
  }
}

// Element e of a lane's W words (bf16 packed two per word, or fp32).
__device__ __forceinline__ float fin_w(bool bf, const uint32_t (&w)[32], int e) {
  if (!bf) return __uint_as_float(w[e]);
  const uint32_t h = (e & 1) ? (w[e >> 1] >> 16) : (w[e >> 1] & 0xffffu);
  return __uint_as_float(h << 16);
}

// Rows of a warp's buffer for turning a tall tile's chunk around: 16 chunk
// columns x 32 wide rows, padded to 33 words (conflict-free both ways).
constexpr int kTurnRows = 16;
constexpr int kTurnLd = 33;
constexpr uint32_t kTurnBytesPerWarp = kTurnRows * kTurnLd * 4;

// Tall W (W[j][i] holds the wide element (i, j)): the warp's 32 x 32 block
// of O' (lane = wide row row0 + lane, v[e] = wide column col0 + e) is turned
// around through the warp's shared-memory buffer in two halves of 16 columns,
// after which each lane holds 16 consecutive elements of one W row (row
// col0 + 16h + lane / 2, from wide row row0 + 16 (lane & 1)) and reads,
// updates and writes them with 16-byte accesses.  Warp-collective: every
// lane of the warp calls it for the same tile.
__device__ __forceinline__ void fin_store_tall(const FinalStore& f, const FinTile& t, int row0,
                                               int col0, const float (&v)[32],
                                               const uint32_t (&w)[32], float* turn, int lane) {
  const bool muon = (f.mode == 1);
  const bool bf = t.bf;
  const int i0 = row0 + 16 * (lane & 1);
  const float* src = turn + (lane >> 1) * kTurnLd + 16 * (lane & 1);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    __syncwarp();  // the previous half's reads are done
#pragma unroll
    for (int e = 0; e < 16; ++e) turn[e * kTurnLd + lane] = v[16 * h + e];
    __syncwarp();
    const int j = col0 + 16 * h + (lane >> 1);
    if (t.base == nullptr || j >= t.m_real || i0 >= t.n_real) continue;
    const int64_t off = static_cast<int64_t>(j) * t.ld + i0;
    const bool whole = i0 + 16 <= t.n_real;
#pragma unroll
    for (int g = 0; g < 2; ++g) {  // 8 elements at a time
      float o[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        o[k] = src[8 * g + k];
        if (muon) o[k] = fmaf(-t.lr_scale, o[k], fin_w(bf, w, 16 * h + 8 * g + k) * t.decay);
      }
      if (whole) {
        if (bf) {
          uint4 u;
          __nv_bfloat162* hp = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
          for (int e = 0; e < 4; ++e) hp[e] = __floats2bfloat162_rn(o[2 * e], o[2 * e + 1]);
          *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(t.base) + off + 8 * g) = u;
        } else {
          float4* d = reinterpret_cast<float4*>(static_cast<float*>(t.base) + off + 8 * g);
          d[0] = make_float4(o[0], o[1], o[2], o[3]);
          d[1] = make_float4(o[4], o[5], o[6], o[7]);
        }
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (i0 + 8 * g + k >= t.n_real) continue;
          if (bf)
            static_cast<__nv_bfloat16*>(t.base)[off + 8 * g + k] = __float2bfloat16_rn(o[k]);
          else
            static_cast<float*>(t.base)[off + 8 * g + k] = o[k];
        }
      }
    }
  }
}

// Wide W: the lane's 32 elements are consecutive in W row `row`.
__device__ __forceinline__ void fin_store(const FinalStore& f, const FinTile& t, int row, int col0,
                                          const float (&v)[32], const uint32_t (&w)[32]) {
  if (t.base == nullptr || row >= t.n_real) return;
  const bool muon = (f.mode == 1);
  const bool bf = t.bf;
  float o[32];
#pragma unroll
  for (int e = 0; e < 32; ++e) o[e] = muon ? fmaf(-t.lr_scale, v[e], fin_w(bf, w, e) * t.decay) : v[e];
  {
    const int64_t roff = static_cast<int64_t>(row) * t.ld;
    if (t.v8 && col0 + 32 <= t.m_real) {
      if (bf) {
        uint4 u[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u[k]);
#pragma unroll
          for (int e = 0; e < 4; ++e) h[e] = __floats2bfloat162_rn(o[8 * k + 2 * e], o[8 * k + 2 * e + 1]);
        }
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(t.base) + roff + col0;
        st_global_v8(dst, u[0], u[1]);
        st_global_v8(dst + 16, u[2], u[3]);
      } else {
        float* dst = static_cast<float*>(t.base) + roff + col0;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          st_global_v8(dst + 8 * k,
                       make_uint4(__float_as_uint(o[8 * k]), __float_as_uint(o[8 * k + 1]),
                                  __float_as_uint(o[8 * k + 2]), __float_as_uint(o[8 * k + 3])),
                       make_uint4(__float_as_uint(o[8 * k + 4]), __float_as_uint(o[8 * k + 5]),
                                  __float_as_uint(o[8 * k + 6]), __float_as_uint(o[8 * k + 7])));
      }
      return;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int j = col0 + 8 * k;
      if (j >= t.m_real) continue;
      const int64_t off = roff + j;
      if (bf) {
        uint4 u;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) h[e] = __floats2bfloat162_rn(o[8 * k + 2 * e], o[8 * k + 2 * e + 1]);
        *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(t.base) + off) = u;
      } else {
        float4* q = reinterpret_cast<float4*>(static_cast<float*>(t.base) + off);
        q[0] = make_float4(o[8 * k], o[8 * k + 1], o[8 * k + 2], o[8 * k + 3]);
        q[1] = make_float4(o[8 * k + 4], o[8 * k + 5], o[8 * k + 6], o[8 * k + 7]);
      }
    }
  }
}

// Epilogue of one 128 x BN tile for the calling warp (TMEM lane quarter q,
// rows tm*128 + q*32 + lane): waits for the accumulator (tfull_bar, parity),
// applies the kernel's epilogue and stores.  The residual operand of the next
// 32-column chunk is loaded while the current chunk is finished.  (Staging the
// mirrored store through shared memory was slower: it competes with the
// tensor core for shared-memory bandwidth.)  With kTmaOut the direct
// (untransposed) store goes through a per-warp 2 KB staging box per plane
// (32 rows x 64 bytes, 64-byte swizzle) and one TMA store per box, so L2
// sees whole 64-byte row segments instead of one request per lane.  The last
// update's epilogue gets the warp's turn-around buffer (kTurnBytesPerWarp) in
// sbuf instead, for tall W.
// Returns false if the wait gave up.
template <int BN, int EPI, bool SYM, int kChunksPerWarp = BN / 32, bool kTmaOut = false>
__device__ __forceinline__ bool epilogue_tile(const GemmParams& p, uint32_t t_acc, int b, int tm,
                                              int tn, int q, int lane, uint64_t* tfull_bar,
                                              uint32_t parity, volatile int* abort_flag,
                                              int c_begin = 0, const CUtensorMap* tmO = nullptr,
                                              const CUtensorMap* tmO2 = nullptr,
                                              uint8_t* sbuf = nullptr, int slice = 0) {
  const int row0 = tm * kBM + q * 32;
  const int row = row0 + lane;
  const bool mirror = SYM && (tn > tm / (BN / kBM));
  constexpr int K = epi_kind(EPI);
  constexpr bool kX3 = epi_x3(EPI);
  const __nv_bfloat16* aux_row =
      (K == kEpiGram) ? nullptr
                        : p.aux + static_cast<int64_t>(b) * p.aux_bstride +
                              static_cast<int64_t>(row) * p.aux_ld + tn * BN;
  uint4 cur_h[4], cur_l[4], nxt_h[4], nxt_l[4];
  // lo planes: the update of the bf16 precision (runtime flags), every kind
  // of the split-bf16 precision except the Gram's input
  const bool lo_in = (K == kEpiUpdate || (kX3 && K == kEpiPoly)) && p.lo_in;
  const bool lo_out = (K == kEpiUpdate || (kX3 && K != kEpiFinal)) && p.lo_out;
  if (K != kEpiGram) {
    load_raw4(aux_row + c_begin * 32, cur_h);
    if (lo_in) load_raw4(aux_row + p.lo_off + c_begin * 32, cur_l);
  }
  constexpr bool kFin = (K == kEpiFinal);
  constexpr bool kTall = kFin && epi_tall(EPI);
  // symmetric kinds of the bf16 precision: the mirrored copy goes out as a
  // TMA store of a transposed box too
  constexpr bool kMirrorTma = kTmaOut && SYM && !kX3;
  FinTile ft{};
  uint32_t w_cur[32], w_nxt[32];
  if (kFin) {
    ft = fin_tile(p.fin, b);
    fin_prefetch(p.fin, ft, row, row0, tn * BN + c_begin * 32, kChunksPerWarp * 32, lane);
    fin_load<kTall>(p.fin, ft, row, row0, tn * BN + c_begin * 32, w_cur);
  }
  // per-tile scalars, loaded before the accumulator wait so that their
  // latency hides behind it: the first iteration's 1/||X|| and, in the
  // update, the fp32 residual of this row's diagonal entry of P
  float ms = 1.f;
  if (p.mscale != nullptr) ms = p.mscale[b];
  float d_row = 0.f;
  if (K == kEpiUpdate || K == kEpiFinal) {
    if (!kX3) d_row = p.pdiag_in[static_cast<int64_t>(b) * p.pdiag_bstride + row];
  }
  if (!mbar_wait_bounded(tfull_bar, parity, abort_flag, p.status, p.timeout_ns)) return false;
  tc_fence_after();
  __nv_bfloat16* out = p.out + static_cast<int64_t>(b) * p.out_bstride;
  const uint32_t t_row = t_acc + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
  for (int i = 0; i < kChunksPerWarp; ++i) {
    const int c = c_begin + i;
    if (K != kEpiGram && i + 1 < kChunksPerWarp) {
      load_raw4(aux_row + (c + 1) * 32, nxt_h);
      if (lo_in) load_raw4(aux_row + p.lo_off + (c + 1) * 32, nxt_l);
      if (kFin) fin_load<kTall>(p.fin, ft, row, row0, tn * BN + (c + 1) * 32, w_nxt);
    }
    uint32_t r[32];
    tmem_ld_32x32b_x32(t_row + c * 32, r);
    tmem_ld_wait(r);
    const int col0 = tn * BN + c * 32;
    if (K == kEpiGram && !kX3 && p.ksplit > 1) {
      // split-K: this slice's raw fp32 sums (k_gram_reduce finishes the Gram)
      float* dst = p.partial + ((static_cast<int64_t>(slice) * (p.total_tiles / p.ksplit /
                                                                 p.tiles_per_matrix) +
                                 b) * p.M + row) * p.M + col0;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        st_global_v8(dst + 8 * k, make_uint4(r[8 * k], r[8 * k + 1], r[8 * k + 2], r[8 * k + 3]),
                     make_uint4(r[8 * k + 4], r[8 * k + 5], r[8 * k + 6], r[8 * k + 7]));
      continue;
    }
    float v[32];
    if (K == kEpiGram) {
      const float s2 = ms * ms * p.cb;
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]) * s2;
    } else {
      float x[32];
      unpack_raw4(cur_h, x);
      if (K == kEpiPoly) {
        if (kX3 && lo_in) {
          float xl[32];
          unpack_raw4(cur_l, xl);
#pragma unroll
          for (int e = 0; e < 32; ++e) x[e] += xl[e];
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = fmaf(p.cc, __uint_as_float(r[e]), p.cb * x[e]);
      } else {
        float xl[32];
        if (lo_in) {
          unpack_raw4(cur_l, xl);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) xl[e] = 0.f;
        }
        if (kX3) {
          // split-bf16: P = bS + cS^2 carries no shift, X' = a X + P X
#pragma unroll
          for (int e = 0; e < 32; ++e)
            v[e] = fmaf(p.ca, x[e] + xl[e], __uint_as_float(r[e])) * ms;
        } else {
          // P = bS + cS^2 + (a - 1) I; its diagonal's rounding residual d;
          // when the product read X hi only, P lo is approximated by its
          // shift part (a - 1) lo (the rest, (bS + cS^2) lo, is small on the
          // directions that are still small and decays on converged ones)
          const float d = d_row;
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float xe = x[e] + xl[e];
            // X + P X + d_row X (+ clo X_lo)
            v[e] = fmaf(d, xe, fmaf(p.clo, xl[e], xe + __uint_as_float(r[e]))) * ms;
          }
        }
      }
    }
    if ((K == kEpiGram || K == kEpiPoly) && (p.pdiag != nullptr || kX3) && row >= col0 &&
        row < col0 + 32) {
      // the (a - 1) I shift; the diagonal's bf16 rounding residual is kept
      // in fp32 so that P's diagonal is exact to fp32 in the update
#pragma unroll
      for (int e = 0; e < 32; ++e)
        if (col0 + e == row) {
          v[e] += p.cd;
          if (p.pdiag != nullptr)
            p.pdiag[static_cast<int64_t>(b) * p.pdiag_bstride + row] =
                v[e] - __bfloat162float(__float2bfloat16_rn(v[e]));
        }
    }
    if (kFin) {
      if (kTall && ft.tall)
        fin_store_tall(p.fin, ft, row0, col0, v, w_cur, reinterpret_cast<float*>(sbuf), lane);
      else
        fin_store(p.fin, ft, row, col0, v, w_cur);
      if (i + 1 < kChunksPerWarp) {
#pragma unroll
        for (int k = 0; k < 4; ++k) cur_h[k] = nxt_h[k];
#pragma unroll
        for (int e = 0; e < 32; ++e) w_cur[e] = w_nxt[e];
      }
      continue;
    }
    uint4 u[4], ul[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u[k]);
      __nv_bfloat162* hl = reinterpret_cast<__nv_bfloat162*>(&ul[k]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float v0 = v[8 * k + 2 * e], v1 = v[8 * k + 2 * e + 1];
        h[e] = __floats2bfloat162_rn(v0, v1);
        if (lo_out) {
          const float2 f = __bfloat1622float2(h[e]);
          hl[e] = __floats2bfloat162_rn(v0 - f.x, v1 - f.y);
        }
      }
    }
    if constexpr (kTmaOut) {
      // the previous chunk's boxes must have been read out of the staging
      // buffers before they are overwritten
      if (lane == 0) tma_store_wait_read0();
      __syncwarp();
      // row `lane` of the box, 16-byte unit k at unit k ^ ((lane >> 1) & 3)
      // (the 64-byte swizzle; conflict-free for each quarter warp)
      const uint32_t sw = (static_cast<uint32_t>(lane) >> 1) & 3u;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t off = static_cast<uint32_t>(lane) * 64u + 16u * (static_cast<uint32_t>(k) ^ sw);
        *reinterpret_cast<uint4*>(sbuf + off) = u[k];
        if (lo_out) *reinterpret_cast<uint4*>(sbuf + 2048 + off) = ul[k];
      }
      if (kMirrorTma && mirror) {
        // transposed box in the second buffer (free: symmetric kinds of the
        // bf16 precision write no lo plane).  Box row c holds tile column
        // col0 + c over the warp's 32 rows.  Word w of a lane packs its
        // columns 2w, 2w+1; after one exchange with the neighbouring lane,
        // an even lane writes (its, neighbour's) value of column 2w and an
        // odd lane (neighbour's, its) value of column 2w + 1: each store
        // instruction fills two 64-byte box rows.
        const uint32_t* wv = reinterpret_cast<const uint32_t*>(u);
        const uint32_t odd = static_cast<uint32_t>(lane) & 1u;
        const uint32_t rbyte = 2u * (static_cast<uint32_t>(lane) & ~1u);
#pragma unroll
        for (int w = 0; w < 16; ++w) {
          const uint32_t x = __shfl_xor_sync(0xffffffffu, wv[w], 1);
          const uint32_t word = odd ? __byte_perm(x, wv[w], 0x7632) : __byte_perm(wv[w], x, 0x5410);
          const uint32_t c = 2u * static_cast<uint32_t>(w) + odd;
          const uint32_t off = c * 64u + ((((rbyte >> 4) ^ ((c >> 1) & 3u))) << 4) + (rbyte & 15u);
          *reinterpret_cast<uint32_t*>(sbuf + 2048 + off) = word;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_3d(tmO, sbuf, col0, row0, b);
        if (lo_out) tma_store_3d(tmO2, sbuf + 2048, col0, row0, b);
        if (kMirrorTma && mirror) tma_store_3d(tmO, sbuf + 2048, row0, col0, b);
        tma_store_commit();
      }
    } else {
      // the row's 32 values as two full-sector stores per plane (workspace
      // rows and planes are 256-byte aligned, col0 is a multiple of 32)
      __nv_bfloat16* drow = out + static_cast<int64_t>(row) * p.out_ld + col0;
      st_global_v8(drow, u[0], u[1]);
      st_global_v8(drow + 16, u[2], u[3]);
      if (lo_out) {
        st_global_v8(drow + p.lo_off, ul[0], ul[1]);
        st_global_v8(drow + p.lo_off + 16, ul[2], ul[3]);
      }
    }
    if (mirror && !kMirrorTma) {
      // transposed copy: for each column e the warp's 32 lanes (32
      // consecutive rows) store 64 contiguous bytes of row col0 + e
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const __nv_bfloat16 h = __float2bfloat16_rn(v[e]);
        out[static_cast<int64_t>(col0 + e) * p.out_ld + row] = h;
        if (kX3 && lo_out)
          out[static_cast<int64_t>(col0 + e) * p.out_ld + row + p.lo_off] =
              __float2bfloat16_rn(v[e] - __bfloat162float(h));
      }
    }
    if (K != kEpiGram) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        cur_h[k] = nxt_h[k];
        if (lo_in) cur_l[k] = nxt_l[k];
      }
    }
  }
  return true;
}

// One CTA per 128 x BN tile (shapes whose tile rows do not pair up, and the
// split-K Grams); every CTA loads its own A and B tiles.
template <int BN, bool B_MN, int EPI, bool SYM>
__global__ void __launch_bounds__(kGemmThreads, 1)
    k_ns_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
              const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmB2,
              const GemmParams p) {
  using C = Cfg<BN>;
  constexpr int kStages = C::kStages;
  constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, BN, B_MN);

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* smA = smem;
  uint8_t* smB = smem + kStages * C::kABytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * C::kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit0 = static_cast<int>(blockIdx.x);
  const int ustep = static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kEpiWarps * 32);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (p.b_lo_mask) tma_prefetch_desc(&tmB2);
    if (p.a_lo_mask) tma_prefetch_desc(&tmA2);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (threadIdx.x == 0) griddep_launch_dependents();
  griddep_wait();  // the previous kernel's outputs are this kernel's inputs
  const int nkb = p.K / kBK;
  const int nkb_total = nkb * p.kplanes;
  // split-K (symmetric Grams with few tiles): unit t is K-slice t % nsplit of tile t / nsplit
  const int nsplit = p.ksplit > 1 ? p.ksplit : 1;
  const int nkb_run = nkb_total / nsplit;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_par = 0;
      bool ok = true;
      for (int t = unit0; ok && t < p.total_tiles; t += ustep) {
        int b, tm, tn;
        decode_unit<BN, SYM, false>(p, t / nsplit, 0u, b, tm, tn);
        int plane = 0, kk = (t % nsplit) * nkb_run;    // operand plane, k-block within it
        for (int kb = 0; kb < nkb_run; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, p.status, p.timeout_ns)) {
            ok = false;
            break;
          }
          const int k0 = kk * kBK;
          const CUtensorMap* ta = ((p.a_lo_mask >> plane) & 1) ? &tmA2 : &tmA;
          const CUtensorMap* tb = ((p.b_lo_mask >> plane) & 1) ? &tmB2 : &tmB;
          if (++kk == nkb) {
            kk = 0;
            ++plane;
          }
          mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
          tma_load_3d(smA + stage * C::kABytes, ta, &full[stage], k0, tm * kBM, b);
          if (!B_MN) {
            tma_load_3d(smB + stage * C::kBBytes, tb, &full[stage], k0, tn * BN, b);
          } else {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              tma_load_3d(smB + stage * C::kBBytes + j * (64 * kBK * 2), tb, &full[stage],
                          tn * BN + j * 64, k0, b);
          }
          issued |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Every load this thread issued must land before the CTA exits.
      for (int s = 0; s < kStages; ++s)
        if ((issued >> s) & 1u) mbar_wait_drain(&full[s], (last_par >> s) & 1u, p.status, p.timeout_ns);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int t = unit0; ok && t < p.total_tiles; t += ustep) {
        if (!mbar_wait_bounded(&tempty[acc], acc_phase ^ 1u, abort_flag, p.status, p.timeout_ns))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < nkb_run; ++kb) {
          if (!mbar_wait_bounded(&full[stage], phase, abort_flag, p.status, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smA + stage * C::kABytes);
          const uint32_t b_addr = smem_u32(smB + stage * C::kBBytes);
#pragma unroll
          for (int ks = 0; ks < kBK / 16; ++ks) {
            // K-major A: 128 rows x 128 B, 8-row groups 1024 B apart; a 16-wide
            // k step is 32 B along the swizzled row.
            const uint64_t ad = smem_desc_sw128(a_addr + ks * 32, 16, 1024);
            uint64_t bd;
            if (B_MN) {
              // MN-major B: 64-element (128 B) wide atoms of kBK k-rows,
              // atoms kBK*128 B apart (LBO), 8 k-rows 1024 B apart (SBO);
              // a 16-deep k step is 16 rows = 2048 B.
              bd = smem_desc_sw128(b_addr + ks * 16 * 128, kBK * 128, 1024);
            } else {
              bd = smem_desc_sw128(b_addr + ks * 32, 16, 1024);
            }
            tc_mma_bf16(d_tmem, ad, bd, kIdesc, (kb | ks) != 0 ? 1u : 0u);
          }
          tc_commit(&empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // All MMAs issued by this thread complete before teardown.
      tc_commit(drain);
      mbar_wait_drain(drain, 0, p.status, p.timeout_ns);
    }
  } else {
    // ------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter of this warp
    // the last update's turn-around buffer for tall W, after the barriers
    uint8_t* turn = epi_tall(EPI)
                        ? smem + kStages * C::kStageBytes + 256 + (warp - 2) * kTurnBytesPerWarp
                        : nullptr;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = unit0; t < p.total_tiles; t += ustep) {
      int b, tm, tn;
      decode_unit<BN, SYM, false>(p, t / nsplit, 0u, b, tm, tn);
      if (!epilogue_tile<BN, EPI, SYM>(p, tmem_base + static_cast<uint32_t>(acc * BN), b, tm, tn,
                                       q, lane, &tfull[acc], acc_phase, abort_flag, 0, nullptr,
                                       nullptr, turn, t % nsplit))
        break;
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}


// Pair-wide (2-SM) variant, BN = 256: the CTA pair computes a 256 x 256 tile
// with one tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16) per k-step,
// issued by the even CTA.  Each CTA stages only its own 128 rows of A and its
// half (128 rows, or 128 columns when MN-major) of B, so a stage is 32 KB per
// CTA and six stages fit; both CTAs' loads complete on the even CTA's full
// barrier.  D is split across the two CTAs' tensor memory (128 rows each);
// each CTA's epilogue drains its own rows and reports to the even CTA's
// accumulator-empty barrier.
#ifndef MUON_TWO_SM_ACC
#define MUON_TWO_SM_ACC 2
#endif
constexpr int kAccBufs2 = MUON_TWO_SM_ACC;  // TMEM accumulators per CTA (256 columns each)
constexpr int kStages2 = 6;
#ifndef MUON_EPI2_WARPS
#define MUON_EPI2_WARPS 8
#endif
constexpr int kEpiWarps2 = MUON_EPI2_WARPS;             // 4 or 8 (two per TMEM lane quarter)
constexpr int kGemmThreads2 = 64 + 32 * kEpiWarps2;
constexpr uint32_t kHalfBytes2 = 128 * kBK * 2;      // 16 KB: 128 rows x 64 bf16
constexpr uint32_t kStageBytes2 = 2 * kHalfBytes2;   // A + B half, per CTA
// TMA-store staging: per epilogue warp one 2 KB box for the hi plane and one
// for the lo plane (every kind but the last update, which writes W itself)
constexpr uint32_t kStagingPerWarp2 = 4096;
// (the last update has no TMA stores; its warps get turn-around buffers)
__host__ __device__ constexpr uint32_t staging_per_warp2(int epi) {
  return epi_kind(epi) != kEpiFinal ? kStagingPerWarp2 : (epi_tall(epi) ? kTurnBytesPerWarp : 0u);
}
__host__ __device__ constexpr uint32_t staging_bytes2(int epi) {
  return kEpiWarps2 * staging_per_warp2(epi);
}
__host__ __device__ constexpr size_t smem_bytes2(int epi) {
  return kStages2 * kStageBytes2 + staging_bytes2(epi) + 1024 + 256;
}

template <bool B_MN, int EPI, bool SYM>
__global__ void __launch_bounds__(kGemmThreads2, 1)
    k_ns_gemm2(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
               const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmB2,
               const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmO2,
               const GemmParams p) {
  constexpr int BN = 256;
  constexpr bool kTmaOut = epi_kind(EPI) != kEpiFinal;
  constexpr uint32_t kTmemCols = kAccBufs2 * BN;
  constexpr uint32_t kIdesc = idesc_bf16_f32(2 * kBM, BN, B_MN);

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* smA = smem;
  uint8_t* smB = smem + kStages2 * kHalfBytes2;
  uint8_t* staging = smem + kStages2 * kStageBytes2;  // 1024-byte aligned
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + staging_bytes2(EPI));
  uint64_t* empty = full + kStages2;
  uint64_t* tfull = empty + kStages2;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = (rank == 0);
  const int unit0 = static_cast<int>(blockIdx.x >> 1);
  const int ustep = static_cast<int>(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages2; ++s) {
      mbar_init(&full[s], 1);    // the even CTA's arrive_expect_tx; bytes from both CTAs
      mbar_init(&empty[s], 1);   // the even CTA's MMA commit, multicast to both
    }
    for (int a = 0; a < kAccBufs2; ++a) {
      mbar_init(&tfull[a], 1);                 // MMA commit, multicast to both
      mbar_init(&tempty[a], 2 * kEpiWarps2);   // one arrival per epilogue warp of both CTAs
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (p.b_lo_mask) tma_prefetch_desc(&tmB2);
    if (p.a_lo_mask) tma_prefetch_desc(&tmA2);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (threadIdx.x == 0) griddep_launch_dependents();
  griddep_wait();  // the previous kernel's outputs are this kernel's inputs
  const int nkb = p.K / kBK;
  const int nkb_total = nkb * p.kplanes;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      const uint32_t full0 = mapa_shared(&full[0], 0);  // the even CTA's full barriers
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_par = 0;
      bool ok = true;
      for (int t = unit0; ok && t < p.total_tiles; t += ustep) {
        int b, tm, tn;
        decode_unit<BN, SYM, true>(p, t, rank, b, tm, tn);
        int plane = 0, kk = 0;
        for (int kb = 0; kb < nkb_total; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, p.status, p.timeout_ns)) {
            ok = false;
            break;
          }
          const int k0 = kk * kBK;
          const CUtensorMap* ta = ((p.a_lo_mask >> plane) & 1) ? &tmA2 : &tmA;
          const CUtensorMap* tb = ((p.b_lo_mask >> plane) & 1) ? &tmB2 : &tmB;
          if (++kk == nkb) {
            kk = 0;
            ++plane;
          }
          const uint32_t bar = full0 + static_cast<uint32_t>(stage) * 8u;
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * kStageBytes2);
          tma_load_3d_pair(smA + stage * kHalfBytes2, ta, bar, k0, tm * kBM, b);
          if (!B_MN) {
            tma_load_3d_pair(smB + stage * kHalfBytes2, tb, bar, k0,
                             tn * BN + static_cast<int>(rank) * 128, b);
          } else {
#pragma unroll
            for (int j = 0; j < 2; ++j)
              tma_load_3d_pair(smB + stage * kHalfBytes2 + j * (64 * kBK * 2), tb, bar,
                               tn * BN + (static_cast<int>(rank) * 2 + j) * 64, k0, b);
          }
          issued |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages2) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // The even CTA's full barriers count both CTAs' bytes: draining them
      // there covers every load of the pair.
      if (leader)
        for (int s = 0; s < kStages2; ++s)
          if ((issued >> s) & 1u)
            mbar_wait_drain(&full[s], (last_par >> s) & 1u, p.status, p.timeout_ns);
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------------------------------------------------- MMA issuer
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int t = unit0; ok && t < p.total_tiles; t += ustep) {
        if (!mbar_wait_bounded(&tempty[acc], acc_phase ^ 1u, abort_flag, p.status, p.timeout_ns))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < nkb_total; ++kb) {
          if (!mbar_wait_bounded(&full[stage], phase, abort_flag, p.status, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smA + stage * kHalfBytes2);
          const uint32_t b_addr = smem_u32(smB + stage * kHalfBytes2);
#pragma unroll
          for (int ks = 0; ks < kBK / 16; ++ks) {
            const uint64_t ad = smem_desc_sw128(a_addr + ks * 32, 16, 1024);
            const uint64_t bd = B_MN ? smem_desc_sw128(b_addr + ks * 16 * 128, kBK * 128, 1024)
                                     : smem_desc_sw128(b_addr + ks * 32, 16, 1024);
            tc_mma_bf16_pair(d_tmem, ad, bd, kIdesc, (kb | ks) != 0 ? 1u : 0u);
          }
          tc_commit_pair_multicast(&empty[stage], 0x3);
          if (++stage == kStages2) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair_multicast(&tfull[acc], 0x3);
        if (++acc == kAccBufs2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      tc_commit_pair_multicast(drain, 0x1);
      mbar_wait_drain(drain, 0, p.status, p.timeout_ns);
    }
  } else {
    // ------------------------------------------------------------- epilogue
    const int q = warp & 3;
    constexpr int kChunksPerWarp2 = (BN / 32) / (kEpiWarps2 / 4);
    const int c_begin = ((warp - 2) >> 2) * kChunksPerWarp2;
    const uint32_t tempty0 = mapa_shared(&tempty[0], 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = unit0; t < p.total_tiles; t += ustep) {
      int b, tm, tn;
      decode_unit<BN, SYM, true>(p, t, rank, b, tm, tn);
      if (!epilogue_tile<BN, EPI, SYM, kChunksPerWarp2, kTmaOut>(
              p, tmem_base + static_cast<uint32_t>(acc * BN), b, tm, tn, q, lane, &tfull[acc],
              acc_phase, abort_flag, c_begin, &tmO, &tmO2,
              staging + (warp - 2) * staging_per_warp2(EPI)))
        break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty0 + static_cast<uint32_t>(acc) * 8u);
      if (++acc == kAccBufs2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // every TMA store this warp issued completes before the CTA exits
    if (kTmaOut && lane == 0) tma_store_wait_all0();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}


// ---- split-K Gram: the sum of the K-slices and the Gram epilogue ---------
// One thread per 4 consecutive columns of a row; the slices are added in
// index order, so the result depends on the matrix alone.  Same epilogue as
// the unsplit Gram: scale (1/||X||^2 on the first iteration, b when the Gram
// writes P directly), the (a - 1) shift on the diagonal with its fp32
// rounding residual, bf16 store, transposed copy of off-diagonal super-blocks.
struct GramReduceArgs {
  const float* partial;   // [ksplit][batch][n][n]
  int ksplit, batch, n, bn;
  __nv_bfloat16* out;     // [batch][n][n]
  float cb, cd;
  const float* mscale;    // [batch] or nullptr
  float* pdiag;           // [batch][n] or nullptr
};

__global__ void __launch_bounds__(256) k_gram_reduce(const GramReduceArgs a) {
  griddep_wait();
  const int q = a.n / 4;
  const int64_t per_mat = static_cast<int64_t>(a.n) * q;
  const int64_t total = per_mat * a.batch;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int b = static_cast<int>(i / per_mat);
    const int rem = static_cast<int>(i - static_cast<int64_t>(b) * per_mat);
    const int row = rem / q;
    const int col = (rem - row * q) * 4;
    const int sr = row / a.bn, sc = col / a.bn;
    if (sc < sr) continue;  // lower super-blocks are written as mirrors
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int sl = 0; sl < a.ksplit; ++sl) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(
          a.partial + ((static_cast<int64_t>(sl) * a.batch + b) * a.n + row) * a.n + col));
      acc[0] += v.x; acc[1] += v.y; acc[2] += v.z; acc[3] += v.w;
    }
    const float ms = a.mscale != nullptr ? a.mscale[b] : 1.f;
    const float f = ms * ms * a.cb;
    __nv_bfloat16 h[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float v = acc[e] * f;
      if (row == col + e) {
        v += a.cd;
        if (a.pdiag != nullptr)
          a.pdiag[static_cast<int64_t>(b) * a.n + row] = v - __bfloat162float(__float2bfloat16_rn(v));
      }
      h[e] = __float2bfloat16_rn(v);
    }
    __nv_bfloat16* o = a.out + static_cast<int64_t>(b) * a.n * a.n;
    uint2 u;
    __nv_bfloat162* hp = reinterpret_cast<__nv_bfloat162*>(&u);
    hp[0] = __halves2bfloat162(h[0], h[1]);
    hp[1] = __halves2bfloat162(h[2], h[3]);
    *reinterpret_cast<uint2*>(o + static_cast<int64_t>(row) * a.n + col) = u;
    if (sc > sr) {
#pragma unroll
      for (int e = 0; e < 4; ++e) o[static_cast<int64_t>(col + e) * a.n + row] = h[e];
    }
  }
}

// ---- split-K Gram of a 128 x 128 S with the polynomial, on CUDA cores -----
// For Grams of at most 128 rows over a long K (the per-head matrices of a
// split_head weight), the K-slices' fp32 sums are added in index order into
// S in shared memory (fp32, scaled by 1/||X||^2 on the first iteration) and
// P = b S + c S^2 + (a - 1) I is formed there directly, in fp32, and stored
// in bf16 with its diagonal's rounding residual: one pass instead of a
// reduction pass, a bf16 S and a 128 x 128 x 128 tensor-core launch whose
// time is all launch latency.  S^2 uses S's symmetry,
// (S^2)_ij = sum_k S_ki S_kj, so that both operands are rows of S.  Each
// block forms kRpRows rows of P of one matrix (k ascending: the result
// depends on the matrix alone).
constexpr int kRpN = 128;
constexpr int kRpRows = 32;
constexpr int kRpThreads = 256;  // (kRpRows / 4) x (kRpN / 4): a 4 x 4 block of P each
constexpr size_t kRpSmem = static_cast<size_t>(kRpN) * kRpN * 4;

struct GramReducePolyArgs {
  const float* partial;   // [ksplit][batch][128][128] raw accumulators
  int ksplit, batch;
  __nv_bfloat16* P;       // [batch][128][128]
  float* pdiag;           // [batch][128]
  const float* mscale;    // [batch] (first iteration: 1/||X||) or nullptr
  float cb, cc, cd;       // P = cb S + cc S^2 + cd I
};

__global__ void __launch_bounds__(kRpThreads) k_gram_reduce_poly(const GramReducePolyArgs a) {
  extern __shared__ __align__(16) float Ssm[];  // [128][128]
  griddep_wait();
  const int b = blockIdx.y, r0 = blockIdx.x * kRpRows, tid = threadIdx.x;
  const float ms = a.mscale != nullptr ? a.mscale[b] : 1.f;
  const float f = ms * ms;
  constexpr int kPer = kRpN * kRpN / 4 / kRpThreads;  // float4 of S per thread
  const int64_t mat = static_cast<int64_t>(kRpN) * kRpN;
  // all of a thread's loads of two slices in flight at once (the sums are
  // latency-bound otherwise); slices added in index order
  float4 sum[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) sum[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int sl = 0; sl < a.ksplit; sl += 2) {
    const float4* s0 = reinterpret_cast<const float4*>(
        a.partial + (static_cast<int64_t>(sl) * a.batch + b) * mat);
    const float4* s1 = reinterpret_cast<const float4*>(
        a.partial + (static_cast<int64_t>(sl + 1) * a.batch + b) * mat);
    const bool two = sl + 1 < a.ksplit;
    float4 x[kPer], y[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      x[i] = __ldcg(s0 + tid + i * kRpThreads);
      y[i] = two ? __ldcg(s1 + tid + i * kRpThreads) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      sum[i].x += x[i].x; sum[i].y += x[i].y; sum[i].z += x[i].z; sum[i].w += x[i].w;
      if (two) {
        sum[i].x += y[i].x; sum[i].y += y[i].y; sum[i].z += y[i].z; sum[i].w += y[i].w;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kPer; ++i)
    reinterpret_cast<float4*>(Ssm)[tid + i * kRpThreads] =
        make_float4(sum[i].x * f, sum[i].y * f, sum[i].z * f, sum[i].w * f);
  __syncthreads();
  const int i0 = r0 + 4 * (tid >> 5), j0 = 4 * (tid & 31);
  float acc[4][4] = {};
#pragma unroll 4
  for (int k = 0; k < kRpN; ++k) {
    const float4 x = *reinterpret_cast<const float4*>(Ssm + k * kRpN + i0);  // S_ki (warp-uniform)
    const float4 y = *reinterpret_cast<const float4*>(Ssm + k * kRpN + j0);  // S_kj
    const float xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
    for (int ii = 0; ii < 4; ++ii)
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) acc[ii][jj] = fmaf(xs[ii], ys[jj], acc[ii][jj]);
  }
  __nv_bfloat16* P = a.P + static_cast<int64_t>(b) * mat;
#pragma unroll
  for (int ii = 0; ii < 4; ++ii) {
    const int i = i0 + ii;
    const float4 sv = *reinterpret_cast<const float4*>(Ssm + i * kRpN + j0);
    float v[4] = {fmaf(a.cc, acc[ii][0], a.cb * sv.x), fmaf(a.cc, acc[ii][1], a.cb * sv.y),
                  fmaf(a.cc, acc[ii][2], a.cb * sv.z), fmaf(a.cc, acc[ii][3], a.cb * sv.w)};
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
      if (i == j0 + jj) {
        v[jj] += a.cd;
        a.pdiag[static_cast<int64_t>(b) * kRpN + i] =
            v[jj] - __bfloat162float(__float2bfloat16_rn(v[jj]));
      }
    uint2 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
    h[0] = __floats2bfloat162_rn(v[0], v[1]);
    h[1] = __floats2bfloat162_rn(v[2], v[3]);
    *reinterpret_cast<uint2*>(P + static_cast<int64_t>(i) * kRpN + j0) = u;
  }
}

// ---- the whole chain on chip: iterates of one 128-row tile ------------------
// For wide iterates of at most 128 rows (n <= 128: the per-head matrices of a
// split_head weight, 128 x 4096, among them) the polynomial and the update
// are short in K and the three-GEMM chain spends its time in launch latency
// and in epilogues that stream X through L2.  Here one cluster of C CTAs runs
// the whole chain of one matrix ("Muon 优化器" §2, the iteration; Algorithm 1's
// Newton–Schulz call): CTA c keeps columns [c w, (c + 1) w) of X for all
// iterations, the hi plane in shared memory in the 128-byte-swizzled layout the
// tensor core reads (K-major for the Gram, MN-major for the update) and the
// lo plane in tensor memory.  Per iteration:
//   Gram    each CTA: the partial S_c = X_c X_c^T (M = N = 128, K = w) in TMEM;
//           its rows, scaled by 1/||X||^2 in the first iteration, in fp16, go
//           to the CTAs that own them (CTA c owns rows [c R, (c + 1) R),
//           R = 128 / C) as one bulk copy per owner;
//   sum     each owner adds the C partials of its rows in rank order (fp32)
//           and sends its rows of S, in bf16, to every other CTA (bulk
//           copies again);
//   poly    every CTA forms the whole P = b S + c S^2 + (a - 1) I (S^2 on the
//           tensor core, M = N = K = 128) and its diagonal's fp32 rounding
//           residual; all CTAs compute the same P from the same bf16 S;
//   update  X_c' = X_c + P X_c in groups of 128 columns (two TMEM
//           accumulators: one group's epilogue overlaps the next group's
//           MMAs), the epilogue writing the new hi plane back into shared
//           memory and the lo plane into tensor memory; once the lo plane is
//           gone the next iteration's Gram MMAs run group by group inside
//           the update, in the lo plane's TMEM columns.
// The arithmetic is that of the tiled chain's bf16 precision (S and P in
// bf16, the shift and the residual planes as described at the top of this
// file).  Each bulk copy completes on an mbarrier of the receiving CTA, and
// every buffer is reused only once the exchange order shows that its readers
// are done.  A dedicated warp issues the MMAs (the issuing thread waits for
// each MMA to be accepted); 16 warps drain TMEM.  The last iteration writes W
// (or the output) directly, W prefetched into L2 when the chain starts;
// without a fused store the final iterate goes back to the workspace.  Every
// wait is bounded; a CTA whose wait gave up skips its remaining work, meets
// the others at the final cluster barrier and then waits (bounded) for the
// copies still owed to it, so that none leaves while another may write or
// read its shared memory.
constexpr int kCcThreads = 512;  // drain warps: lane quarter warp & 3, 32-column quarter warp >> 2;
                                 // the block adds one warp that issues the MMAs
constexpr int kCcMaxIters = 64;
constexpr int kCcMaxCluster = 16;  // 16: a non-portable cluster size, used where the GPU places it
constexpr int kCcMaxW = 512;
constexpr uint32_t kCcBlk = 128 * 128;  // a 128-row x 64-column bf16 block (16 KB)
constexpr uint32_t kCcTmemCols = 512;   // accumulators [0, 256), lo plane [256, 256 + w / 2)

struct ClusterChainParams {
  int C, w;                   // CTAs per matrix, columns per CTA (multiple of 128, <= kCcMaxW)
  int m_pad;
  const __nv_bfloat16* x;     // first iterate, hi plane [batch][128][m_pad]; lo at +lo_off
  __nv_bfloat16* xout;        // fin.mode == 0: the final iterate (its lo at +lo_off if it has one)
  int64_t lo_off;
  const float* inv_s;         // [batch] (1/||X||, first iteration), or nullptr
  int iters;
  float coef[kCcMaxIters][3];
  FinalStore fin;
  uint32_t* status;
  uint64_t timeout_ns;
};

__host__ __device__ constexpr size_t cc_smem_bytes(int w) {
  return static_cast<size_t>(w / 64) * kCcBlk   // X hi
         + 2 * kCcBlk                           // S (bf16)
         + 2 * kCcBlk                           // partial rows sent, then P (bf16)
         + 2 * kCcBlk                           // partial rows received; turn-around buffers
         + 128 * 4                              // diagonal residual of P
         + 128                                  // barriers, TMEM slot, abort flag
         + 1024;                                // alignment
}

// 16-byte unit u of a 128-byte row r in a 128-byte-swizzled block.
__device__ __forceinline__ uint32_t sw128(int r, int u) {
  return static_cast<uint32_t>(r) * 128u + ((static_cast<uint32_t>(u) ^ (r & 7)) << 4);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_f16x2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Bulk copy (the TMA engine) of `bytes` from this CTA's shared memory into
// the shared memory of a CTA of the cluster, completing the bytes on that
// CTA's mbarrier (both cluster addresses from mapa).
__device__ __forceinline__ void bulk_copy_to_cluster(uint32_t dst_cluster, uint32_t src,
                                                     uint32_t bytes, uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst_cluster),
      "r"(src), "r"(bytes), "r"(bar_cluster)
      : "memory");
}

// The last update's W store (W <- W*decay - lr_scale*O', or O' itself into
// the output), 16 wide columns at a time.  Wide W: the lane's 16 values are
// consecutive in W row `row`.
__device__ __forceinline__ void cc_fin_wide16(const FinalStore& f, const FinTile& t, int row,
                                              int col0, const float (&v)[16]) {
  if (t.base == nullptr || row >= t.n_real) return;
  const bool muon = (f.mode == 1);
  const int64_t roff = static_cast<int64_t>(row) * t.ld;
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    const int j = col0 + 8 * g;
    if (j >= t.m_real) continue;  // m_real is a multiple of 8
    float o[8];
    if (t.bf) {
      uint4* q = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(t.base) + roff + j);
      if (muon) {
        const uint4 u = *q;
        const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 8; ++k)
          o[k] = fmaf(-t.lr_scale, v[8 * g + k],
                      __uint_as_float((k & 1) ? (wd[k >> 1] & 0xffff0000u) : (wd[k >> 1] << 16)) * t.decay);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) o[k] = v[8 * g + k];
      }
      *q = make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]), pack_bf16x2(o[4], o[5]),
                      pack_bf16x2(o[6], o[7]));
    } else {
      float4* q = reinterpret_cast<float4*>(static_cast<float*>(t.base) + roff + j);
      if (muon) {
        const float4 a = q[0], c = q[1];
        const float wf[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) o[k] = fmaf(-t.lr_scale, v[8 * g + k], wf[k] * t.decay);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) o[k] = v[8 * g + k];
      }
      q[0] = make_float4(o[0], o[1], o[2], o[3]);
      q[1] = make_float4(o[4], o[5], o[6], o[7]);
    }
  }
}

// Tall W (W[j][i] holds the wide element (i, j)): the warp's 32 x 16 block of
// O' (lane = wide row row0 + lane, v[e] = wide column col0 + e) turned around
// through the warp's 2 KB buffer (16 rows of 32 words, word c of row e at
// c ^ e: conflict-free both ways), after which the lane holds 16 consecutive
// elements of W row col0 + lane / 2, from wide row row0 + 16 (lane & 1).
// Warp-collective.
constexpr uint32_t kCcTurnBytes = 16 * 32 * 4;

__device__ __forceinline__ void cc_fin_tall16(const FinalStore& f, const FinTile& t, int row0,
                                              int col0, const float (&v)[16], float* turn,
                                              int lane) {
  __syncwarp();  // the buffer's previous readers are done
#pragma unroll
  for (int e = 0; e < 16; ++e) turn[e * 32 + (lane ^ e)] = v[e];
  __syncwarp();
  const int j = col0 + (lane >> 1), i0 = row0 + 16 * (lane & 1);
  if (t.base == nullptr || j >= t.m_real || i0 >= t.n_real) return;
  const bool muon = (f.mode == 1);
  const int er = lane >> 1;                    // buffer row (chunk column)
  const float* src = turn + er * 32;
  const int64_t off = static_cast<int64_t>(j) * t.ld + i0;
  const bool whole = i0 + 16 <= t.n_real;
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    float o[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) o[k] = src[(16 * (lane & 1) + 8 * g + k) ^ er];
    if (whole) {
      if (t.bf) {
        uint4* q = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(t.base) + off + 8 * g);
        if (muon) {
          const uint4 u = *q;
          const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int k = 0; k < 8; ++k)
            o[k] = fmaf(-t.lr_scale, o[k],
                        __uint_as_float((k & 1) ? (wd[k >> 1] & 0xffff0000u) : (wd[k >> 1] << 16)) * t.decay);
        }
        *q = make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]), pack_bf16x2(o[4], o[5]),
                        pack_bf16x2(o[6], o[7]));
      } else {
        float4* q = reinterpret_cast<float4*>(static_cast<float*>(t.base) + off + 8 * g);
        if (muon) {
          const float4 a = q[0], c = q[1];
          const float wf[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
          for (int k = 0; k < 8; ++k) o[k] = fmaf(-t.lr_scale, o[k], wf[k] * t.decay);
        }
        q[0] = make_float4(o[0], o[1], o[2], o[3]);
        q[1] = make_float4(o[4], o[5], o[6], o[7]);
      }
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int i = i0 + 8 * g + k;
        if (i >= t.n_real) continue;
        if (t.bf) {
          __nv_bfloat16* e = static_cast<__nv_bfloat16*>(t.base) + off + 8 * g + k;
          const float wv = muon ? fmaf(-t.lr_scale, o[k], __bfloat162float(*e) * t.decay) : o[k];
          *e = __float2bfloat16_rn(wv);
        } else {
          float* e = static_cast<float*>(t.base) + off + 8 * g + k;
          *e = muon ? fmaf(-t.lr_scale, o[k], *e * t.decay) : o[k];
        }
      }
    }
  }
}

// 16 columns of the update epilogue: X' = X + P X + d X (+ clo X_lo), scaled
// by 1/||X|| in the first iteration; hi back into shared memory (units u0,
// u0 + 1 of row `row` of block xr), lo (kLoOut) into tensor memory.
template <bool kLoIn, bool kLoOut>
__device__ __forceinline__ void cc_update16(uint32_t t_acc, uint32_t t_lo, uint8_t* xr, int row,
                                            int u0, float d, float clo, float msc) {
  uint32_t r[16], l[8];
  tmem_ld_32x32b_x16(t_acc, r);
  if (kLoIn) tmem_ld_32x32b_x8(t_lo, l);
  const uint4 h0 = *reinterpret_cast<const uint4*>(xr + sw128(row, u0));
  const uint4 h1 = *reinterpret_cast<const uint4*>(xr + sw128(row, u0 + 1));
  tmem_ld_wait();
  tmem_ld_tie(r);
  if (kLoIn) tmem_ld_tie(l);
  const uint32_t hw_in[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
  uint32_t hw[8], lw[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hw_in[k]));
    float v0, v1;
    if (kLoIn) {
      const float2 xl = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&l[k]));
      const float xe0 = x.x + xl.x, xe1 = x.y + xl.y;
      v0 = fmaf(d, xe0, fmaf(clo, xl.x, xe0 + __uint_as_float(r[2 * k]))) * msc;
      v1 = fmaf(d, xe1, fmaf(clo, xl.y, xe1 + __uint_as_float(r[2 * k + 1]))) * msc;
    } else {
      v0 = fmaf(d, x.x, x.x + __uint_as_float(r[2 * k])) * msc;
      v1 = fmaf(d, x.y, x.y + __uint_as_float(r[2 * k + 1])) * msc;
    }
    const __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
    hw[k] = *reinterpret_cast<const uint32_t*>(&h);
    if (kLoOut) {
      const float2 f2 = __bfloat1622float2(h);
      lw[k] = pack_bf16x2(v0 - f2.x, v1 - f2.y);
    }
  }
  *reinterpret_cast<uint4*>(xr + sw128(row, u0)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
  *reinterpret_cast<uint4*>(xr + sw128(row, u0 + 1)) = make_uint4(hw[4], hw[5], hw[6], hw[7]);
  if (kLoOut) tmem_st_32x32b_x8(t_lo, lw);
}

// The update's MMAs for group g (128 columns): D[g & 1] = P X_g, A = P
// (K-major), B = X (MN-major), eight k steps of 16; completion on `full`.
__device__ __forceinline__ void cc_issue_update(uint32_t tmem, uint64_t dP, uint64_t dXmn, int g,
                                                uint64_t* full) {
  constexpr uint32_t kIdescMN = idesc_bf16_f32(128, 128, true);
  const uint32_t d_tm = tmem + static_cast<uint32_t>((g & 1) * 128);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint64_t ad = dP + static_cast<uint64_t>(((ks >> 2) * kCcBlk + (ks & 3) * 32) >> 4);
    const uint64_t bd = dXmn + static_cast<uint64_t>((2 * g * kCcBlk + ks * 2048) >> 4);
    tc_mma_bf16(d_tm, ad, bd, kIdescMN, ks != 0 ? 1u : 0u);
  }
  tc_commit(full);
}

// The next iteration's Gram over the two X blocks of group g, accumulated in
// TMEM columns [256, 384); completion on `done` after the last group.
__device__ __forceinline__ void cc_issue_gram(uint32_t tmem, uint64_t dX, int g, uint64_t* done) {
  constexpr uint32_t kIdescKK = idesc_bf16_f32(128, 128, false);
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      const uint64_t dd = dX + static_cast<uint64_t>(((2 * g + j) * kCcBlk + ks * 32) >> 4);
      tc_mma_bf16(tmem + 256, dd, dd, kIdescKK, (g | j | ks) != 0 ? 1u : 0u);
    }
  if (done != nullptr) tc_commit(done);
}

template <int C>
__global__ void __launch_bounds__(kCcThreads + 32, 1)
    k_ns_cluster_chain(const __grid_constant__ CUtensorMap tmX,
                       const __grid_constant__ ClusterChainParams p) {
  constexpr int R = 128 / C;  // rows of S this CTA sums
  static_assert(R % 8 == 0, "cluster size");
  constexpr int kItems = (R * 16 + kCcThreads - 1) / kCcThreads;  // 8-column units per thread
  constexpr uint32_t kSlot = R * 256;  // one CTA's fp16 partial rows for one owner
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const int nb = p.w / 64, nq = p.w / 128;
  uint8_t* sX = smem;
  uint8_t* sS = smem + nb * kCcBlk;  // S (bf16, K-major, two blocks)
  uint8_t* sT = sS + 2 * kCcBlk;     // partial rows to send [owner][R][128] fp16, then P
  uint8_t* sV = sT + 2 * kCcBlk;     // partial rows received [sender][R][128] fp16;
                                     // turn-around buffers in the last update
  float* pdiag = reinterpret_cast<float*>(sV + 2 * kCcBlk);
  uint64_t* bars = reinterpret_cast<uint64_t*>(pdiag + 128);
  uint64_t* mma_bar = bars;       // Gram / polynomial MMAs done
  uint64_t* tma_bar = bars + 1;   // first iterate loaded
  uint64_t* ufull = bars + 2;     // [2] update accumulators full
  uint64_t* uempty = bars + 4;    // [2] update accumulators drained (one arrival per warp)
  uint64_t* pbar = bars + 6;      // partial rows received
  uint64_t* sbar = bars + 7;      // rows of S received
  uint64_t* drain = bars + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 9);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  constexpr int kWarps = kCcThreads / 32;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // warps 0-15 drain TMEM (lane quarter warp & 3, 32-column quarter warp >> 2);
  // warp 16 issues the tensor-core MMAs (an issuing thread waits for each MMA
  // to be accepted, about as long as the MMA runs)
  const bool mma_warp = (warp == kWarps);
  const bool mma_thread = mma_warp && lane == 0;
  const int q = warp & 3, h4 = (warp >> 2) & 3;
  const int row = 32 * q + lane;
  const uint32_t rank = cluster_ctarank();
  const int b = static_cast<int>(blockIdx.x) / C;
  const int col_base = static_cast<int>(rank) * p.w;

  if (tid == 0) {
    mbar_init(mma_bar, 1);
    mbar_init(tma_bar, 1);
    mbar_init(&ufull[0], 1);
    mbar_init(&ufull[1], 1);
    mbar_init(&uempty[0], kWarps);
    mbar_init(&uempty[1], kWarps);
    mbar_init(pbar, 1);
    mbar_init(sbar, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmX);
  }
  if (mma_warp) {
    tmem_alloc(tmem_slot, kCcTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // every CTA's barriers are initialised before any copy completes on them
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_row = tmem + (static_cast<uint32_t>(32 * q) << 16);  // this warp's lanes
  const uint32_t t_lo = t_row + 256;
  const uint32_t aX = smem_u32(sX), aS = smem_u32(sS), aT = smem_u32(sT), aV = smem_u32(sV);
  constexpr uint32_t kIdescKK = idesc_bf16_f32(128, 128, false);
  constexpr uint32_t kIdescMN = idesc_bf16_f32(128, 128, true);

  griddep_wait();  // X and 1/||X|| come from the previous kernels
  const float ms = p.inv_s != nullptr ? p.inv_s[b] : 1.f;
  // ---- first iterate: hi plane by TMA (64-column boxes of 128 rows), lo
  // plane into tensor memory (column j at TMEM column j / 2, two per word)
  if (tid == 0) {
    mbar_arrive_expect_tx(tma_bar, static_cast<uint32_t>(nb) * kCcBlk);
    for (int kb = 0; kb < nb; ++kb)
      tma_load_3d(sX + kb * kCcBlk, &tmX, tma_bar, col_base + kb * 64, 0, b);
  }
  const int64_t row_off = (static_cast<int64_t>(b) * 128 + row) * p.m_pad + col_base;
  if (kLoIters > 0 && !mma_warp) {
    for (int g = 0; g < nq; ++g) {
      const int cs = 128 * g + 32 * h4;
      const uint4* src = reinterpret_cast<const uint4*>(p.x + p.lo_off + row_off + cs);
      uint32_t u[16];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 v = src[k];
        u[4 * k] = v.x; u[4 * k + 1] = v.y; u[4 * k + 2] = v.z; u[4 * k + 3] = v.w;
      }
      tmem_st_32x32b_x16(t_lo + cs / 2, u);
    }
    tmem_st_wait();
  }
  const bool tma_done = mbar_wait_bounded(tma_bar, 0, abort_flag, p.status, p.timeout_ns);
  bool ok = __syncthreads_and(tma_done) != 0;

  const bool has_fin = p.fin.mode != 0;
  FinTile ft{};
  if (has_fin) ft = fin_tile(p.fin, b);
  // the W this CTA's last update reads, into L2 now (it is read once, at the end)
  if (has_fin && !mma_warp)
    for (int g = 0; g < nq; ++g)
      fin_prefetch(p.fin, ft, row, 32 * q, col_base + 128 * g + 32 * h4, 32, lane);
  // the last update's turn-around buffers, one per epilogue warp
  float* turn = reinterpret_cast<float*>(sV + (warp & 15) * kCcTurnBytes);
  // descriptors of the operand blocks (start-address field advanced per k step)
  const uint64_t dX = smem_desc_sw128(aX, 16, 1024);          // K-major X
  const uint64_t dXmn = smem_desc_sw128(aX, kCcBlk, 1024);    // MN-major X
  const uint64_t dS = smem_desc_sw128(aS, 16, 1024);
  const uint64_t dP = smem_desc_sw128(aT, 16, 1024);
  uint32_t mma_ph = 0, uf_ph = 0, ue_ph = 0, x_ph = 0;  // uf / ue: bit g & 1 per accumulator
  int armed = 0;            // exchange phases armed on pbar / sbar and not yet seen complete
  bool gram_early = false;  // this iteration's Gram was issued during the previous update

  for (int it = 0; it < p.iters; ++it) {
    const float ca = p.coef[it][0], cb = p.coef[it][1], cc = p.coef[it][2];
    const bool first = (it == 0), last = (it + 1 == p.iters);
    const bool fin_now = last && has_fin;
    const bool lo_in = it < kLoIters;
    const bool lo_out = it + 1 < kLoIters && !fin_now;
    const float clo = lo_in ? ca - 1.f : 0.f;
    const float msc = first ? ms : 1.f;
    // Once the lo plane is gone its TMEM columns hold the next iteration's
    // Gram, whose MMAs then start group by group inside this update.
    const bool gram_next = !lo_in && !lo_out && !last;
    const uint32_t g_acc = gram_early ? 256u : 0u;
    if (!ok) break;

    // this iteration's exchanges: C partial slots in, the other CTAs' rows of S in
    if (tid == 0) {
      mbar_arrive_expect_tx(pbar, static_cast<uint32_t>(C) * kSlot);
      mbar_arrive_expect_tx(sbar, static_cast<uint32_t>(C - 1) * kSlot);
    }
    armed = 2;

    // ---- Gram: partial S of this CTA's columns
    if (mma_thread && !gram_early) {
      tc_fence_after();
      for (int kb = 0; kb < nb; ++kb)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t dd = dX + static_cast<uint64_t>((kb * kCcBlk + ks * 32) >> 4);
          tc_mma_bf16(tmem, dd, dd, kIdescKK, (kb | ks) != 0 ? 1u : 0u);
        }
      tc_commit(mma_bar);
    }
    {
      const bool w = mbar_wait_bounded(mma_bar, mma_ph, abort_flag, p.status, p.timeout_ns);
      mma_ph ^= 1u;
      ok = __syncthreads_and(w) != 0;
      if (!ok) break;
    }
    if (!mma_warp) {
      tc_fence_after();
      // row `row`, columns [32 h4, 32 h4 + 32) of the partial, scaled by
      // 1/||X||^2 in the first iteration (every entry is then at most the
      // squared spectral norm of the iterate, about 1.5), in fp16, into the
      // owner's slot of the send buffer: 16-byte units (8 columns) swizzled
      // by row, unit u at (u & ~7) | ((u ^ row) & 7)
      const float f = first ? ms * ms : 1.f;
      uint8_t* dst = sT + (row / R) * kSlot + (row % R) * 256;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t r[16];
        tmem_ld_32x32b_x16(t_row + g_acc + 32 * h4 + 16 * half, r);
        tmem_ld_wait();
        tmem_ld_tie(r);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int u = 4 * h4 + 2 * half + k;
          const int phys = (u & ~7) | ((u ^ row) & 7);
          *reinterpret_cast<uint4*>(dst + phys * 16) = make_uint4(
              pack_f16x2(__uint_as_float(r[8 * k]) * f, __uint_as_float(r[8 * k + 1]) * f),
              pack_f16x2(__uint_as_float(r[8 * k + 2]) * f, __uint_as_float(r[8 * k + 3]) * f),
              pack_f16x2(__uint_as_float(r[8 * k + 4]) * f, __uint_as_float(r[8 * k + 5]) * f),
              pack_f16x2(__uint_as_float(r[8 * k + 6]) * f, __uint_as_float(r[8 * k + 7]) * f));
        }
      }
      fence_proxy_async_smem();  // the copies read these rows through the async proxy
      tc_fence_before();
    }
    __syncthreads();
    if (tid == 0)
      for (int o = 0; o < C; ++o)
        bulk_copy_to_cluster(mapa_shared_u32(aV + rank * kSlot, static_cast<uint32_t>(o)),
                             aT + o * kSlot, kSlot, mapa_shared(pbar, static_cast<uint32_t>(o)));

    // ---- sum: rows [rank R, rank R + R) of S, the C slots added in rank
    // order in fp32, stored in bf16 (K-major, 128-byte swizzle)
    {
      const bool w = mbar_wait_bounded(pbar, x_ph, abort_flag, p.status, p.timeout_ns);
      ok = __syncthreads_and(w) != 0;
      if (!ok) break;
      armed = 1;
    }
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
      const int i = tid + k * kCcThreads;
      if (!mma_warp && i < R * 16) {
        const int lr = i >> 4, u = i & 15;
        const int r = static_cast<int>(rank) * R + lr;
        const uint32_t off = lr * 256 + (((u & ~7) | ((u ^ r) & 7)) << 4);
        uint4 v[C];
#pragma unroll
        for (int pr = 0; pr < C; ++pr) v[pr] = *reinterpret_cast<const uint4*>(sV + pr * kSlot + off);
        float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int pr = 0; pr < C; ++pr) {
          const uint32_t wv[4] = {v[pr].x, v[pr].y, v[pr].z, v[pr].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 h = __half22float2(*reinterpret_cast<const __half2*>(&wv[j]));
            s[2 * j] += h.x;
            s[2 * j + 1] += h.y;
          }
        }
        // columns 8u .. 8u + 7: block u / 8, unit u % 8
        *reinterpret_cast<uint4*>(sS + (u >> 3) * kCcBlk + sw128(r, u & 7)) =
            make_uint4(pack_bf16x2(s[0], s[1]), pack_bf16x2(s[2], s[3]), pack_bf16x2(s[4], s[5]),
                       pack_bf16x2(s[6], s[7]));
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && C > 1) {
      // this CTA's rows of S (R rows of each block, contiguous) to every other CTA
      for (int o = 0; o < C; ++o) {
        if (o == static_cast<int>(rank)) continue;
        const uint32_t bar = mapa_shared(sbar, static_cast<uint32_t>(o));
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          const uint32_t off = blk * kCcBlk + rank * R * 128;
          bulk_copy_to_cluster(mapa_shared_u32(aS + off, static_cast<uint32_t>(o)), aS + off,
                               R * 128, bar);
        }
      }
    }
    {
      const bool w = mbar_wait_bounded(sbar, x_ph, abort_flag, p.status, p.timeout_ns);
      x_ph ^= 1u;
      ok = __syncthreads_and(w) != 0;
      if (!ok) break;
      armed = 0;
    }

    // ---- polynomial: P = b S + c S^2 + (a - 1) I, into the send buffer
    if (cc != 0.f) {
      if (mma_thread) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t dd = dS + static_cast<uint64_t>(((ks >> 2) * kCcBlk + (ks & 3) * 32) >> 4);
          tc_mma_bf16(tmem + 128, dd, dd, kIdescKK, ks != 0 ? 1u : 0u);
        }
        tc_commit(mma_bar);
      }
      const bool w = mbar_wait_bounded(mma_bar, mma_ph, abort_flag, p.status, p.timeout_ns);
      mma_ph ^= 1u;
      ok = __syncthreads_and(w) != 0;
      if (!ok) break;
      tc_fence_after();
    }
    if (!mma_warp) {
      // row `row`, columns [32 h4, 32 h4 + 32): block h4 / 2, units 4 (h4 & 1) .. + 3,
      // in two 16-column halves; the warps with q == h4 hold the diagonal
      // (column `lane` of their chunk)
      const uint8_t* srow = sS + (h4 >> 1) * kCcBlk;
      uint8_t* prow = sT + (h4 >> 1) * kCcBlk;
      const bool diag = (q == h4);
      float s_d = 0.f, a_d = 0.f;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int u0 = 4 * (h4 & 1) + 2 * half;
        uint32_t r[16];
        if (cc != 0.f) tmem_ld_32x32b_x16(t_row + 128 + 32 * h4 + 16 * half, r);
        const uint4 sv0 = *reinterpret_cast<const uint4*>(srow + sw128(row, u0));
        const uint4 sv1 = *reinterpret_cast<const uint4*>(srow + sw128(row, u0 + 1));
        if (cc != 0.f) {
          tmem_ld_wait();
          tmem_ld_tie(r);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) r[e] = 0u;
        }
        const uint32_t sw[8] = {sv0.x, sv0.y, sv0.z, sv0.w, sv1.x, sv1.y, sv1.z, sv1.w};
        if (diag && (lane >> 4) == half) {
          // predicated selects (an indexed read would put r in local memory)
          uint32_t ab = 0u, sb = 0u;
          const int idx = lane & 15;
#pragma unroll
          for (int e0 = 0; e0 < 16; ++e0) {
            const uint32_t wd = sw[e0 >> 1];
            const uint32_t sv = (e0 & 1) ? (wd & 0xffff0000u) : (wd << 16);
            asm volatile(
                "{\n\t.reg .pred p;\n\tsetp.eq.s32 p, %4, %5;\n\t"
                "selp.b32 %0, %2, %0, p;\n\tselp.b32 %1, %3, %1, p;\n\t}"
                : "+r"(ab), "+r"(sb)
                : "r"(r[e0]), "r"(sv), "r"(e0), "r"(idx));
          }
          a_d = __uint_as_float(ab);
          s_d = __uint_as_float(sb);
        }
        uint32_t out[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float2 sf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&sw[j]));
          out[j] = pack_bf16x2(fmaf(cc, __uint_as_float(r[2 * j]), cb * sf.x),
                               fmaf(cc, __uint_as_float(r[2 * j + 1]), cb * sf.y));
        }
        *reinterpret_cast<uint4*>(prow + sw128(row, u0)) = make_uint4(out[0], out[1], out[2], out[3]);
        *reinterpret_cast<uint4*>(prow + sw128(row, u0 + 1)) = make_uint4(out[4], out[5], out[6], out[7]);
      }
      if (diag) {
        const int e = lane;
        // the (a - 1) shift on the diagonal; its fp32 rounding residual kept
        const float vd = fmaf(cc, a_d, cb * s_d) + (ca - 1.f);
        const __nv_bfloat16 hd = __float2bfloat16_rn(vd);
        pdiag[row] = vd - __bfloat162float(hd);
        *reinterpret_cast<__nv_bfloat16*>(prow + sw128(row, 4 * (h4 & 1) + (e >> 3)) + (e & 7) * 2) = hd;
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- update: X_c' = X_c + P X_c, groups of 128 columns (TMEM
    // accumulator g & 1), MN-major B straight from the X blocks.  Warp 0's
    // first lane issues the MMAs; every warp reports a drained accumulator
    // on uempty and goes on to the next group.
    if (mma_warp) {
      // issue the first two groups, then each further group (and the next
      // iteration's Gram over the columns just written) once every warp has
      // drained the accumulator it reuses
      if (lane == 0) {
        tc_fence_after();
        cc_issue_update(tmem, dP, dXmn, 0, &ufull[0]);
        if (nq > 1) cc_issue_update(tmem, dP, dXmn, 1, &ufull[1]);
        for (int g = 0; g < nq; ++g) {
          // every group completes a phase of uempty[g & 1]; the phases not
          // waited for here have completed before the next iteration's waits
          const uint32_t bit = 1u << (g & 1);
          const uint32_t par = (ue_ph & bit) ? 1u : 0u;
          ue_ph ^= bit;
          if (!ok || (g + 2 >= nq && !gram_next)) continue;
          if (!mbar_wait_bounded(&uempty[g & 1], par, abort_flag, p.status, p.timeout_ns)) {
            ok = false;
            continue;
          }
          tc_fence_after();
          if (g + 2 < nq) cc_issue_update(tmem, dP, dXmn, g + 2, &ufull[g & 1]);
          if (gram_next) cc_issue_gram(tmem, dX, g, g + 1 == nq ? mma_bar : nullptr);
        }
      }
      __syncwarp();
    } else {
      const float d = pdiag[row];
      for (int g = 0; g < nq; ++g) {
        const uint32_t bit = 1u << (g & 1);
        bool w = ok && mbar_wait_bounded(&ufull[g & 1], (uf_ph & bit) ? 1u : 0u, abort_flag,
                                         p.status, p.timeout_ns);
        uf_ph ^= bit;
        w = __all_sync(0xffffffffu, w);
        ok = ok && w;
        const int cs = 128 * g + 32 * h4;  // slice column of the thread's chunk
        uint8_t* xr = sX + (cs >> 6) * kCcBlk;
        const int u0 = (cs & 63) >> 3;
        const uint32_t t_acc = t_row + (g & 1) * 128 + 32 * h4;
        if (ok) tc_fence_after();
        if (fin_now) {
          // O' in two 16-column halves (the last iteration never reads the lo
          // plane)
          uint4 hv[4];
          if (ok) {
#pragma unroll
            for (int k = 0; k < 4; ++k) hv[k] = *reinterpret_cast<const uint4*>(xr + sw128(row, u0 + k));
          }
          const uint32_t* hw_in = reinterpret_cast<const uint32_t*>(hv);
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float v[16];
            if (ok) {
              uint32_t r[16];
              tmem_ld_32x32b_x16(t_acc + 16 * half, r);
              tmem_ld_wait();
              tmem_ld_tie(r);
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const float2 x = __bfloat1622float2(
                    *reinterpret_cast<const __nv_bfloat162*>(&hw_in[8 * half + k]));
                v[2 * k] = fmaf(d, x.x, x.x + __uint_as_float(r[2 * k])) * msc;
                v[2 * k + 1] = fmaf(d, x.y, x.y + __uint_as_float(r[2 * k + 1])) * msc;
              }
            }
            const int col0 = col_base + cs + 16 * half;
            if (ft.tall) {
              if (ok) cc_fin_tall16(p.fin, ft, 32 * q, col0, v, turn, lane);
            } else if (ok) {
              cc_fin_wide16(p.fin, ft, row, col0, v);
            }
          }
        } else if (ok) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const uint32_t ta = t_acc + 16 * half, tl = t_lo + cs / 2 + 8 * half;
            if (lo_in && lo_out)
              cc_update16<true, true>(ta, tl, xr, row, u0 + 2 * half, d, clo, msc);
            else if (lo_in)
              cc_update16<true, false>(ta, tl, xr, row, u0 + 2 * half, d, clo, msc);
            else
              cc_update16<false, false>(ta, tl, xr, row, u0 + 2 * half, d, clo, msc);
          }
        }
        if (gram_next) fence_proxy_async_smem();  // X' blocks of group g feed the next Gram
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&uempty[g & 1]);
      }
    }
    if (lo_out) tmem_st_wait();
    fence_proxy_async_smem();
    tc_fence_before();
    gram_early = gram_next;
    ok = __syncthreads_and(ok) != 0;
  }

  // ---- the final iterate back to the workspace (no fused store)
  if (ok && !has_fin && p.iters > 0 && !mma_warp) {
    const bool lo = p.iters < kLoIters;
    __nv_bfloat16* dst = p.xout + row_off;
    for (int g = 0; g < nq; ++g) {
      const int cs = 128 * g + 32 * h4;
      const uint8_t* xr = sX + (cs >> 6) * kCcBlk;
      const int u0 = (cs & 63) >> 3;
      uint4 hv[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) hv[k] = *reinterpret_cast<const uint4*>(xr + sw128(row, u0 + k));
      st_global_v8(dst + cs, hv[0], hv[1]);
      st_global_v8(dst + cs + 16, hv[2], hv[3]);
      if (lo) {
        uint32_t l[16];
        tmem_ld_32x32b_x16(t_lo + cs / 2, l);
        tmem_ld_wait();
        tmem_ld_tie(l);
        st_global_v8(dst + p.lo_off + cs, make_uint4(l[0], l[1], l[2], l[3]),
                     make_uint4(l[4], l[5], l[6], l[7]));
        st_global_v8(dst + p.lo_off + cs + 16, make_uint4(l[8], l[9], l[10], l[11]),
                     make_uint4(l[12], l[13], l[14], l[15]));
      }
    }
  }

  // ---- teardown.  Every MMA and the first load complete; then, once all
  // CTAs of the cluster have stopped issuing copies (the cluster barrier),
  // the copies this CTA still expected after a wait gave up have landed
  // (bounded waits), so that none writes into shared memory after the CTA
  // has left it.
  if (mma_thread) {
    tc_commit(drain);
    mbar_wait_drain(drain, 0, p.status, p.timeout_ns);
  }
  if (tid == 0) {
    griddep_launch_dependents();
    if (!tma_done) mbar_wait_drain(tma_bar, 0, p.status, p.timeout_ns);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (tid == 0) {
    if (armed == 2) mbar_wait_drain(pbar, x_ph, p.status, p.timeout_ns);
    if (armed >= 1) mbar_wait_drain(sbar, x_ph, p.status, p.timeout_ns);
  }
  __syncthreads();
  if (mma_warp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kCcTmemCols);
  }
}

// Gram and polynomial of one iteration in one launch of the pair-wide
// kernel (bf16 precision, c != 0).  The launch's work units are numbered by
// tickets: every Gram unit (matrix-major) before any polynomial unit.  Each
// CTA pair claims its next ticket from a per-launch counter (one atomic
// add by the even CTA's producer, one unit ahead of the one it loads) and
// records it in its row of a ticket log in global memory, stamped with the
// launch's number; the odd CTA's producer and both CTAs' epilogue warps read
// their units from that row, and the MMA issuer from a per-stage tag the
// producer writes next to the operand stage (ticket_unit gives the order of
// the units).  A polynomial unit of matrix b
// reads S_b, written by all of b's Gram units: every epilogue warp adds 1 to
// the matrix's arrival counter once its TMA stores of a Gram unit are
// complete (counted at the start of its next unit, before that unit's
// accumulator wait, never after it), and the polynomial's producer and
// epilogue wait (bounded) until the counter reaches the launch's target.
// Because a ticket is only ever held by a CTA pair that is running, and every
// Gram ticket of a matrix is handed out before its first polynomial ticket,
// every Gram unit a polynomial unit waits for belongs to a resident pair that
// finishes it without waiting on anything (a pair's Gram units precede its
// polynomial units of the same matrices): the launch makes progress however
// few of its clusters the GPU runs at a time (other work may hold SMs).
// On a diagonal super-block each CTA's half of B is its own A rows: the
// operand is loaded once and the MMA reads it as both.  The
// counters are cumulative over a call's launches (zeroed by k_finalize_norm);
// the ticket counters and log are zeroed once per chain.
constexpr int kArrivalsPerUnit = 2 * kEpiWarps2;  // epilogue warps of a CTA pair
constexpr int kTicketDone = 0xFFFFFF;             // log entry: no further unit
constexpr int kTicketMask = 0xFFFFFF;
constexpr int kTagDone = -1;                      // stage tag: no further unit

struct GramPolyParams {
  GemmParams g;   // Gram phase
  GemmParams q;   // polynomial phase
  int* ctr;       // [batch] Gram arrivals, cumulative over the call's launches
  int target;     // counter value at which this launch's Gram of a matrix is complete
  int* tick;      // this launch's ticket counter (zero on entry)
  int* log;       // [clusters][log_cap] tickets claimed by each CTA pair, as stamp | (ticket + 1)
  int log_cap;    // entries per pair (>= all tickets + 2)
  int stamp;      // this launch's number within the chain, << 24
  int blk;        // matrices per ticket block
};

// Ticket -> phase (0 Gram, 1 polynomial) and unit index within the phase.
// Tickets run in blocks of `blk` matrices, each block's polynomial units one
// block behind its Gram units:
//   [G_0] [G_1 P_0] [G_2 P_1] ... [G_last P_last-1] [P_last]
// so that every Gram ticket of a matrix precedes its polynomial tickets (the
// hand-over's progress needs that) and S is read back about one block after
// it is written, while it is still in L2.  Units within a phase are
// matrix-major, as decode_unit takes them.
__device__ __forceinline__ void ticket_unit(const GramPolyParams& P, int T, int& ph, int& t) {
  const int total = P.g.total_tiles;                 // units per phase
  const int F = P.blk * P.g.tiles_per_matrix;        // units of a full block
  const int nb = (total + F - 1) / F;
  if (nb <= 1) {
    ph = T >= total ? 1 : 0;
    t = ph ? T - total : T;
    return;
  }
  if (T < F) {
    ph = 0;
    t = T;
    return;
  }
  T -= F;
  const int q = T / (2 * F);
  if (q < nb - 2) {  // the pair (G_{q+1}, P_q)
    const int r = T - q * 2 * F;
    ph = r < F ? 0 : 1;
    t = r < F ? (q + 1) * F + r : q * F + (r - F);
    return;
  }
  T -= (nb - 2) * 2 * F;
  const int last = total - (nb - 1) * F;  // units of the last block
  if (T < last) {
    ph = 0;
    t = (nb - 1) * F + T;
  } else if (T < last + F) {
    ph = 1;
    t = (nb - 2) * F + (T - last);
  } else {
    ph = 1;
    t = (nb - 1) * F + (T - last - F);
  }
}

__global__ void __launch_bounds__(kGemmThreads2, 1)
    k_ns_gram_poly(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmS,
                   const __grid_constant__ CUtensorMap tmSo,
                   const __grid_constant__ CUtensorMap tmPo,
                   const __grid_constant__ GramPolyParams P) {
  constexpr int BN = 256;
  constexpr uint32_t kTmemCols = kAccBufs2 * BN;
  constexpr uint32_t kIdesc = idesc_bf16_f32(2 * kBM, BN, false);

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* smA = smem;
  uint8_t* smB = smem + kStages2 * kHalfBytes2;
  uint8_t* staging = smem + kStages2 * kStageBytes2;  // 1024-byte aligned
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + staging_bytes2(kEpiPoly));
  uint64_t* empty = full + kStages2;
  uint64_t* tfull = empty + kStages2;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* first_bar = drain + 1;  // odd CTA: its first ticket has arrived
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(first_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // even CTA: for the stage holding a unit's first k-block, the unit's
  // k-blocks << 1 | whether it is diagonal (or kTagDone)
  volatile int* unit_tag = reinterpret_cast<volatile int*>(tmem_slot + 2);
  volatile int* first_tick = reinterpret_cast<volatile int*>(tmem_slot + 2 + kStages2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = (rank == 0);
  uint32_t* const status = P.g.status;
  const uint64_t timeout_ns = P.g.timeout_ns;
  const int n_tickets = P.g.total_tiles + P.q.total_tiles;
  int* const my_log = P.log + static_cast<int64_t>(blockIdx.x >> 1) * P.log_cap;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages2; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < kAccBufs2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * kEpiWarps2);
    }
    mbar_init(drain, 1);
    mbar_init(first_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmS);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (threadIdx.x == 0) griddep_launch_dependents();
  // The even CTA claims tickets two units ahead of the one it loads and logs
  // them.  Its first two claims are made before the wait for the previous
  // kernel (they touch only this launch's own counter), and the first goes
  // to the odd CTA's shared memory directly; the log is written only after
  // the wait, since the fused launch before the previous kernel may still be
  // reading its rows until then.  The odd CTA reads its later units from the
  // log, each written a whole unit before it is needed.
  auto enc = [&](int t) { return P.stamp | (t >= n_tickets ? kTicketDone : t + 1); };
  auto dec = [](int e) { return (e & kTicketMask) == kTicketDone ? kTicketDone : (e & kTicketMask) - 1; };
  int T = kTicketDone, nxt = kTicketDone;
  if (warp == 0 && lane == 0 && leader) {
    T = atomicAdd(P.tick, 1);
    if (T >= n_tickets) T = kTicketDone;
    st_shared_cluster(mapa_shared(const_cast<int*>(first_tick), 1), T);
    mbar_arrive_release_cluster(mapa_shared(first_bar, 1));
    if (T != kTicketDone) {
      nxt = atomicAdd(P.tick, 1);
      if (nxt >= n_tickets) nxt = kTicketDone;
    }
  }
  griddep_wait();  // the previous kernel's outputs are this kernel's inputs
  if (warp == 0 && lane == 0 && leader) {
    st_relaxed_gpu(my_log, enc(T));
    if (T != kTicketDone) st_relaxed_gpu(my_log + 1, enc(nxt));
  }

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      const uint32_t full0 = mapa_shared(&full[0], 0);
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_par = 0;
      bool ok = true;
      if (!leader) {
        ok = mbar_wait_acquire_cluster(first_bar, 0, abort_flag, status, timeout_ns);
        T = *first_tick;
      }
      for (int j = 0; ok; ++j) {
        if (T == kTicketDone) {
          if (leader) {
            // tell the MMA issuer there is no further unit
            if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, status, timeout_ns))
              break;
            unit_tag[stage] = kTagDone;
            mbar_arrive(&full[stage]);
            // the drain below waits for this (at once complete) phase of the
            // stage, not for the one before it
            issued |= 1u << stage;
            last_par = (last_par & ~(1u << stage)) | (phase << stage);
          }
          break;
        }
        int ph, t;
        ticket_unit(P, T, ph, t);
        const GemmParams& p = ph ? P.q : P.g;
        const CUtensorMap* tm_ab = ph ? &tmS : &tmX;
        const int nkb = p.K / kBK;
        int b, tm, tn;
        decode_unit<BN, true, true>(p, t, rank, b, tm, tn);
        const bool diag = (tm >> 1) == tn;  // B's rows of this CTA = its A rows
        if (ph) {
          // S_b complete (normally long since)
          if (!wait_counter_bounded(P.ctr + b, P.target, abort_flag, status, timeout_ns)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();  // the TMA loads below read what the acquire saw
        }
        // even CTA: the unit after next, claimed now (its atomic completes
        // while this unit's k-blocks are issued) and logged with the last one
        int nn = kTicketDone;
        if (leader && nxt != kTicketDone && j + 2 < P.log_cap) nn = atomicAdd(P.tick, 1);
        int peek = 0;  // odd CTA: the log entry of the next unit, loaded ahead
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, status, timeout_ns)) {
            ok = false;
            break;
          }
          const uint32_t bar = full0 + static_cast<uint32_t>(stage) * 8u;
          if (leader) {
            if (kb == 0) unit_tag[stage] = (nkb << 1) | (diag ? 1 : 0);
            mbar_arrive_expect_tx(&full[stage], diag ? 2 * kHalfBytes2 : 2 * kStageBytes2);
          }
          tma_load_3d_pair(smA + stage * kHalfBytes2, tm_ab, bar, kb * kBK, tm * kBM, b);
          if (!diag)
            tma_load_3d_pair(smB + stage * kHalfBytes2, tm_ab, bar, kb * kBK,
                             tn * BN + static_cast<int>(rank) * 128, b);
          if (!leader && kb == 0) peek = ld_relaxed_gpu(my_log + j + 1);
          if (leader && kb == nkb - 1 && nxt != kTicketDone && j + 2 < P.log_cap) {
            if (nn >= n_tickets) nn = kTicketDone;
            st_relaxed_gpu(my_log + j + 2, enc(nn));
          }
          issued |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages2) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (leader) {
          T = nxt;
          nxt = nn;
        } else {
          if ((peek & ~kTicketMask) != P.stamp &&
              !wait_stamped_bounded(my_log + j + 1, P.stamp, &peek, abort_flag, status, timeout_ns))
            break;
          T = dec(peek);
        }
      }
      if (leader)
        for (int s = 0; s < kStages2; ++s)
          if ((issued >> s) & 1u)
            mbar_wait_drain(&full[s], (last_par >> s) & 1u, status, timeout_ns);
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------------------------------------------------- MMA issuer
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      while (true) {
        // the unit's first stage carries its length and kind
        if (!mbar_wait_bounded(&full[stage], phase, abort_flag, status, timeout_ns)) break;
        const int tag = unit_tag[stage];
        if (tag == kTagDone) break;
        const int nkb = tag >> 1;
        const bool diag = (tag & 1) != 0;
        if (!mbar_wait_bounded(&tempty[acc], acc_phase ^ 1u, abort_flag, status, timeout_ns))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (kb > 0 && !mbar_wait_bounded(&full[stage], phase, abort_flag, status, timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smA + stage * kHalfBytes2);
          const uint32_t b_addr = diag ? a_addr : smem_u32(smB + stage * kHalfBytes2);
#pragma unroll
          for (int ks = 0; ks < kBK / 16; ++ks) {
            const uint64_t ad = smem_desc_sw128(a_addr + ks * 32, 16, 1024);
            const uint64_t bd = smem_desc_sw128(b_addr + ks * 32, 16, 1024);
            tc_mma_bf16_pair(d_tmem, ad, bd, kIdesc, (kb | ks) != 0 ? 1u : 0u);
          }
          tc_commit_pair_multicast(&empty[stage], 0x3);
          if (++stage == kStages2) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair_multicast(&tfull[acc], 0x3);
        if (++acc == kAccBufs2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      tc_commit_pair_multicast(drain, 0x1);
      mbar_wait_drain(drain, 0, status, timeout_ns);
    }
  } else {
    // ------------------------------------------------------------- epilogue
    const int q = warp & 3;
    constexpr int kChunks = (BN / 32) / (kEpiWarps2 / 4);
    const int c_begin = ((warp - 2) >> 2) * kChunks;
    const uint32_t tempty0 = mapa_shared(&tempty[0], 0);
    uint8_t* sbuf = staging + (warp - 2) * kStagingPerWarp2;
    int acc = 0;
    uint32_t acc_phase = 0;
    int pending = -1;  // matrix of the last Gram unit whose arrival is not yet counted
    int peek = lane == 0 ? ld_relaxed_gpu(my_log) : 0;  // log entry of the next unit
    for (int j = 0;; ++j) {
      int e = peek, ok = 1;
      if (lane == 0 && (e & ~kTicketMask) != P.stamp)
        ok = wait_stamped_bounded(my_log + j, P.stamp, &e, abort_flag, status, timeout_ns);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      e = __shfl_sync(0xffffffffu, e, 0);
      if (!ok || (e & kTicketMask) == kTicketDone) break;
      if (lane == 0 && j + 1 < P.log_cap) peek = ld_relaxed_gpu(my_log + j + 1);
      if (pending >= 0) {
        if (lane == 0) {
          tma_store_wait_all0();
          fence_proxy_async_global();
          red_release_gpu_add(P.ctr + pending, 1);
        }
        pending = -1;
      }
      int ph, t;
      ticket_unit(P, (e & kTicketMask) - 1, ph, t);
      const GemmParams& p = ph ? P.q : P.g;
      int b, tm, tn;
      decode_unit<BN, true, true>(p, t, rank, b, tm, tn);
      bool r;
      if (ph == 0) {
        r = epilogue_tile<BN, kEpiGram, true, kChunks, true>(
            p, tmem_base + static_cast<uint32_t>(acc * BN), b, tm, tn, q, lane, &tfull[acc],
            acc_phase, abort_flag, c_begin, &tmSo, &tmSo, sbuf);
      } else {
        // the epilogue reads S_b itself (b S term): wait for it here too
        int ready = 1;
        if (lane == 0)
          ready = wait_counter_bounded(P.ctr + b, P.target, abort_flag, status, timeout_ns);
        ready = __shfl_sync(0xffffffffu, ready, 0);
        if (!ready) break;
        __syncwarp();  // lane 0's acquire orders every lane's reads of S_b
        r = epilogue_tile<BN, kEpiPoly, true, kChunks, true>(
            p, tmem_base + static_cast<uint32_t>(acc * BN), b, tm, tn, q, lane, &tfull[acc],
            acc_phase, abort_flag, c_begin, &tmPo, &tmPo, sbuf);
      }
      if (!r) break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty0 + static_cast<uint32_t>(acc) * 8u);
      if (++acc == kAccBufs2) {
        acc = 0;
        acc_phase ^= 1u;
      }
      if (ph == 0) pending = b;
    }
    if (lane == 0) {
      tma_store_wait_all0();
      if (pending >= 0) {
        fence_proxy_async_global();
        red_release_gpu_add(P.ctr + pending, 1);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

double l2_bytes() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev) != cudaSuccess || v <= 0)
    return 64.0 * (1 << 20);
  return static_cast<double>(v);
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

// K-major operand: [batch][rows][K] bf16, box = 64 (K) x box_rows.
bool map_kmajor(CUtensorMap* m, const void* base, int batch, int rows, int K, int box_rows) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(batch)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2,
                                 static_cast<cuuint64_t>(rows) * K * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// MN-major operand: [batch][K rows][N cols] bf16, box = 64 (N) x 64 (K).
bool map_mnmajor(CUtensorMap* m, const void* base, int batch, int K, int N) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(K),
                              static_cast<cuuint64_t>(batch)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(N) * 2,
                                 static_cast<cuuint64_t>(K) * N * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kBK), 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Store boxes of a [batch][rows][cols] bf16 output: 32 columns (64 bytes,
// the 64-byte swizzle span) x 32 rows, one box per epilogue warp and chunk.
bool map_store(CUtensorMap* m, const void* base, int batch, int rows, int cols) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(batch)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2,
                                 static_cast<cuuint64_t>(rows) * cols * 2};
  const cuuint32_t box[3] = {32, 32, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, bool B_MN, int EPI, bool SYM>
cudaError_t launch_gemm(const CUtensorMap& ta, const CUtensorMap& ta2, const CUtensorMap& tb,
                        const CUtensorMap& tb2, const GemmParams& p, double alg_flops,
                        cudaStream_t st) {
  auto kern = k_ns_gemm<BN, B_MN, EPI, SYM>;
  const size_t smem = Cfg<BN>::kSmemBytes + (epi_tall(EPI) ? kEpiWarps * kTurnBytesPerWarp : 0);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const KernelKind kind = epi_kind(EPI) == kEpiGram ? kKindGram
                          : (epi_kind(EPI) == kEpiPoly ? kKindPoly : kKindUpdate);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  const int units = std::max(1, std::min(p.total_tiles, sm_count()));
  cfg.gridDim = dim3(units);
  if (kUsePdl) {
    attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs += 1;
  }
  prof_begin(kind, st);
  e = cudaLaunchKernelEx(&cfg, kern, ta, ta2, tb, tb2, p);
  prof_end(kind, st, alg_flops, 0.0);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}


template <bool B_MN, int EPI, bool SYM>
cudaError_t launch_gemm2(const CUtensorMap& ta, const CUtensorMap& ta2, const CUtensorMap& tb,
                         const CUtensorMap& tb2, const CUtensorMap& to, const CUtensorMap& to2,
                         const GemmParams& p, double alg_flops, cudaStream_t st) {
  auto kern = k_ns_gemm2<B_MN, EPI, SYM>;
  constexpr size_t kSmem = smem_bytes2(EPI);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmem));
  if (e != cudaSuccess) return e;
  const KernelKind kind = epi_kind(EPI) == kEpiGram ? kKindGram
                          : (epi_kind(EPI) == kEpiPoly ? kKindPoly : kKindUpdate);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.blockDim = dim3(kGemmThreads2);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = st;
  cfg.gridDim = dim3(2);
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
  if (e != cudaSuccess) return e;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  const int units = std::max(1, std::min(p.total_tiles, clusters));
  cfg.gridDim = dim3(2 * units);
  if (kUsePdl) {
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
  }
  prof_begin(kind, st);
  e = cudaLaunchKernelEx(&cfg, kern, ta, ta2, tb, tb2, to, to2, p);
  prof_end(kind, st, alg_flops, 0.0);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}


// Gram + polynomial of one iteration as one launch (k_ns_gram_poly).
cudaError_t launch_gram_poly(const CUtensorMap& x, const CUtensorMap& sk, const CUtensorMap& so,
                             const CUtensorMap& po, const GramPolyParams& gp, double flops,
                             cudaStream_t st) {
  auto kern = k_ns_gram_poly;
  constexpr size_t kSmem = smem_bytes2(kEpiPoly);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.blockDim = dim3(kGemmThreads2);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = st;
  cfg.gridDim = dim3(2);
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
  if (e != cudaSuccess) return e;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  // at most one pair per Gram unit (more would only claim polynomial units
  // early and wait) and per row of the ticket log; the ticket hand-over needs
  // no pair to be resident alongside any other
  const int units = std::max(1, std::min(std::min(gp.g.total_tiles, clusters), kGpMaxClusters));
  cfg.gridDim = dim3(2 * units);
  if (kUsePdl) {
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
  }
  prof_begin(kKindGramPoly, st);
  e = cudaLaunchKernelEx(&cfg, kern, x, sk, so, po, gp);
  prof_end(kKindGramPoly, st, flops, 0.0);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Shape of the on-chip chain for a padded wide shape n_pad x m_pad: C CTAs
// per matrix (a power of two, at most kCcMaxCluster) of w columns each (a
// multiple of 128, at most kCcMaxW), the fewest CTAs that fit: the exchange
// between a cluster's CTAs costs about the same whatever their width, so wide
// slices give the most work per exchange (a 128 x 1024 matrix on 8 CTAs of 128
// columns ran at half the tiled chain's rate for large batches).  A function
// of the shape alone: a matrix's result does not depend on its batch.
bool cluster_chain_shape(int n_pad, int m_pad, int* C, int* w) {
  if (n_pad != kBM) return false;
  for (int c = 1; c <= kCcMaxCluster; c <<= 1) {
    if (m_pad % (c * 128) != 0) continue;
    if (m_pad / c > kCcMaxW) continue;
    *C = c;
    *w = m_pad / c;
    return true;
  }
  return false;
}

// The whole chain of every matrix in one launch of k_ns_cluster_chain;
// cudaErrorNotSupported where the GPU cannot hold one cluster of that shape.
cudaError_t launch_cluster_chain(const CUtensorMap& tmx, const NsChainArgs& a, int C, int w,
                                 double flops, cudaStream_t st) {
  auto kern = C == 16 ? k_ns_cluster_chain<16>
              : C == 8 ? k_ns_cluster_chain<8>
              : C == 4 ? k_ns_cluster_chain<4>
              : C == 2 ? k_ns_cluster_chain<2>
                       : k_ns_cluster_chain<1>;
  const size_t smem = cc_smem_bytes(w);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (C > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      return cudaErrorNotSupported;
    }
  }
  if (a.fin.mode != 0 && a.iters <= kLoIters) return cudaErrorNotSupported;
  ClusterChainParams p{};
  p.C = C;
  p.w = w;
  p.m_pad = a.m_pad;
  p.x = a.X0;
  p.xout = (a.iters & 1) ? a.X1 : a.X0;
  p.lo_off = a.lo_off;
  p.inv_s = a.inv_s;
  p.iters = a.iters;
  for (int it = 0; it < a.iters; ++it)
    for (int k = 0; k < 3; ++k) p.coef[it][k] = a.coeffs[3 * it + k];
  p.fin = a.fin;
  p.status = a.status;
  p.timeout_ns = a.timeout_ns;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.blockDim = dim3(kCcThreads + 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.gridDim = dim3(static_cast<unsigned>(C));
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
  if (e != cudaSuccess || clusters < 1) {
    (void)cudaGetLastError();
    return cudaErrorNotSupported;  // the tiled chain instead
  }
  cfg.gridDim = dim3(static_cast<unsigned>(a.batch * C));
  if (kUsePdl) {
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
  }
  prof_begin(kKindChain, st);
  e = cudaLaunchKernelEx(&cfg, kern, tmx, p);
  prof_end(kKindChain, st, flops, 0.0);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Tensor maps of one operand: K-major with 128-row boxes (A, and the B half a
// CTA of a pair loads) and BN-row boxes (unpaired B), MN-major (the update's
// B), each for the hi and the lo plane.  Operands without a lo plane carry
// their hi map in the lo slots (never read: the plane masks select hi only).
struct OperandMaps {
  CUtensorMap k128, kbn, mn, k128_lo, kbn_lo, mn_lo;
  CUtensorMap st, st_lo;  // 32 x 32 store boxes (pair-wide kernels' epilogue)
};

// Gram / polynomial: A and B are the same symmetric operand (X or S).
// `pair`: the pair-wide kernel (tile rows pair up and BN = 256).
template <int EPI>
cudaError_t launch_sym(int bn, bool pair, const OperandMaps& A, const OperandMaps& O,
                       const GemmParams& p, double f, cudaStream_t st) {
  if (bn == 256 && pair)
    return launch_gemm2<false, EPI, true>(A.k128, A.k128_lo, A.k128, A.k128_lo, O.st, O.st_lo, p,
                                          f, st);
  if (bn == 256)
    return launch_gemm<256, false, EPI, true>(A.k128, A.k128_lo, A.kbn, A.kbn_lo, p, f, st);
  return launch_gemm<128, false, EPI, true>(A.k128, A.k128_lo, A.kbn, A.kbn_lo, p, f, st);
}

// Update: A = P (K-major), B = X (MN-major).
template <int EPI>
cudaError_t launch_upd(int bn, bool pair, const OperandMaps& Pm, const OperandMaps& Xm,
                       const OperandMaps& Om, const GemmParams& p, double f, cudaStream_t st) {
  if (bn == 256 && pair)
    return launch_gemm2<true, EPI, false>(Pm.k128, Pm.k128_lo, Xm.mn, Xm.mn_lo, Om.st, Om.st_lo,
                                          p, f, st);
  if (bn == 256)
    return launch_gemm<256, true, EPI, false>(Pm.k128, Pm.k128_lo, Xm.mn, Xm.mn_lo, p, f, st);
  return launch_gemm<128, true, EPI, false>(Pm.k128, Pm.k128_lo, Xm.mn, Xm.mn_lo, p, f, st);
}

bool map_square(OperandMaps* o, const __nv_bfloat16* hi, const __nv_bfloat16* lo, int batch, int n,
                int bn) {
  if (!map_kmajor(&o->k128, hi, batch, n, n, kBM) || !map_kmajor(&o->kbn, hi, batch, n, n, bn) ||
      !map_store(&o->st, hi, batch, n, n))
    return false;
  if (lo == nullptr) {
    o->k128_lo = o->k128;
    o->kbn_lo = o->kbn;
    o->st_lo = o->st;
    return true;
  }
  return map_kmajor(&o->k128_lo, lo, batch, n, n, kBM) &&
         map_kmajor(&o->kbn_lo, lo, batch, n, n, bn) && map_store(&o->st_lo, lo, batch, n, n);
}

}  // namespace

bool ns_final_fused(int iters, bool x3) { return !x3 && iters > kLoIters; }

int gram_ksplit(int n_pad, int m_pad, bool x3) {
  // single-tile Grams (n <= 128) over a long K: up to 8 slices of >= 16 k-blocks
  if (x3 || n_pad != kBM) return 1;
  const int nkb = m_pad / kBK;
  int sl = 1;
  while (sl * 2 <= 8 && nkb / (sl * 2) >= 16 && nkb % (sl * 2) == 0) sl *= 2;
  return sl;
}

bool ns_final_has_lo(int iters, bool x3) { return x3 || iters < kLoIters; }

size_t gram_poly_log_ints(int batch, int n_pad, bool x3) {
  if (x3 || n_pad % 256 != 0) return 0;
  const int64_t S = n_pad / 256;
  const int64_t tickets = 2 * static_cast<int64_t>(batch) * (S * (S + 1) / 2);
  return static_cast<size_t>(kGpMaxLaunches + kGpMaxClusters * (tickets + 2));
}

cudaError_t run_ns_chain(const NsChainArgs& a, cudaStream_t st) {
  if (a.iters == 0) return cudaSuccess;
  if (encode_fn() == nullptr) return cudaErrorNotSupported;
  const int n = a.n_pad, m = a.m_pad, batch = a.batch;
  const int bn_sq = (n % 256 == 0) ? 256 : 128;
  // update tile width: 256 where the tile rows pair up (pair-wide kernel);
  // otherwise 128, twice the tiles for a short-K, epilogue-bound update
  const int bn_up = (m % 256 == 0 && n % 256 == 0) ? 256 : 128;
  const bool x3 = a.x3 != 0;

  // iterates of one 128-row tile: the whole chain on chip, one launch
  int cc_c = 0, cc_w = 0;
  if (kUseClusterChain && !x3 && a.iters <= kCcMaxIters && batch <= 65535 * 256 &&
      cluster_chain_shape(n, m, &cc_c, &cc_w)) {
    CUtensorMap tmx;
    if (!map_kmajor(&tmx, a.X0, batch, n, m, kBM)) return cudaErrorInvalidValue;
    const double nr = a.n, mr = a.m;
    const double flops = static_cast<double>(a.iters) * batch * (3.0 * nr * nr * mr + nr * nr * nr);
    const cudaError_t e = launch_cluster_chain(tmx, a, cc_c, cc_w, flops, st);
    if (e != cudaErrorNotSupported) return e;
    (void)cudaGetLastError();
  }

  OperandMaps X[2], S, P;
  __nv_bfloat16* xb[2] = {a.X0, a.X1};
  for (int i = 0; i < 2; ++i) {
    const __nv_bfloat16* lo = xb[i] + a.lo_off;
    if (!map_kmajor(&X[i].k128, xb[i], batch, n, m, kBM) ||
        !map_kmajor(&X[i].kbn, xb[i], batch, n, m, bn_sq) ||
        !map_mnmajor(&X[i].mn, xb[i], batch, n, m) ||
        !map_kmajor(&X[i].k128_lo, lo, batch, n, m, kBM) ||
        !map_kmajor(&X[i].kbn_lo, lo, batch, n, m, bn_sq) ||
        !map_mnmajor(&X[i].mn_lo, lo, batch, n, m) || !map_store(&X[i].st, xb[i], batch, n, m) ||
        !map_store(&X[i].st_lo, lo, batch, n, m))
      return cudaErrorInvalidValue;
  }
  if (!map_square(&S, a.A, x3 ? a.A + a.sq_lo_off : nullptr, batch, n, bn_sq) ||
      !map_square(&P, a.B, x3 ? a.B + a.sq_lo_off : nullptr, batch, n, bn_sq))
    return cudaErrorInvalidValue;

  // Algorithmic flops per launch (unpadded n x m, symmetric products at half
  // their dense count): Gram n^2 m, polynomial n^3, update 2 n^2 m per matrix.
  // The split-bf16 precision does three products for each (not counted).
  const double nr = a.n, mr = a.m;
  const double f_gram = batch * nr * nr * mr, f_poly = batch * nr * nr * nr,
               f_update = 2.0 * batch * nr * nr * mr;
  const int tm_sq = n / kBM;
  const int S_sq = n / bn_sq;
  const int sym_tiles = (bn_sq / kBM) * S_sq * (S_sq + 1) / 2;
  // split-bf16: planes (hi, hi), (hi, lo), (lo, hi) of (A, B)
  const int x3_planes = 3, x3_a_lo = 0b100, x3_b_lo = 0b010;

  // Consecutive launches walk the batch in opposite directions, so that each
  // starts on the matrices its predecessor wrote last (still in L2); the
  // first Gram follows the prepare pass, which writes the batch in order.
  int launch = 0;
  int gp_launches = 0;  // fused Gram + polynomial launches so far (counter targets)
  for (int it = 0; it < a.iters; ++it) {
    const float ca = a.coeffs[3 * it], cb = a.coeffs[3 * it + 1], cc = a.coeffs[3 * it + 2];
    const int cur = it & 1;
    const bool first = (it == 0);
    cudaError_t e;

    // The pair-wide kernel wherever the tile rows come in pairs (n_pad % 256 == 0).
    const bool pair = kUseTwoSm && (n % 256 == 0);

    GemmParams g{};
    g.M = n; g.N = n; g.K = m;
    g.tiles_m = tm_sq; g.tiles_n = S_sq;
    g.tiles_per_matrix = (pair && bn_sq == 256) ? S_sq * (S_sq + 1) / 2 : sym_tiles;
    g.total_tiles = g.tiles_per_matrix * batch;
    g.out = (cc != 0.f) ? a.A : a.B;   // c == 0: the Gram epilogue writes P directly
    g.out_ld = n; g.out_bstride = static_cast<int64_t>(n) * n;
    g.cb = (cc != 0.f) ? 1.f : cb;
    g.cd = (cc != 0.f || x3) ? 0.f : ca - 1.f;   // split-bf16: no (a - 1) I shift
    g.pdiag = (cc != 0.f || x3) ? nullptr : a.pdiag;
    g.pdiag_bstride = n;
    g.kplanes = 1;
    if (x3) {
      g.kplanes = x3_planes; g.a_lo_mask = x3_a_lo; g.b_lo_mask = x3_b_lo;
      g.lo_off = a.sq_lo_off; g.lo_out = 1;
    }
    g.mscale = first ? a.inv_s : nullptr;
    g.status = a.status; g.timeout_ns = a.timeout_ns;
    g.reverse = (launch++ & 1) == 0;
    const int ksplit = (a.partial != nullptr && !pair) ? gram_ksplit(n, m, x3) : 1;
    // polynomial parameters (c != 0)
    GemmParams q = g;
    q.K = n;
    q.out = a.B;
    q.aux = a.A; q.aux_ld = n; q.aux_bstride = static_cast<int64_t>(n) * n;
    q.cb = cb; q.cc = cc; q.cd = x3 ? 0.f : ca - 1.f;
    q.pdiag = x3 ? nullptr : a.pdiag;
    q.mscale = nullptr;
    if (x3) q.lo_in = 1;
    // Gram and polynomial in one launch where both run on CTA pairs (bf16)
    const bool gp_fuse = kFuseGramPoly && !x3 && pair && bn_sq == 256 && cc != 0.f &&
                         a.gp_ctr != nullptr && a.gp_log != nullptr && ksplit == 1 &&
                         gp_launches < kGpMaxLaunches;
    if (gp_fuse) {
      GramPolyParams gp{};
      gp.g = g;
      gp.q = q;
      gp.g.reverse = 0;  // both phases walk forward (the polynomial trails the Gram)
      gp.q.reverse = 0;
      gp.ctr = a.gp_ctr;
      gp.tick = a.gp_tick + gp_launches;
      gp.log = a.gp_log;
      gp.log_cap = g.total_tiles + q.total_tiles + 2;
      gp.stamp = (gp_launches + 1) << 24;
      // a ticket block spans at least a round of tiles on every SM pair; the
      // polynomial trails the Gram by a block only where a block's X and S
      // fit in half of L2 (otherwise the two streams would evict each other:
      // all Gram units first)
      gp.blk = std::max(1, (sm_count() / 2 + g.tiles_per_matrix - 1) / g.tiles_per_matrix);
      const double block_bytes = static_cast<double>(gp.blk) * 2.0 * n * (static_cast<double>(m) + n);
      if (block_bytes > 0.5 * l2_bytes()) gp.blk = batch;
      gp.target = (++gp_launches) * g.tiles_per_matrix * kArrivalsPerUnit;
      e = launch_gram_poly(X[cur].k128, S.k128, S.st, P.st, gp, f_gram + f_poly, st);
      if (e != cudaSuccess) return e;
      launch = 0;  // the update walks backwards, from the matrices the polynomial ended on
    } else if (ksplit > 1 && cc != 0.f && batch <= 65535) {
      // split-K: raw slice sums into the partial buffer, then S and P in one
      // CUDA-core pass
      GemmParams gs = g;
      gs.ksplit = ksplit;
      gs.partial = a.partial;
      gs.total_tiles = g.total_tiles * ksplit;
      gs.reverse = 0;
      e = launch_sym<kEpiGram>(bn_sq, pair, X[cur], S, gs, f_gram, st);
      if (e != cudaSuccess) return e;
      GramReducePolyArgs ra{};
      ra.partial = a.partial;
      ra.ksplit = ksplit;
      ra.batch = batch;
      ra.P = a.B;
      ra.pdiag = a.pdiag;
      ra.mscale = g.mscale;
      ra.cb = cb;
      ra.cc = cc;
      ra.cd = ca - 1.f;
      e = cudaFuncSetAttribute(k_gram_reduce_poly, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kRpSmem));
      if (e != cudaSuccess) return e;
      cudaLaunchConfig_t rc = {};
      cudaLaunchAttribute rattr[1];
      rc.blockDim = dim3(kRpThreads);
      rc.gridDim = dim3(kRpN / kRpRows, static_cast<unsigned>(batch));
      rc.dynamicSmemBytes = kRpSmem;
      rc.stream = st;
      if (kUsePdl) {
        rattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        rattr[0].val.programmaticStreamSerializationAllowed = 1;
        rc.attrs = rattr;
        rc.numAttrs = 1;
      }
      prof_begin(kKindPoly, st);
      e = cudaLaunchKernelEx(&rc, k_gram_reduce_poly, ra);
      prof_end(kKindPoly, st, f_poly, 0.0);
      if (e == cudaSuccess) e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    } else if (ksplit > 1) {
      // split-K: raw slice sums into the partial buffer, then k_gram_reduce
      GemmParams gs = g;
      gs.ksplit = ksplit;
      gs.partial = a.partial;
      gs.total_tiles = g.total_tiles * ksplit;
      gs.reverse = 0;
      e = launch_sym<kEpiGram>(bn_sq, pair, X[cur], (cc != 0.f) ? S : P, gs, f_gram, st);
      if (e != cudaSuccess) return e;
      GramReduceArgs ra{};
      ra.partial = a.partial;
      ra.ksplit = ksplit;
      ra.batch = batch;
      ra.n = n;
      ra.bn = bn_sq;
      ra.out = g.out;
      ra.cb = g.cb;
      ra.cd = g.cd;
      ra.mscale = g.mscale;
      ra.pdiag = g.pdiag;
      cudaLaunchConfig_t rc = {};
      cudaLaunchAttribute rattr[1];
      rc.blockDim = dim3(256);
      const int64_t work = static_cast<int64_t>(batch) * n * (n / 4);
      rc.gridDim = dim3(static_cast<unsigned>(
          std::max<int64_t>(1, std::min<int64_t>((work + 255) / 256, 8 * sm_count()))));
      rc.stream = st;
      if (kUsePdl) {
        rattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        rattr[0].val.programmaticStreamSerializationAllowed = 1;
        rc.attrs = rattr;
        rc.numAttrs = 1;
      }
      prof_begin(kKindGram, st);
      e = cudaLaunchKernelEx(&rc, k_gram_reduce, ra);
      prof_end(kKindGram, st, 0.0, 0.0);
      if (e == cudaSuccess) e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    } else {
      const OperandMaps& gram_out = (cc != 0.f) ? S : P;
      e = x3 ? launch_sym<kEpiGram | kEpiX3>(bn_sq, pair, X[cur], gram_out, g, f_gram, st)
             : launch_sym<kEpiGram>(bn_sq, pair, X[cur], gram_out, g, f_gram, st);
      if (e != cudaSuccess) return e;
    }

    if (cc != 0.f && !gp_fuse && (ksplit == 1 || batch > 65535)) {
      q.reverse = (launch++ & 1) == 0;
      e = x3 ? launch_sym<kEpiPoly | kEpiX3>(bn_sq, pair, S, P, q, f_poly, st)
             : launch_sym<kEpiPoly>(bn_sq, pair, S, P, q, f_poly, st);
      if (e != cudaSuccess) return e;
    }

    GemmParams u{};
    u.M = n; u.N = m; u.K = n;
    u.tiles_m = n / kBM; u.tiles_n = m / bn_up;
    u.tiles_per_matrix = (pair && bn_up == 256) ? (u.tiles_m / 2) * u.tiles_n
                                                : u.tiles_m * u.tiles_n;
    u.total_tiles = u.tiles_per_matrix * batch;
    u.out = xb[cur ^ 1]; u.out_ld = m; u.out_bstride = static_cast<int64_t>(n) * m;
    u.aux = xb[cur]; u.aux_ld = m; u.aux_bstride = static_cast<int64_t>(n) * m;
    u.lo_off = a.lo_off;
    u.ca = 1.f; u.cb = 1.f; u.cc = 0.f; u.cd = 0.f;
    u.pdiag_in = a.pdiag; u.pdiag_bstride = n;
    u.mscale = first ? a.inv_s : nullptr;
    u.status = a.status; u.timeout_ns = a.timeout_ns;
    u.reverse = (launch++ & 1) == 0;
    if (x3) {
      u.kplanes = x3_planes; u.a_lo_mask = x3_a_lo; u.b_lo_mask = x3_b_lo;
      u.lo_in = 1; u.lo_out = 1;
      u.ca = ca;
      e = launch_upd<kEpiUpdate | kEpiX3>(bn_up, pair, P, X[cur], X[cur ^ 1], u, f_update, st);
      if (e != cudaSuccess) return e;
      continue;
    }
    u.kplanes = (it < kResidualIters) ? 2 : 1;   // product reads X hi (and lo)
    u.b_lo_mask = (u.kplanes == 2) ? 0b10 : 0;
    u.lo_in = it < kLoIters;
    u.lo_out = it + 1 < kLoIters;
    u.clo = (u.kplanes == 1 && u.lo_in) ? ca - 1.f : 0.f;
    if ((it + 1 == a.iters) && a.fin.mode != 0) {
      // the last update writes W (or the output); it has no lo plane
      u.fin = a.fin;
      u.lo_in = false;
      u.lo_out = false;
      bool any_tall = false;
      for (int k = 0; k < a.fin.nseg; ++k) any_tall = any_tall || a.fin.seg[k].tall != 0;
      e = any_tall ? launch_upd<kEpiFinal | kEpiTall>(bn_up, pair, P, X[cur], X[cur ^ 1], u, f_update, st)
                   : launch_upd<kEpiFinal>(bn_up, pair, P, X[cur], X[cur ^ 1], u, f_update, st);
    } else {
      e = launch_upd<kEpiUpdate>(bn_up, pair, P, X[cur], X[cur ^ 1], u, f_update, st);
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace muon
