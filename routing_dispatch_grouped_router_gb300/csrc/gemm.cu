// Persistent grouped-GEMM engine on tcgen05 (sm_103a) for the experts' SwiGLU
// FFN: forward gate/up + SwiGLU, forward down, and the backward dgrad/wgrad
// GEMMs, plus the router logit GEMM.
//
// Sources (page title, section):
//   [gtnt] "MoK揭秘：NVL72上大规模MoE训练工程方案深度解读", §1.3 and §2.2: the
//     many small per-expert GEMMs are run as one grouped GEMM so the tensor
//     cores stay busy.
//   [dothoosh] "Cursor Mixture-of-Kittens cuts MoE training latency by 5.8x",
//     "MoK technical details", bullet "Overlap granularity": every
//     expert-grouped GEMM is given at least two full waves of SMs; bullet
//     "Precision and scheduling": BF16 GEMMs, SwiGLU backward fused with the
//     router-weight gradient.
//
// Design (one CTA per SM, 320 threads):
//   warp 0      TMA producer: 128B-swizzled tiles of A (128 x 64) and B
//               (BN x 64) into a STAGES-deep shared-memory ring (mbarriers).
//   warp 1      TMEM owner and MMA issuer: one thread issues
//               tcgen05.mma.kind::f16 (M=128, N=BN, K=16) x 4 per stage into
//               one of two fp32 accumulators in TMEM (2*BN columns), and
//               commits stage release / accumulator-ready to mbarriers.
//   warps 2..9  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM
//               lanes 32*(w%4).., columns half (w-2)/4), fused math, stores.
//               fp32 results leave through a per-warp 4 KB swizzled staging
//               buffer and a TMA tensor store (32 x 32 box), so HBM sees whole
//               128-byte lines.  Double-buffered accumulators let tile i's
//               epilogue overlap tile i+1's MMAs.
// Tiles are walked in a static round-robin (tile = blockIdx.x + i*gridDim.x),
// every tile is computed by exactly one CTA with a fixed K order, so results
// are bitwise reproducible.  Per-expert tile tables come from the dispatch
// plan (prefix sums of 128-row tiles), read on the device: the host never
// waits for routing results.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "mok_internal.h"
#include "mx.cuh"
#include "ptx.cuh"

namespace mok {

enum Sched : int { SCHED_DENSE = 0, SCHED_MGROUP = 1, SCHED_KGROUP = 2 };
enum Epi : int {
  EPI_BF16 = 0,
  EPI_F32 = 1,
  EPI_SWIGLU_FWD = 2,
  EPI_SWIGLU_BWD = 3,
  EPI_F32_T = 4,  // KGROUP: fp32 C^T through TMA (the tile is stored transposed)
  EPI_BF16_TMA = 5,  // KGROUP: C rounded to bf16, through TMA
  EPI_BF16_T = 6,    // KGROUP: C^T rounded to bf16, through TMA
};
// Split operands: a bf16 "hi" tile plus a bf16 "lo" tile (value - hi) whose
// products are accumulated into the same fp32 accumulator, giving the GEMM
// an operand with ~16 significant bits.
// SPLIT_MX: not a split but the MXFP8 operand mode: A and B are E4M3 codes
// (K-major, 128 K values per stage) with one E8M0 scale byte per 32 K values,
// multiplied by tcgen05.mma.kind::mxf8f6f4.block_scale (single CTA, BN=128).
// SPLIT_NV: the NVFP4 operand mode (CTA pairs only): A and B are packed E2M1
// codes (K-major, 256 K values = 128 bytes per stage) with one E4M3 scale per
// 16 K values, multiplied by tcgen05.mma.kind::mxf4nvf4.block_scale
// (scale_vec::4X); the tensor scales of A and B multiply the accumulator in
// the epilogue.
enum Split : int { SPLIT_NONE = 0, SPLIT_A = 1, SPLIT_B = 2, SPLIT_MX = 3, SPLIT_NV = 4 };
constexpr bool block_scaled(int split) { return split == SPLIT_MX || split == SPLIT_NV; }

struct GemmArgs {
  int E;             // groups (experts); 1 for dense
  int m_tiles;       // DENSE/KGROUP: 128-row tiles of M
  int n_tiles;       // N tiles
  int num_kb;        // DENSE/MGROUP: K / 64
  int b_group_rows;  // MGROUP: rows of B per expert in its 2-D view
  int m_rows;        // KGROUP: rows of C per group (C viewed as [E*m_rows, N])
  int I;             // SwiGLU epilogues: FFN width
  int m_valid, n_valid;  // valid rows / columns of C (DENSE; M- and K-grouped: 0 = all)
  const int* mtile_prefix;  // MGROUP: [E+1] prefix of 128-row tiles per expert, then
                            // [E+1] prefix of tile pairs (an odd count rounded up)
  const int* poff;          // MGROUP/KGROUP: [E+1] padded row offsets
  void* out;                // C (bf16 or fp32)
  long long ldo;            // C row stride (elements)
  long long out_group_stride;  // KGROUP: elements between experts' C
  void* out2;               // SWIGLU_FWD: H [rows,I] (NULL: not stored); SWIGLU_BWD: P_hi = bf16(p*h) [rows,I]
  void* out3;               // SWIGLU_BWD: dGU_lo [rows,2I]
  void* out4;               // SWIGLU_BWD: P_lo [rows,I]
  uint8_t* dgu_codes;       // SWIGLU_BWD with mx: dG, dU as E4M3 codes [rows,2I] (dgrad operand)
  uint8_t* dgu_scales;      // ... and its E8M0 bytes (tiled layout, mx_tiled_off)
  int mx;                   // SwiGLU epilogues: quantise the derived GEMM operands to MXFP8
  const uint8_t* sa;        // SPLIT_MX: A scale bytes, tiled layout (mx_tiled_off)
  const uint8_t* sb;        // SPLIT_MX: B scale bytes, tiled layout
  int ks;                   // SPLIT_MX: K / 32 (scale bytes per row); SPLIT_NV: K / 64
  const float* ga;          // SPLIT_NV: device tensor scale of A
  const float* gb;          // SPLIT_NV: device tensor scale of B
  uint8_t* h_codes;         // SWIGLU_FWD with SPLIT_MX: h as E4M3 codes [rows, I] (NULL: none)
  uint8_t* h_scales;        // ... and its E8M0 bytes (tiled layout, mx_tiled_off)
  int accumulate;           // fp32 TMA-store epilogue: add into C instead of overwriting
  int store_c;              // SWIGLU_FWD: write g, u through the C map
  int evict_first;          // TMA-store epilogues: C is not read again soon (L2 evict-first)
  int k_splits;             // DENSE: K split into this many partial products (0 or 1: none)
  const void* in_gu;        // SWIGLU_BWD: saved fp32 pre-activations [rows,2I]
  const float* row_w;       // SWIGLU_BWD: routing weight of each row
  float* dp_part;           // SWIGLU_BWD: [rows, np] partial <dA,h>
  int np;
  // KGROUP over several row spaces (deferred weight gradients of a micro-
  // batched backward): segment s of expert e is rows [poff_s[e], poff_s[e+1])
  // of row space s, poff_s = poff + s*poff_stride, at operand row s*seg_rows.
  // The K loop runs through the segments in order.  nseg <= 1: one row space.
  int nseg;
  int poff_stride;
  int seg_rows;
  // KGROUP: [E+1] real (unpadded) row offsets in the same layout as poff, or
  // NULL.  Given, the K loop of expert e in a row space covers its real rows
  // rounded up to a 64-row block instead of its 128-padded rows: the padding
  // rows of every weight-gradient operand are zero, so the skipped products
  // are exact zeros and the sums do not change.
  // MGROUP: the same offsets, or NULL.  Given, the rows of expert e past its
  // real rows rounded up to 64 (the plan's token -2 rows, which only whole-
  // tile GEMMs read, for output rows nothing reads) get no epilogue: no
  // operand loads, no stores, whole 32-row quarters.
  const int* coff;
  int* status;
};

// Extra output maps: the SwiGLU backward stores dG/dU (hi, lo) and p*h (hi,
// lo) through TMA, boxes of 32 rows x 16 bf16 columns.
// MXFP8 on CTA pairs: the A and B scales (tiled layout) viewed as rows of 256
// bytes, one 512-byte block = 2 rows.
struct OutMaps {
  CUtensorMap dgu_hi, dgu_lo, p_hi, p_lo;
  CUtensorMap sfa, sfb;
  // SwiGLU forward with bf16 h: h [rows, I], 32 x 32 blocks of 64-byte rows
  // (64-byte swizzle); a zeroed map (no h, or h as MXFP8 codes) is unused
  CUtensorMap h;
};

constexpr int kThreads = 320;
constexpr int kEpiWarps = 8;
constexpr int kStagingBytes = 4096;  // per epilogue warp: 32 rows x 128 bytes

// PAIR: the tile is 256 x BN, computed by a cluster of two CTAs with
// tcgen05.mma.cta_group::2; each CTA stages its own 128 rows of A and BN/2
// rows of B, and holds its 128 x BN accumulator in its own TMEM.
// Staging bytes per epilogue warp: 4 KB (TMA-store blocks); the SwiGLU
// backward stages its fp32 g, u operands in one 4 KB buffer (the next chunk's
// copies go out as soon as the warp holds the current one in registers) and
// the six bf16 output blocks of a chunk (6 x 1 KB).  One g, u buffer instead
// of two gives the pair kernel a fourth operand stage (imbalanced workload:
// 1922 -> 1679 us; fine 255 -> 252 us).
constexpr int kGuBufBytes = 4096;
constexpr int kSwigluBwdStaging = kGuBufBytes + 6 * 1024;
// The SwiGLU backward with its outputs stored straight from registers (DB on
// EPI_SWIGLU_BWD): no output staging, so two more operand stages.  Faster
// where the K loop (d) is long and the weights stream: large workload,
// d = 7168, 3117 -> 2977 us; slower where the epilogue dominates: fine,
// d = 2048, 257 -> 327 us (16-byte stores, half a sector per lane and store).
// This form keeps two g, u buffers (chunk n + 1's copies in flight while
// chunk n waits): with one, and a sixth operand stage, it measured slower
// (2977 -> 3211 us).
constexpr int kSwigluBwdStagingDirect = 2 * kGuBufBytes;
constexpr int kSwigluBwdDirectMinD = 6144;
// Double-buffered store staging (DB: a block is written while the previous
// block's store still reads shared memory), chosen per launch for the fp32
// weight gradients (K-grouped, plain and transposed stores) whose tiles run
// few K blocks (short_k_wgrad): there the epilogue's store chain, not the
// MMAs, sets the pace (large workload: 29.7 -> 29.0 ms per step), while with
// long K loops the operand stage it costs matters more (fine workload: the
// gate/up weight gradient 366 -> 419 us with it).  Off for the M-grouped
// GEMMs: it costs the 256-wide pair kernels their sixth operand stage, and
// measured slower there (fwd_gate_up 245 -> 260 us, fwd_down 132 -> 151 us on
// the fine workload), as it did for the block-scaled pairs' register epilogues
// (their fifth stage: NVFP4 fwd_down 713 -> 805 us).
template <int EPI, int SPLIT, int SCHED, bool DB>
constexpr int staging_bytes() {
  return EPI == EPI_SWIGLU_BWD ? (DB ? kSwigluBwdStagingDirect : kSwigluBwdStaging)
                               : (DB ? 2 * kStagingBytes : kStagingBytes);
}

template <int BN, int SPLIT = SPLIT_NONE, bool PAIR = false, int STG = kStagingBytes>
struct Cfg {
  static constexpr int BM = 128, BK = 64;
  static constexpr int B_ROWS = PAIR ? BN / 2 : BN;  // rows of B staged by one CTA
  static constexpr int A_BYTES = BM * BK * 2;        // 16 KB
  static constexpr int B_BYTES = B_ROWS * BK * 2;    // 32 KB (BN=256) / 16 KB (BN=128 or PAIR)
  static constexpr int A_TILES = SPLIT == SPLIT_A ? 2 : 1;
  static constexpr int B_TILES = SPLIT == SPLIT_B ? 2 : 1;
  static constexpr int B_OFF = A_TILES * A_BYTES;  // B tile(s) follow the A tile(s)
  // SPLIT_MX: 128-row x 128-byte code tiles (the bf16 tile sizes) and the two
  // 512-byte scale blocks of the stage (A's 128 rows, B's 128 rows)
  static constexpr int SF_OFF = A_TILES * A_BYTES + B_TILES * B_BYTES;
  // (CTA pairs: the CTA's 128 A rows, and all 256 B rows of the pair's tile)
  // SPLIT_NV (pairs): four 512-byte blocks per 128 rows (one per K = 64 MMA):
  // 2 KB for the CTA's A rows, 4 KB for the 256 B rows
  static constexpr int SF_BYTES =
      SPLIT == SPLIT_MX ? (PAIR ? 1536 : 1024) : (SPLIT == SPLIT_NV ? 6144 : 0);
  static constexpr int STAGE_BYTES =
      block_scaled(SPLIT) ? (SF_OFF + SF_BYTES + 1023) / 1024 * 1024 : SF_OFF;
  // accumulators; block-scaled pairs keep one (256 columns) so that the
  // stages' scale columns fit beside it (MXFP8: 12 per stage, 4 for A and 8
  // for B; NVFP4: 48, 16 for A and 32 for B)
  static constexpr int NACC = (block_scaled(SPLIT) && PAIR) ? 1 : 2;
  static constexpr int SF_COLS =
      SPLIT == SPLIT_MX ? (PAIR ? 12 : 8) : (SPLIT == SPLIT_NV ? 48 : 0);
  static constexpr int BAR_BYTES = 512;
  static constexpr int STAGE_ROOM = 232448 - 1024 - BAR_BYTES - kEpiWarps * STG;
  static constexpr int STAGES = (STAGE_ROOM / STAGE_BYTES) < 6 ? (STAGE_ROOM / STAGE_BYTES) : 6;
  // SPLIT_MX: after the accumulators, 8 columns of scales per stage
  static constexpr int TMEM_COLS = block_scaled(SPLIT) ? 512 : 2 * BN;
  static constexpr int STAGING_OFF = STAGES * STAGE_BYTES;
  static constexpr int STAGING_PER_WARP = STG;
  static constexpr int BAR_OFF = STAGING_OFF + kEpiWarps * STG;
  static constexpr int SMEM_BYTES = 1024 + BAR_OFF + BAR_BYTES;
};
static_assert(Cfg<256>::SMEM_BYTES <= 232448, "smem");
static_assert(Cfg<128>::SMEM_BYTES <= 232448, "smem");
static_assert(Cfg<256, SPLIT_A>::SMEM_BYTES <= 232448 && Cfg<256, SPLIT_A>::STAGES >= 3, "smem");
static_assert(Cfg<128, SPLIT_B>::SMEM_BYTES <= 232448 && Cfg<128, SPLIT_B>::STAGES >= 4, "smem");
static_assert(Cfg<256, SPLIT_NONE, true>::SMEM_BYTES <= 232448 &&
                  Cfg<256, SPLIT_NONE, true>::STAGES == 6, "smem");
static_assert(Cfg<256, SPLIT_A, true>::SMEM_BYTES <= 232448 &&
                  Cfg<256, SPLIT_A, true>::STAGES >= 4, "smem");
static_assert(Cfg<256, SPLIT_NONE, true, kSwigluBwdStaging>::SMEM_BYTES <= 232448 &&
                  Cfg<256, SPLIT_NONE, true, kSwigluBwdStaging>::STAGES == 4 &&
                  Cfg<256, SPLIT_NONE, true, kSwigluBwdStagingDirect>::STAGES == 5, "smem");
static_assert(Cfg<256, SPLIT_NONE, false, kSwigluBwdStaging>::STAGES >= 2 &&
                  Cfg<128, SPLIT_NONE, false, kSwigluBwdStaging>::STAGES >= 3, "smem");
static_assert(Cfg<128, SPLIT_MX>::STAGES == 5 && Cfg<128, SPLIT_MX>::STAGE_BYTES % 1024 == 0 &&
                  2 * 128 + 8 * Cfg<128, SPLIT_MX>::STAGES <= 512,
              "MXFP8 stages");
static_assert(Cfg<256, SPLIT_NV, true>::STAGES == 5 &&
                  Cfg<256, SPLIT_NV, true>::STAGE_BYTES % 1024 == 0 &&
                  256 + 48 * Cfg<256, SPLIT_NV, true>::STAGES <= 512,
              "NVFP4 pair stages");
static_assert(Cfg<256, SPLIT_MX, true>::STAGES == 5 &&
                  Cfg<256, SPLIT_MX, true>::STAGE_BYTES % 1024 == 0 &&
                  256 + 12 * Cfg<256, SPLIT_MX, true>::STAGES <= 512,
              "MXFP8 pair stages");
static_assert(Cfg<256, SPLIT_NONE, true, 2 * kStagingBytes>::STAGES == 5 &&
                  Cfg<256, SPLIT_NONE, false, 2 * kStagingBytes>::STAGES == 3 &&
                  Cfg<128, SPLIT_NONE, false, 2 * kStagingBytes>::STAGES == 5,
              "stages with double-buffered store staging");
// stage counts of the other configurations are unchanged by the 512-byte barrier block
static_assert(Cfg<256>::STAGES == 4 && Cfg<128>::STAGES == 6 && Cfg<256, SPLIT_A>::STAGES == 3 &&
                  Cfg<128, SPLIT_B>::STAGES == 4 && Cfg<256, SPLIT_NONE, true>::STAGES == 6 &&
                  Cfg<256, SPLIT_A, true>::STAGES == 4,
              "stages");

struct Tile {
  int e, m_tile, n_tile;
  int row0;    // MGROUP/DENSE: first row of A and C; KGROUP: first row of C_e
  int k_row0;  // KGROUP: first K row (padded offset of the expert)
  int num_kb;
  int kb0;     // DENSE with split K: first K block of this split (e = the split)
};

template <int SCHED>
__device__ __forceinline__ int total_tiles(const GemmArgs& a) {
  if (SCHED == SCHED_MGROUP) return __ldg(a.mtile_prefix + a.E) * a.n_tiles;
  if (SCHED == SCHED_KGROUP) return a.E * a.m_tiles * a.n_tiles;
  return a.m_tiles * a.n_tiles * (a.k_splits > 1 ? a.k_splits : 1);
}

// K blocks of expert e in row space s of a KGROUP launch: its real rows
// rounded up to 64 when the real offsets are given, else its padded rows.
__device__ __forceinline__ int seg_kb(const GemmArgs& a, int s, int e) {
  const long long o = static_cast<long long>(s) * a.poff_stride;
  if (a.coff) return (__ldg(a.coff + o + e + 1) - __ldg(a.coff + o + e) + 63) / 64;
  return (__ldg(a.poff + o + e + 1) - __ldg(a.poff + o + e)) / 64;
}

// K blocks of expert e over all row spaces of a KGROUP launch.
__device__ __forceinline__ int kgroup_kb(const GemmArgs& a, int e) {
  const int ns = a.nseg > 1 ? a.nseg : 1;
  int n = 0;
  for (int s = 0; s < ns; ++s) n += seg_kb(a, s, e);
  return n;
}

// Walks a KGROUP K loop through its segments: the operand row of K block kb.
struct SegWalk {
  int seg, first_kb, nkb, row;
  __device__ __forceinline__ void load(const GemmArgs& a, int e) {
    const int* p = a.poff + static_cast<long long>(seg) * a.poff_stride;
    nkb = seg_kb(a, seg, e);
    row = seg * a.seg_rows + __ldg(p + e);
  }
  __device__ __forceinline__ void init(const GemmArgs& a, int e) {
    seg = 0;
    first_kb = 0;
    load(a, e);
  }
  // kb below the expert's total: the loop ends within its segments
  __device__ __forceinline__ int row_of(const GemmArgs& a, int e, int kb) {
    while (kb >= first_kb + nkb) {
      first_kb += nkb;
      ++seg;
      load(a, e);
    }
    return row + (kb - first_kb) * 64;
  }
};

// Tiles of 256 rows for CTA pairs: MGROUP pairs the 128-row tiles of one
// expert (2j, 2j+1); when an expert has an odd number, the odd CTA of its
// last pair stages the even CTA's rows again and stores nothing (*valid =
// false).  KGROUP pairs the 128-row tiles of C (their number is even).
template <int SCHED>
__device__ __forceinline__ int total_pairs(const GemmArgs& a) {
  if (SCHED == SCHED_MGROUP) return __ldg(a.mtile_prefix + 2 * a.E + 1) * a.n_tiles;
  return a.E * (a.m_tiles / 2) * a.n_tiles;
}

template <int SCHED>
__device__ __forceinline__ Tile decode_pair(const GemmArgs& a, int t, int rank, bool* valid) {
  Tile tl;
  if (SCHED == SCHED_MGROUP) {
    const int* pre = a.mtile_prefix + a.E + 1;
    int lo = 0, hi = a.E;  // invariant: pre[lo]*nt <= t < pre[hi]*nt
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(pre + mid) * a.n_tiles <= t) lo = mid; else hi = mid;
    }
    const int e = lo;
    const int q0 = __ldg(pre + e);
    const int np_e = __ldg(pre + e + 1) - q0;
    const int local = t - q0 * a.n_tiles;
    const int mt_e = __ldg(a.mtile_prefix + e + 1) - __ldg(a.mtile_prefix + e);
    tl.e = e;
    tl.n_tile = local / np_e;
    const int pair = local - tl.n_tile * np_e;
    int m = 2 * pair + rank;
    *valid = m < mt_e;
    if (!*valid) m = 2 * pair;
    tl.m_tile = m;
    tl.row0 = __ldg(a.poff + e) + m * 128;
    tl.k_row0 = 0;
    tl.num_kb = a.num_kb;
    tl.kb0 = 0;
  } else {
    const int mp = a.m_tiles / 2;
    const int tpe = mp * a.n_tiles;
    const int e = t / tpe;
    const int local = t - e * tpe;
    tl.e = e;
    tl.n_tile = local / mp;
    tl.m_tile = 2 * (local - tl.n_tile * mp) + rank;
    tl.row0 = tl.m_tile * 128;
    tl.k_row0 = __ldg(a.poff + e);
    tl.num_kb = kgroup_kb(a, e);
    tl.kb0 = 0;
    *valid = true;
  }
  return tl;
}

template <int SCHED>
__device__ __forceinline__ Tile decode_tile(const GemmArgs& a, int t) {
  Tile tl;
  if (SCHED == SCHED_MGROUP) {
    // largest e with prefix[e] * n_tiles <= t (empty experts are skipped)
    const int* pre = a.mtile_prefix;
    int lo = 0, hi = a.E;  // invariant: pre[lo]*nt <= t < pre[hi]*nt
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(pre + mid) * a.n_tiles <= t) lo = mid; else hi = mid;
    }
    const int e = lo;
    const int p0 = __ldg(pre + e);
    const int mt_e = __ldg(pre + e + 1) - p0;
    const int local = t - p0 * a.n_tiles;
    tl.e = e;
    tl.n_tile = local / mt_e;
    tl.m_tile = local - tl.n_tile * mt_e;
    tl.row0 = __ldg(a.poff + e) + tl.m_tile * 128;
    tl.k_row0 = 0;
    tl.num_kb = a.num_kb;
    tl.kb0 = 0;
  } else if (SCHED == SCHED_KGROUP) {
    const int tpe = a.m_tiles * a.n_tiles;
    const int e = t / tpe;
    const int local = t - e * tpe;
    tl.e = e;
    tl.n_tile = local / a.m_tiles;
    tl.m_tile = local - tl.n_tile * a.m_tiles;
    tl.row0 = tl.m_tile * 128;
    tl.k_row0 = __ldg(a.poff + e);
    tl.num_kb = kgroup_kb(a, e);
    tl.kb0 = 0;
  } else {
    // DENSE: split-K partial products go to separate C blocks (e = split)
    const int mn = a.m_tiles * a.n_tiles;
    const int split = t / mn;
    const int tt = t - split * mn;
    tl.e = split;
    tl.n_tile = tt / a.m_tiles;
    tl.m_tile = tt - tl.n_tile * a.m_tiles;
    tl.row0 = tl.m_tile * 128;
    tl.k_row0 = 0;
    tl.num_kb = a.num_kb;
    tl.kb0 = split * a.num_kb;
  }
  return tl;
}

// silu(g) = g * sigmoid(g); the sigmoid through the hardware exponential and a
// correctly rounded reciprocal.
__device__ __forceinline__ float silu_f(float g, float* sig_out) {
  const float s = __frcp_rn(1.0f + __expf(-g));
  *sig_out = s;
  return g * s;
}

// ---------------------------------------------------------------- epilogues --

// Loads 32 consecutive accumulator columns (two x16 loads, one wait).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r0[16], r1[16];
  tmem_ld16(taddr, r0);
  tmem_ld16(taddr + 16, r1);
  tmem_ld_wait();
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    v[j] = __uint_as_float(r0[j]);
    v[16 + j] = __uint_as_float(r1[j]);
  }
}

__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* p, const float (&v)[32]) {
  uint4 w[4];
  uint32_t* u = reinterpret_cast<uint32_t*>(w);
#pragma unroll
  for (int j = 0; j < 16; ++j) u[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
  uint4* q = reinterpret_cast<uint4*>(p);
#pragma unroll
  for (int j = 0; j < 4; ++j) q[j] = w[j];
}

__device__ __forceinline__ void load_bf16x32(const __nv_bfloat16* p, float (&v)[32]) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 w = q[j];
    v[8 * j + 0] = bf16lo(w.x); v[8 * j + 1] = bf16hi(w.x);
    v[8 * j + 2] = bf16lo(w.y); v[8 * j + 3] = bf16hi(w.y);
    v[8 * j + 4] = bf16lo(w.z); v[8 * j + 5] = bf16hi(w.z);
    v[8 * j + 6] = bf16lo(w.w); v[8 * j + 7] = bf16hi(w.w);
  }
}

// Stores 16 values as bf16 hi = bf16(v) and lo = bf16(v - hi).
__device__ __forceinline__ void store_hi_lo16(__nv_bfloat16* hi, __nv_bfloat16* lo,
                                              const float (&v)[16]) {
  uint4* ph = reinterpret_cast<uint4*>(hi);
  uint4* pl = reinterpret_cast<uint4*>(lo);
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float v0 = v[8 * q + 2 * j], v1 = v[8 * q + 2 * j + 1];
      const float a0 = bf16_round(v0), a1 = bf16_round(v1);
      h[j] = pack_bf16x2(a0, a1);
      l[j] = pack_bf16x2(v0 - a0, v1 - a1);
    }
    ph[q] = make_uint4(h[0], h[1], h[2], h[3]);
    pl[q] = make_uint4(l[0], l[1], l[2], l[3]);
  }
}

// One warp writes its 32 rows x 32 fp32 columns to the 4 KB staging buffer in
// the 128-byte swizzled layout (16-byte chunk j of row r at chunk j ^ (r%8)),
// then lane 0 stores it with one TMA tensor store at (x, y).
// Lane 0: the TMA store (or reduce-add) of one staged block, with an
// evict-first L2 policy for output that is not read again soon.
__device__ __forceinline__ void tma_out_2d(const CUtensorMap* tmC, const void* buf, int x, int y,
                                           bool add, bool evict_first) {
  if (evict_first) {
    const uint64_t pol = l2_policy_evict_first();
    if (add) tma_reduce_add_2d_hint(tmC, buf, x, y, pol);
    else tma_store_2d_hint(tmC, buf, x, y, pol);
  } else {
    if (add) tma_reduce_add_2d(tmC, buf, x, y);
    else tma_store_2d(tmC, buf, x, y);
  }
  bulk_commit();
}

// DBUF: `base` holds two buffers used alternately (n counts this warp's
// stores); a buffer is rewritten once the store two back has read it.
template <bool DBUF = false>
__device__ __forceinline__ void stage_and_store_f32(uint8_t* base, uint32_t& n,
                                                    const CUtensorMap* tmC,
                                                    const float (&v)[32], int lane, int x, int y,
                                                    bool add = false, bool evict_first = false) {
  uint8_t* buf = DBUF ? base + (n & 1u) * kStagingBytes : base;
  ++n;
  if (lane == 0) {  // the store that last used this buffer has read it
    if (DBUF) bulk_wait_read<1>();
    else bulk_wait_read<0>();
  }
  __syncwarp();
  uint8_t* row = buf + lane * 128;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int pj = j ^ (lane & 7);
    *reinterpret_cast<float4*>(row + pj * 16) =
        make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) tma_out_2d(tmC, buf, x, y, add, evict_first);
}

// As stage_and_store_f32, but the warp's 32 x 32 block is stored transposed:
// lane i holds row i of the accumulator block (v[j] = column j), and the
// staging buffer receives column j of the block as its row j, so the TMA store
// at (x, y) writes element (i, j) to output row y + j, column x + i.
// DBUF: `base` holds two buffers used alternately (as stage_and_store_f32).
template <bool DBUF = false>
__device__ __forceinline__ void stage_and_store_f32_t(uint8_t* base, uint32_t& n,
                                                      const CUtensorMap* tmC,
                                                      const float (&v)[32], int lane, int x,
                                                      int y, bool add, bool evict_first) {
  uint8_t* buf = DBUF ? base + (n & 1u) * kStagingBytes : base;
  ++n;
  if (lane == 0) {  // the store that last used this buffer has read it
    if (DBUF) bulk_wait_read<1>();
    else bulk_wait_read<0>();
  }
  __syncwarp();
  const int chunk = lane >> 2, word = (lane & 3) * 4;
#pragma unroll
  for (int j = 0; j < 32; ++j)
    *reinterpret_cast<float*>(buf + j * 128 + ((chunk ^ (j & 7)) << 4) + word) = v[j];
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) tma_out_2d(tmC, buf, x, y, add, evict_first);
}

// As stage_and_store_f32, but a 32 x 64 block (columns x .. x+63: v0 then
// v1) is rounded to bf16 (nearest even) and stored as 128-byte rows, in the
// same 128B-swizzled layout (16-byte chunk j of row r at chunk j ^ (r % 8)).
__device__ __forceinline__ void stage_and_store_bf16(uint8_t* buf, const CUtensorMap* tmC,
                                                     const float (&v0)[32], const float (&v1)[32],
                                                     int lane, int x, int y, bool evict_first) {
  if (lane == 0) bulk_wait_read<0>();
  __syncwarp();
  uint8_t* row = buf + lane * 128;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float* v = j < 4 ? v0 + 8 * j : v1 + 8 * (j - 4);
    *reinterpret_cast<uint4*>(row + ((j ^ (lane & 7)) << 4)) =
        make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                   pack_bf16x2(v[6], v[7]));
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) tma_out_2d(tmC, buf, x, y, false, evict_first);
}

// The transposed form (see stage_and_store_f32_t) in bf16: staging row j is
// column j of the block, lane i's element at 16-byte chunk (i / 8) ^ ((j >> 1)
// & 3), byte 2 * (i % 8).
__device__ __forceinline__ void stage_and_store_bf16_t(uint8_t* buf, const CUtensorMap* tmC,
                                                       const float (&v)[32], int lane, int x,
                                                       int y, bool evict_first) {
  if (lane == 0) bulk_wait_read<0>();
  __syncwarp();
  const int chunk = lane >> 3, off = (lane & 7) * 2;
#pragma unroll
  for (int j = 0; j < 32; ++j)
    *reinterpret_cast<__nv_bfloat16*>(buf + j * 64 + ((chunk ^ ((j >> 1) & 3)) << 4) + off) =
        __float2bfloat16_rn(v[j]);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) tma_out_2d(tmC, buf, x, y, false, evict_first);
}

// A warp's 32 rows x 32 values rounded to bf16 (nearest even), lane i
// holding row i: staging row i is 64 bytes in the 64-byte-swizzled layout
// (16-byte chunk j of row r at chunk j ^ ((r >> 1) & 3)), stored with one TMA
// store at (x, y): whole 32-byte sectors instead of one lane's 16-byte
// pieces of 32 rows per store instruction.
__device__ __forceinline__ void stage_and_store_bf16_rows32(uint8_t* buf, const CUtensorMap* tm,
                                                            const float (&v)[32], int lane,
                                                            int x, int y) {
  if (lane == 0) bulk_wait_read<0>();  // earlier stores have read the staging
  __syncwarp();
  uint8_t* row = buf + lane * 64;
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    *reinterpret_cast<uint4*>(row + ((j ^ sw) << 4)) =
        make_uint4(pack_bf16x2(v[8 * j], v[8 * j + 1]), pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                   pack_bf16x2(v[8 * j + 4], v[8 * j + 5]),
                   pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tm, buf, x, y);
    bulk_commit();
  }
}

template <int BN, int SCHED, int EPI, bool DBUF, int SPLIT>
__device__ __forceinline__ void epilogue_tile(const GemmArgs& a, const Tile& tl, uint32_t taddr,
                                              int q, int lane, int half, uint8_t* stage_buf,
                                              uint32_t& nst, const CUtensorMap* tmC,
                                              const CUtensorMap* tmH) {
  constexpr int HALF_COLS = BN / 2;
  const int row_in_tile = q * 32 + lane;
  const bool zero_k = (tl.num_kb == 0);
  // NVFP4: the product of the operands' tensor scales (the block scales were
  // applied by the tensor cores)
  const float alpha = SPLIT == SPLIT_NV ? __ldg(a.ga) * __ldg(a.gb) : 1.0f;
  if ((EPI == EPI_F32 || EPI == EPI_BF16_TMA) && SCHED != SCHED_DENSE) {
    // fp32 (or bf16) C through TMA stores; C viewed as 2-D [rows, N]
    const int y = (SCHED == SCHED_KGROUP ? tl.e * a.m_rows : 0) + tl.row0 + q * 32;
    const int col0 = tl.n_tile * BN + half * HALF_COLS;
    // a ragged last tile (M or N a multiple of 32, not of the tile): this
    // warp's 32 rows and each 32-column chunk lie wholly inside or outside C,
    // and what lies outside belongs to the next expert's block or past C, so
    // it is not stored
    if (a.m_valid > 0 && tl.row0 + q * 32 >= a.m_valid) return;
    if constexpr (EPI == EPI_BF16_TMA) {
      // 64 columns per store: 128-byte rows
#pragma unroll 1
      for (int c = 0; c < HALF_COLS; c += 64) {
        if (a.n_valid > 0 && col0 + c >= a.n_valid) break;  // (a partial box is clipped)
        float v0[32], v1[32];
        if (!zero_k) {
          tmem_ld32(taddr + half * HALF_COLS + c, v0);
          tmem_ld32(taddr + half * HALF_COLS + c + 32, v1);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v0[j] = v1[j] = 0.f;
        }
        stage_and_store_bf16(stage_buf, tmC, v0, v1, lane, col0 + c, y, a.evict_first != 0);
      }
    } else {
#pragma unroll 1
      for (int c = 0; c < HALF_COLS; c += 32) {
        if (a.n_valid > 0 && col0 + c >= a.n_valid) break;
        float v[32];
        if (!zero_k) {
          tmem_ld32(taddr + half * HALF_COLS + c, v);
          if (SPLIT == SPLIT_NV) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] *= alpha;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0.f;
        }
        stage_and_store_f32<DBUF>(stage_buf, nst, tmC, v, lane, col0 + c, y, a.accumulate != 0,
                                  a.evict_first != 0);
      }
    }
  } else if (EPI == EPI_F32_T || EPI == EPI_BF16_T) {
    // C^T through TMA: accumulator rows are output columns; C viewed as
    // [E * N, M] with group e's block at rows e*N
    const int x = tl.row0 + q * 32;
    if (a.m_valid > 0 && x >= a.m_valid) return;  // a ragged M tile (M a multiple of 32)
    const int col0 = tl.n_tile * BN + half * HALF_COLS;
#pragma unroll 1
    for (int c = 0; c < HALF_COLS; c += 32) {
      float v[32];
      if (!zero_k) {
        tmem_ld32(taddr + half * HALF_COLS + c, v);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0.f;
      }
      if (EPI == EPI_BF16_T)
        stage_and_store_bf16_t(stage_buf, tmC, v, lane, x, tl.e * a.ldo + col0 + c,
                               a.evict_first != 0);
      else
        stage_and_store_f32_t<DBUF>(stage_buf, nst, tmC, v, lane, x, tl.e * a.ldo + col0 + c,
                              a.accumulate != 0, a.evict_first != 0);
    }
  } else if (EPI == EPI_BF16 || EPI == EPI_F32) {
    constexpr int esz = EPI == EPI_F32 ? 4 : 2;
    const long long grow = tl.row0 + row_in_tile;
    char* base = static_cast<char*>(a.out);
    if (SCHED != SCHED_MGROUP) base += (long long)tl.e * a.out_group_stride * esz;
    const bool row_ok = (SCHED != SCHED_DENSE) || grow < a.m_valid;
    const int col0 = tl.n_tile * BN + half * HALF_COLS;
#pragma unroll 1
    for (int c = 0; c < HALF_COLS; c += 32) {
      float v[32];
      if (!zero_k) {
        tmem_ld32(taddr + half * HALF_COLS + c, v);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0.f;
      }
      if (!row_ok) continue;
      if (EPI == EPI_BF16) {
        __nv_bfloat16* p = reinterpret_cast<__nv_bfloat16*>(base) + grow * a.ldo + col0 + c;
        store_bf16x32(p, v);
      } else {
        // router logits: the last column tile may extend past N
        float* p = reinterpret_cast<float*>(base) + grow * a.ldo;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int col = col0 + c + j;
          if (col < a.n_valid) p[col] = v[j];
        }
      }
    }
  } else if (EPI == EPI_SWIGLU_FWD && SPLIT == SPLIT_MX && BN == 128) {
    // BN = 128: accumulator columns [0,64) gate, [64,128) up, for FFN columns
    // n0 .. n0+63 (n0 = n_tile*64); this warp: 32 of them, one MX block of h
    const long long r = tl.row0 + row_in_tile;
    const int I = a.I;
    const int c0 = half * 32;
    const int n0 = tl.n_tile * 64 + c0;
    const int y = tl.row0 + q * 32;
    float g[32], u[32];
    tmem_ld32(taddr + c0, g);
    tmem_ld32(taddr + 64 + c0, u);
    if (a.h_codes) {
      float hv[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        float s;
        hv[j] = silu_f(g[j], &s) * u[j];
      }
      uint32_t w[8];
      const uint32_t sbyte = mx_encode32(hv, w);
      uint4* cp = reinterpret_cast<uint4*>(a.h_codes + r * I + n0);
      cp[0] = make_uint4(w[0], w[1], w[2], w[3]);
      cp[1] = make_uint4(w[4], w[5], w[6], w[7]);
      a.h_scales[mx_tiled_off(r, n0 / 32, I / 128)] = static_cast<uint8_t>(sbyte);
    }
    if (a.store_c) {
      stage_and_store_f32<DBUF>(stage_buf, nst, tmC, g, lane, n0, y, false, a.evict_first != 0);
      stage_and_store_f32<DBUF>(stage_buf, nst, tmC, u, lane, I + n0, y, false,
                                a.evict_first != 0);
    }
  } else if (EPI == EPI_SWIGLU_FWD) {
    // BN = 256: accumulator columns [0,128) gate, [128,256) up, for FFN
    // columns n0 .. n0+127 with n0 = n_tile*128.  This thread: 64 of them.
    // g and u are kept in fp32 (TMA stores into GU [rows, 2I]); h = silu(g) u
    // is rounded to bf16, the operand of the down projection.
    const long long r = tl.row0 + row_in_tile;
    const int I = a.I;
    const int n0 = tl.n_tile * 128 + half * 64;
    const int y = tl.row0 + q * 32;
#pragma unroll 1
    for (int c = 0; c < 64; c += 32) {
      if (n0 + c >= I) break;  // a ragged last tile (I a multiple of 32)
      float g[32], u[32];
      tmem_ld32(taddr + half * 64 + c, g);
      tmem_ld32(taddr + 128 + half * 64 + c, u);
      if (SPLIT == SPLIT_NV) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          g[j] *= alpha;
          u[j] *= alpha;
        }
      }
      if (SPLIT == SPLIT_MX ? a.h_codes != nullptr : a.out2 != nullptr) {
        float hv[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          float s;
          hv[j] = silu_f(g[j], &s) * u[j];
        }
        if (SPLIT == SPLIT_MX) {
          // MXFP8 operand of the down projection: one block of 32 columns
          uint32_t w[8];
          const uint32_t sbyte = mx_encode32(hv, w);
          uint4* cp = reinterpret_cast<uint4*>(a.h_codes + r * I + n0 + c);
          cp[0] = make_uint4(w[0], w[1], w[2], w[3]);
          cp[1] = make_uint4(w[4], w[5], w[6], w[7]);
          a.h_scales[mx_tiled_off(r, (n0 + c) / 32, I / 128)] = static_cast<uint8_t>(sbyte);
        } else {
          if (a.mx) mx_fake32(hv);  // one MX block: 32 consecutive columns of a row
          stage_and_store_bf16_rows32(stage_buf, tmH, hv, lane, n0 + c, y);
        }
      }
      if (a.store_c) {
        stage_and_store_f32<DBUF>(stage_buf, nst, tmC, g, lane, n0 + c, y, false,
                                  a.evict_first != 0);
        stage_and_store_f32<DBUF>(stage_buf, nst, tmC, u, lane, I + n0 + c, y, false,
                                  a.evict_first != 0);
      }
    }
  }
}

// ------------------------------- block-scaled pairs: accumulator in registers --
// The block-scaled pair GEMMs keep one accumulator (their scale columns fill
// the rest of TMEM), so the MMAs of the next tile wait for this tile's
// epilogue.  These epilogues first copy the warp's 128 accumulator columns
// into registers; the caller then frees the accumulator, and the stores run
// while the next tile's MMAs do.

// The warp's 128 columns: EPI_F32, columns half*128 .. +127; SwiGLU forward,
// gate columns half*64 .. +63 then up columns 128 + half*64 .. +63.
template <int EPI>
__device__ __forceinline__ void acc_to_regs(uint32_t taddr, int half, float (&acc)[128]) {
  uint32_t r[8][16];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t col = EPI == EPI_SWIGLU_FWD
                             ? (j < 4 ? half * 64 + 16 * j : 128 + half * 64 + 16 * (j - 4))
                             : half * 128 + 16 * j;
    tmem_ld16(taddr + col, r[j]);
  }
  tmem_ld_wait();
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[16 * j + i] = __uint_as_float(r[j][i]);
}

template <int EPI, int SPLIT, bool DBUF>
__device__ __forceinline__ void epilogue_regs(const GemmArgs& a, const Tile& tl,
                                              float (&acc)[128], int q, int lane, int half,
                                              uint8_t* stage_buf, uint32_t& nst,
                                              const CUtensorMap* tmC, const CUtensorMap* tmH) {
  // NVFP4: the product of the operands' tensor scales (the block scales were
  // applied by the tensor cores)
  const float alpha = SPLIT == SPLIT_NV ? __ldg(a.ga) * __ldg(a.gb) : 1.0f;
  if (SPLIT == SPLIT_NV) {
#pragma unroll
    for (int j = 0; j < 128; ++j) acc[j] *= alpha;
  }
  const int y = tl.row0 + q * 32;
  if constexpr (EPI == EPI_F32) {
    const int col0 = tl.n_tile * 256 + half * 128;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float v[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = acc[32 * c + j];
      stage_and_store_f32<DBUF>(stage_buf, nst, tmC, v, lane, col0 + 32 * c, y,
                                a.accumulate != 0, a.evict_first != 0);
    }
  } else {
    // gate acc[0..63], up acc[64..127] for FFN columns n0 .. n0+63
    const long long r = tl.row0 + q * 32 + lane;
    const int I = a.I;
    const int n0 = tl.n_tile * 128 + half * 64;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float g[32], u[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        g[j] = acc[32 * c + j];
        u[j] = acc[64 + 32 * c + j];
      }
      // g and u leave first; h then takes g's registers
      if (a.store_c) {
        stage_and_store_f32<DBUF>(stage_buf, nst, tmC, g, lane, n0 + 32 * c, y, false,
                                  a.evict_first != 0);
        stage_and_store_f32<DBUF>(stage_buf, nst, tmC, u, lane, I + n0 + 32 * c, y, false,
                                  a.evict_first != 0);
      }
      if (SPLIT == SPLIT_MX ? a.h_codes != nullptr : a.out2 != nullptr) {
        float (&hv)[32] = g;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          float sg;
          hv[j] = silu_f(g[j], &sg) * u[j];
        }
        if (SPLIT == SPLIT_MX) {
          uint32_t w[8];
          const uint32_t sbyte = mx_encode32(hv, w);
          uint4* cp = reinterpret_cast<uint4*>(a.h_codes + r * I + n0 + 32 * c);
          cp[0] = make_uint4(w[0], w[1], w[2], w[3]);
          cp[1] = make_uint4(w[4], w[5], w[6], w[7]);
          a.h_scales[mx_tiled_off(r, (n0 + 32 * c) / 32, I / 128)] =
              static_cast<uint8_t>(sbyte);
        } else {
          stage_and_store_bf16_rows32(stage_buf, tmH, hv, lane, n0 + 32 * c, y);
        }
      }
    }
  }
}

// ------------------------------------------ SwiGLU backward, TMA operands --
// g, u of one chunk: 32 rows (this warp's lane quarter) x 16 fp32 columns of
// each, TMA-loaded into one of the warp's NBUF 4 KB staging buffers (g at +0,
// u at +2048, 64-byte swizzle: 16-byte chunk j of row r at chunk
// j ^ ((r >> 1) & 3)).  The warp's chunks are numbered from the kernel
// start; chunk n uses buffer n % NBUF and completes phase n / NBUF of that
// buffer's barrier.
template <int BN, int NBUF>
__device__ __forceinline__ void gu_issue(const GemmArgs& a, const Tile& tl, int q, int lane,
                                         int half, int c, uint8_t* stage_buf, uint64_t* wbar,
                                         uint32_t count, const CUtensorMap* tmG) {
  // every lane's earlier reads of the buffer come before the copy rewrites it
  fence_proxy_async_smem();
  __syncwarp();
  if (lane != 0) return;
  const int b = NBUF == 2 ? static_cast<int>(count & 1u) : 0;
  uint8_t* buf = stage_buf + b * kGuBufBytes;
  const int x = tl.n_tile * BN + half * (BN / 2) + c;
  const int y = tl.row0 + q * 32;
  mbar_arrive_expect_tx(&wbar[b], kGuBufBytes);
  tma_load_2d(buf, tmG, &wbar[b], x, y);
  tma_load_2d(buf + 2048, tmG, &wbar[b], a.I + x, y);
}

// The SwiGLU backward epilogue of one tile with g, u staged by TMA, chunk 0
// already requested; the next chunk's copies are in flight while this one is
// computed (with one buffer they are issued once every lane holds the current
// chunk's g, u in registers; with two, before waiting for it).  DIRECT stores
// the outputs from registers and keeps two buffers.  Returns the updated
// chunk count.  With a.mx, dG and dU are also
// quantised to MXFP8 (the gate/up dgrad's A operand): a block is 32
// consecutive columns of a row, so each odd chunk encodes itself together
// with the even chunk before it (n0 is a multiple of 32).
template <int BN, bool DIRECT>
__device__ __forceinline__ uint32_t swiglu_bwd_tma(const GemmArgs& a, const Tile& tl,
                                                   uint32_t taddr, int q, int lane, int half,
                                                   uint8_t* stage_buf, uint64_t* wbar,
                                                   uint32_t count, const CUtensorMap* tmG,
                                                   const OutMaps* om, volatile int* vabort) {
  constexpr int HALF_COLS = BN / 2;
  const long long r = tl.row0 + q * 32 + lane;
  const int I = a.I;
  const int n0 = tl.n_tile * BN + half * HALF_COLS;
  const int y = tl.row0 + q * 32;
  constexpr int NBUF = DIRECT ? 2 : 1;
  // output blocks of a chunk, 32 rows x 32 bytes each: dG hi, dG lo, dU hi,
  // dU lo, P hi, P lo
  uint8_t* ostage = stage_buf + NBUF * kGuBufBytes;
  const float p = a.row_w[r];
  float dp = 0.f;
  const int sw = (lane >> 1) & 3;
  float t_prev[16], dA_prev[16];  // mx: the even chunk's dG, dU
#pragma unroll 1
  for (int c = 0; c < HALF_COLS; c += 16, ++count) {
    if (NBUF == 2 && c + 16 < HALF_COLS)
      gu_issue<BN, NBUF>(a, tl, q, lane, half, c + 16, stage_buf, wbar, count + 1, tmG);
    const int b = NBUF == 2 ? static_cast<int>(count & 1u) : 0;
    const uint32_t par = NBUF == 2 ? ((count >> 1) & 1u) : (count & 1u);
    if (!mbar_wait(&wbar[b], par, vabort)) {
      *vabort = 1;
      set_status(a.status, MOK_ERR_DEVICE_TIMEOUT);
    }
    const uint8_t* buf = stage_buf + b * kGuBufBytes + lane * 64;
    float g[16], u[16], dA[16], t[16];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 a4 = *reinterpret_cast<const float4*>(buf + ((j ^ sw) << 4));
      const float4 b4 = *reinterpret_cast<const float4*>(buf + 2048 + ((j ^ sw) << 4));
      g[4 * j] = a4.x; g[4 * j + 1] = a4.y; g[4 * j + 2] = a4.z; g[4 * j + 3] = a4.w;
      u[4 * j] = b4.x; u[4 * j + 1] = b4.y; u[4 * j + 2] = b4.z; u[4 * j + 3] = b4.w;
    }
    // one buffer: it is free again, so the next chunk's copies go out
    // (gu_issue orders every lane's reads above before them)
    if (NBUF == 1 && c + 16 < HALF_COLS)
      gu_issue<BN, NBUF>(a, tl, q, lane, half, c + 16, stage_buf, wbar, count + 1, tmG);
    // a ragged last tile (I a multiple of 32): columns past I have no outputs
    // and add nothing to dp (their g, u were still staged, and are dropped)
    if (n0 + c >= I) continue;
    {
      uint32_t r0[16];
      tmem_ld16(taddr + half * HALF_COLS + c, r0);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) dA[j] = __uint_as_float(r0[j]);
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float sg;
      const float sl = silu_f(g[j], &sg);
      const float uu = u[j];
      const float dh = p * dA[j];
      dp = fmaf(dA[j], sl * uu, dp);
      t[j] = dh * uu * (sg * (1.0f + g[j] * (1.0f - sg)));
      dA[j] = dh * sl;
      u[j] = p * sl * uu;
    }
    if (a.mx) {
      if ((c & 16) == 0) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          t_prev[j] = t[j];
          dA_prev[j] = dA[j];
        }
      } else {
        const int col = n0 + c - 16;  // first column of the block
        const long long base = r * (2LL * I);
        float blk[32];
        uint32_t w[8];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          blk[j] = t_prev[j];
          blk[16 + j] = t[j];
        }
        uint32_t sbyte = mx_encode32(blk, w);
        uint4* cp = reinterpret_cast<uint4*>(a.dgu_codes + base + col);
        cp[0] = make_uint4(w[0], w[1], w[2], w[3]);
        cp[1] = make_uint4(w[4], w[5], w[6], w[7]);
        a.dgu_scales[mx_tiled_off(r, col / 32, 2 * I / 128)] = static_cast<uint8_t>(sbyte);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          blk[j] = dA_prev[j];
          blk[16 + j] = dA[j];
        }
        sbyte = mx_encode32(blk, w);
        cp = reinterpret_cast<uint4*>(a.dgu_codes + base + I + col);
        cp[0] = make_uint4(w[0], w[1], w[2], w[3]);
        cp[1] = make_uint4(w[4], w[5], w[6], w[7]);
        a.dgu_scales[mx_tiled_off(r, (I + col) / 32, 2 * I / 128)] = static_cast<uint8_t>(sbyte);
      }
    }
    if constexpr (DIRECT) {
      // the row's 16 columns of the six outputs from registers: 32
      // contiguous bytes per output and lane
      const long long o2 = r * (2LL * I) + n0 + c, o1 = r * static_cast<long long>(I) + n0 + c;
      __nv_bfloat16* gh = static_cast<__nv_bfloat16*>(a.out);
      __nv_bfloat16* gl = static_cast<__nv_bfloat16*>(a.out3);
      store_hi_lo16(gh + o2, gl + o2, t);
      store_hi_lo16(gh + o2 + I, gl + o2 + I, dA);
      store_hi_lo16(static_cast<__nv_bfloat16*>(a.out2) + o1,
                    static_cast<__nv_bfloat16*>(a.out4) + o1, u);
      continue;
    }
    if (lane == 0) bulk_wait_read<0>();  // the previous chunk's stores have read staging
    __syncwarp();
    uint8_t* row = ostage + lane * 32;
    store_hi_lo16(reinterpret_cast<__nv_bfloat16*>(row), reinterpret_cast<__nv_bfloat16*>(row + 1024),
                  t);
    store_hi_lo16(reinterpret_cast<__nv_bfloat16*>(row + 2048),
                  reinterpret_cast<__nv_bfloat16*>(row + 3072), dA);
    store_hi_lo16(reinterpret_cast<__nv_bfloat16*>(row + 4096),
                  reinterpret_cast<__nv_bfloat16*>(row + 5120), u);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(&om->dgu_hi, ostage, n0 + c, y);
      tma_store_2d(&om->dgu_lo, ostage + 1024, n0 + c, y);
      tma_store_2d(&om->dgu_hi, ostage + 2048, I + n0 + c, y);
      tma_store_2d(&om->dgu_lo, ostage + 3072, I + n0 + c, y);
      tma_store_2d(&om->p_hi, ostage + 4096, n0 + c, y);
      tma_store_2d(&om->p_lo, ostage + 5120, n0 + c, y);
      bulk_commit();
    }
  }
  __syncwarp();
  a.dp_part[r * a.np + tl.n_tile * 2 + half] = dp;
  return count;
}

// ------------------------------------------------------------------- kernel --

template <int BN, bool A_MN, bool B_MN, int SCHED, int EPI, int SPLIT, bool PAIR, bool DB>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmL,
                const __grid_constant__ GemmArgs args, const __grid_constant__ OutMaps om) {
  using C = Cfg<BN, SPLIT, PAIR, staging_bytes<EPI, SPLIT, SCHED, DB>()>;
  constexpr bool kDbuf = DB;
  static_assert(!DB || ((EPI == EPI_F32 || EPI == EPI_F32_T) && SCHED == SCHED_KGROUP) ||
                    (EPI == EPI_SWIGLU_BWD && PAIR),
                "DB: double-buffered staging of the fp32 weight gradients, or the SwiGLU "
                "backward's stores from registers");
  static_assert(!PAIR || (SCHED != SCHED_DENSE && SPLIT != SPLIT_B && BN == 256), "pair");
  static_assert(SPLIT != SPLIT_MX ||
                    (!A_MN && !B_MN && BN == (PAIR ? 256 : 128) && SCHED == SCHED_MGROUP),
                "MXFP8 operands: K-major, 128-wide tiles (256 on CTA pairs)");
  static_assert(SPLIT != SPLIT_NV || (PAIR && BN == 256 && !A_MN && !B_MN &&
                                      SCHED == SCHED_MGROUP &&
                                      (EPI == EPI_SWIGLU_FWD || EPI == EPI_F32)),
                "NVFP4 operands: K-major, M-grouped, CTA pairs");
  // TMA x coordinate per stage: K values (bf16), code bytes (MXFP8, NVFP4)
  constexpr int KX = block_scaled(SPLIT) ? 128 : 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* tiles = smem;
  uint8_t* staging = smem + C::STAGING_OFF;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  // SwiGLU backward: two g/u staging buffers per epilogue warp, one barrier each
  uint64_t* gu_bar = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF + 256);
  constexpr bool kTmaStore = (EPI == EPI_F32 && SCHED != SCHED_DENSE) || EPI == EPI_SWIGLU_FWD ||
                             EPI == EPI_F32_T || EPI == EPI_SWIGLU_BWD || EPI == EPI_BF16_TMA ||
                             EPI == EPI_BF16_T;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // work units: tiles (one CTA) or tile pairs (one cluster of two CTAs)
  const int rank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;
  const bool leader = rank == 0;
  const int first = PAIR ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
  const int step = PAIR ? static_cast<int>(cluster_count_x()) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      // PAIR: the leader's MMA waits for the epilogues of both CTAs
      mbar_init(&tempty[i], PAIR ? 2 * kEpiWarps : kEpiWarps);
    }
    mbar_init(drain, 1);
    if (EPI == EPI_SWIGLU_BWD)
      for (int i = 0; i < 2 * kEpiWarps; ++i) mbar_init(&gu_bar[i], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (threadIdx.x == 32) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (kTmaStore) tma_prefetch_desc(&tmC);
    if (block_scaled(SPLIT) && PAIR) {
      tma_prefetch_desc(&om.sfa);
      tma_prefetch_desc(&om.sfb);
    }
    if (EPI == EPI_SWIGLU_FWD && SPLIT != SPLIT_MX) tma_prefetch_desc(&om.h);
    if (EPI == EPI_SWIGLU_BWD) {
      tma_prefetch_desc(&om.dgu_hi);
      tma_prefetch_desc(&om.dgu_lo);
      tma_prefetch_desc(&om.p_hi);
      tma_prefetch_desc(&om.p_lo);
    }
    if (SPLIT != SPLIT_NONE) tma_prefetch_desc(&tmL);
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, C::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before_sync();
  if (PAIR) cluster_sync(); else __syncthreads();
  tc_fence_after_sync();
  // Everything above touches only shared memory, TMEM and the kernel's
  // parameters, so as a programmatic dependent it overlaps the previous
  // kernel's tail; from here on that kernel's results are visible.
  grid_dep_wait();
  grid_dep_launch();
  const uint32_t tmem_base = *tmem_slot;
  volatile int* vabort = abort_flag;
  const int total = PAIR ? total_pairs<SCHED>(args) : total_tiles<SCHED>(args);
  auto tile_at = [&](int t, bool* valid) -> Tile {
    if (PAIR) return decode_pair<SCHED>(args, t, rank, valid);
    *valid = true;
    return decode_tile<SCHED>(args, t);
  };
  // bounded waits; barriers that the other CTA of a pair completes are
  // acquired at cluster scope
  auto wait = [&](uint64_t* bar, uint32_t par) -> bool {
    return PAIR ? mbar_wait_cluster(bar, par, vabort) : mbar_wait(bar, par, vabort);
  };

  if (warp == 0) {
    // single-CTA SPLIT_MX: every lane gathers scale bytes; lane 0 alone
    // issues the TMA (CTA pairs load the scale blocks by TMA as well)
    if (lane == 0 || (SPLIT == SPLIT_MX && !PAIR)) {
      // ------------------------------------------------------- producer --
      // PAIR: both CTAs load their halves; the copies complete on the
      // leader's `full` barrier, which the leader arms for both
      const uint32_t full_leader = PAIR ? mapa_shared(smem_addr(full), 0) : 0u;
      int stage = 0;
      uint32_t phase = 0;
      int issued_par[C::STAGES];
#pragma unroll
      for (int s = 0; s < C::STAGES; ++s) issued_par[s] = -1;
      bool ok = true;
      for (int t = first; t < total && ok; t += step) {
        bool valid;
        const Tile tl = tile_at(t, &valid);
        SegWalk walk;
        if (SCHED == SCHED_KGROUP) walk.init(args, tl.e);
        for (int kb = 0; kb < tl.num_kb; ++kb) {
          // K-grouped: this K block's operand row, through the row spaces
          const int kgy = SCHED == SCHED_KGROUP ? walk.row_of(args, tl.e, kb) : 0;
          if (!wait(&empty[stage], phase ^ 1u)) {
            ok = false;
            break;
          }
          uint8_t* sA = tiles + stage * C::STAGE_BYTES;
          uint8_t* sB = sA + C::B_OFF;
          const uint32_t bar_c = full_leader + 8u * stage;
          if (SPLIT == SPLIT_MX && !PAIR) {
            // the stage's scale blocks from the tiled layout (each row's four
            // K-block bytes are one word there): A rows row0.., then the B
            // tile's rows (SWIGLU_FWD: 64 gate rows, then the 64 up rows)
            const long long nkg = args.ks / 4, j0 = (long long)(tl.kb0 + kb) * 4;
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
              w[j] = *reinterpret_cast<const uint32_t*>(
                  args.sa + mx_tiled_off(tl.row0 + lane + 32 * j, j0, nkg));
            *reinterpret_cast<uint4*>(sA + C::SF_OFF + lane * 16) = make_uint4(w[0], w[1], w[2], w[3]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int t = lane + 32 * j;  // row of the B tile
              long long grow;
              if (EPI == EPI_SWIGLU_FWD)
                grow = (long long)tl.e * args.b_group_rows + tl.n_tile * (BN / 2) +
                       (t < BN / 2 ? t : args.I + t - BN / 2);
              else
                grow = (long long)tl.e * args.b_group_rows + tl.n_tile * BN + t;
              w[j] = *reinterpret_cast<const uint32_t*>(args.sb + mx_tiled_off(grow, j0, nkg));
            }
            *reinterpret_cast<uint4*>(sA + C::SF_OFF + 512 + lane * 16) =
                make_uint4(w[0], w[1], w[2], w[3]);
            fence_proxy_async_smem();  // read by tcgen05.cp through the async proxy
            __syncwarp();
          }
          auto load = [&](void* dst, const CUtensorMap* tm, int x, int y) {
            if (SPLIT == SPLIT_MX && lane != 0) return;
            if (PAIR) tma_load_2d_pair(dst, tm, bar_c, x, y);
            else tma_load_2d(dst, tm, &full[stage], x, y);
          };
          // the stage's TMA bytes: the code or bf16 tiles (SF_OFF), and on
          // MXFP8 pairs the scale blocks as well
          if (!PAIR) {
            if (lane == 0) mbar_arrive_expect_tx(&full[stage], C::SF_OFF);
          } else if (leader) {
            if (lane == 0)
              mbar_arrive_expect_tx(&full[stage],
                                    2 * (C::SF_OFF + (block_scaled(SPLIT) ? C::SF_BYTES : 0)));
          }
          if (PAIR && SPLIT == SPLIT_MX) {
            // scale blocks by TMA: this CTA's A rows, and all BN rows of B
            const int nkg = args.ks / 4, kg = tl.kb0 + kb;
            load(sA + C::SF_OFF, &om.sfa, 0, 2 * ((tl.row0 >> 7) * nkg + kg));
#pragma unroll
            for (int blk = 0; blk < BN / 128; ++blk) {
              const int g0 = EPI == EPI_SWIGLU_FWD
                                 ? tl.e * args.b_group_rows + tl.n_tile * 128 + (blk ? args.I : 0)
                                 : tl.e * args.b_group_rows + tl.n_tile * BN + blk * 128;
              load(sA + C::SF_OFF + 512 + blk * 512, &om.sfb, 0, 2 * ((g0 >> 7) * nkg + kg));
            }
          }
          if (PAIR && SPLIT == SPLIT_NV) {
            // the stage's four scale blocks per 128 rows (2 KB, one TMA copy
            // each): this CTA's A rows, and both 128-row halves of B
            const int nkb = args.ks, k4 = 4 * (tl.kb0 + kb);
            load(sA + C::SF_OFF, &om.sfa, 0, 2 * ((tl.row0 >> 7) * nkb + k4));
#pragma unroll
            for (int blk = 0; blk < 2; ++blk) {
              const int g0 = EPI == EPI_SWIGLU_FWD
                                 ? tl.e * args.b_group_rows + tl.n_tile * 128 + (blk ? args.I : 0)
                                 : tl.e * args.b_group_rows + tl.n_tile * BN + blk * 128;
              load(sA + C::SF_OFF + 2048 + blk * 2048, &om.sfb, 0, 2 * ((g0 >> 7) * nkb + k4));
            }
          }
          // A tile: 128 rows (M) x 64 (K)  (+ its lo tile with SPLIT_A)
          if (!A_MN) {
            load(sA, &tmA, (tl.kb0 + kb) * KX, tl.row0);
          } else {
            const int ky = SCHED == SCHED_KGROUP ? kgy : tl.k_row0 + (tl.kb0 + kb) * 64;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              load(sA + j * 8192, &tmA, tl.row0 + 64 * j, ky);
              if (SPLIT == SPLIT_A) load(sA + C::A_BYTES + j * 8192, &tmL, tl.row0 + 64 * j, ky);
            }
          }
          // B tile: B_ROWS rows (N) x 64 (K); PAIR: this CTA's half of N
          if (!B_MN) {
            if (EPI == EPI_SWIGLU_FWD) {
              // gate rows n0..n0+BN/2-1, then the matching up rows (+I)
              const int r0 = tl.e * args.b_group_rows + tl.n_tile * (BN / 2);
              if (PAIR) {
                load(sB, &tmB, kb * KX, r0 + rank * args.I);
              } else {
                load(sB, &tmB, kb * KX, r0);
                load(sB + (BN / 2) * 128, &tmB, kb * KX, r0 + args.I);
              }
            } else {
              const int r0 = (SCHED == SCHED_DENSE ? 0 : tl.e * args.b_group_rows) +
                             tl.n_tile * BN + rank * C::B_ROWS;
              load(sB, &tmB, (tl.kb0 + kb) * KX, r0);
            }
          } else {
            int ky;
            if (SCHED == SCHED_KGROUP) ky = kgy;
            else if (SCHED == SCHED_DENSE) ky = (tl.kb0 + kb) * 64;
            else ky = tl.e * args.b_group_rows + kb * 64;
            const int x0 = tl.n_tile * BN + rank * C::B_ROWS;
#pragma unroll
            for (int j = 0; j < C::B_ROWS / 64; ++j) {
              load(sB + j * 8192, &tmB, x0 + 64 * j, ky);
              if (SPLIT == SPLIT_B) load(sB + C::B_BYTES + j * 8192, &tmL, x0 + 64 * j, ky);
            }
          }
          issued_par[stage] = static_cast<int>(phase);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        *vabort = 1;
        set_status(args.status, MOK_ERR_DEVICE_TIMEOUT);
        // let the copies already issued land before the CTA can exit: their
        // barriers where this CTA holds them, else a fixed millisecond
        const int zero = 0;
        if (!PAIR || leader) {
          for (int s = 0; s < C::STAGES; ++s)
            if (issued_par[s] >= 0)
              mbar_wait(&full[s], static_cast<uint32_t>(issued_par[s]), &zero);
        } else {
          spin_ns(1000000ull);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------------------ MMA --
      constexpr uint32_t idesc = idesc_bf16_f32(PAIR ? 256 : 128, BN, A_MN, B_MN);
      constexpr uint32_t lbo_a = A_MN ? 8192u : 16u;
      constexpr uint32_t lbo_b = B_MN ? 8192u : 16u;
      constexpr uint32_t kstep_a = A_MN ? 2048u : 32u;
      constexpr uint32_t kstep_b = B_MN ? 2048u : 32u;
      auto mma = [&](uint32_t d, uint64_t ad, uint64_t bd, uint32_t acc_in) {
        if (PAIR) mma_bf16_pair(d, ad, bd, idesc, acc_in);
        else mma_bf16(d, ad, bd, idesc, acc_in);
      };
      auto commit = [&](uint64_t* bar) {
        if (PAIR) mma_commit_pair(bar);
        else mma_commit(bar);
      };
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int t = first; t < total && ok; t += step, ++it) {
        bool valid;
        const Tile tl = tile_at(t, &valid);
        const int acc = C::NACC == 2 ? (it & 1) : 0;
        const uint32_t acc_par = static_cast<uint32_t>(C::NACC == 2 ? ((it >> 1) & 1) : (it & 1));
        if (!wait(&tempty[acc], acc_par ^ 1u)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < tl.num_kb; ++kb) {
          if (!wait(&full[stage], phase)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a_base = smem_addr(tiles + stage * C::STAGE_BYTES);
          const uint32_t b_base = a_base + C::B_OFF;
          if constexpr (SPLIT == SPLIT_NV) {
            // per K = 64 MMA j: the A scale block to 4 columns, the two B
            // half blocks to 8 (rows 0..127, then 128..255), each CTA's
            // blocks to its own TMEM; then the block-scaled FP4 MMA
            const uint32_t sfa = tmem_base + C::NACC * BN + C::SF_COLS * stage;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              tmem_cp_sf_pair(sfa + 4u * j, smem_desc_sf(a_base + C::SF_OFF + 512 * j));
              tmem_cp_sf_pair(sfa + 16u + 8u * j,
                              smem_desc_sf(a_base + C::SF_OFF + 2048 + 512 * j));
              tmem_cp_sf_pair(sfa + 20u + 8u * j,
                              smem_desc_sf(a_base + C::SF_OFF + 4096 + 512 * j));
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint64_t ad = smem_desc_sw128(a_base + j * 32, 16, 1024);
              const uint64_t bd = smem_desc_sw128(b_base + j * 32, 16, 1024);
              mma_nvf4_pair(d_tmem, ad, bd, idesc_nvf4(256, BN), sfa + 4u * j,
                            sfa + 16u + 8u * j, (kb | j) != 0 ? 1u : 0u);
            }
          } else if constexpr (SPLIT == SPLIT_MX) {
            // scales to TMEM (SF_COLS columns per stage after the
            // accumulators), then four K=32 block-scaled MMAs, scale byte j
            // each; CTA pairs copy each CTA's blocks to its own TMEM
            const uint32_t sfa = tmem_base + C::NACC * BN + C::SF_COLS * stage;
            if (PAIR) {
              tmem_cp_sf_pair(sfa, smem_desc_sf(a_base + C::SF_OFF));
              tmem_cp_sf_pair(sfa + 4u, smem_desc_sf(a_base + C::SF_OFF + 512));
              tmem_cp_sf_pair(sfa + 8u, smem_desc_sf(a_base + C::SF_OFF + 1024));
            } else {
              tmem_cp_sf(sfa, smem_desc_sf(a_base + C::SF_OFF));
              tmem_cp_sf(sfa + 4u, smem_desc_sf(a_base + C::SF_OFF + 512));
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint64_t ad = smem_desc_sw128(a_base + j * 32, 16, 1024);
              const uint64_t bd = smem_desc_sw128(b_base + j * 32, 16, 1024);
              const uint32_t id = idesc_mxf8(PAIR ? 256 : 128, BN, static_cast<uint32_t>(j));
              if (PAIR)
                mma_mxf8_pair(d_tmem, ad, bd, id, sfa, sfa + 4u, (kb | j) != 0 ? 1u : 0u);
              else
                mma_mxf8(d_tmem, ad, bd, id, sfa, sfa + 4u, (kb | j) != 0 ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint64_t ad = smem_desc_sw128(a_base + j * kstep_a, lbo_a, 1024);
              const uint64_t bd = smem_desc_sw128(b_base + j * kstep_b, lbo_b, 1024);
              mma(d_tmem, ad, bd, (kb | j) != 0 ? 1u : 0u);
              if (SPLIT == SPLIT_A) {
                const uint64_t ad2 =
                    smem_desc_sw128(a_base + C::A_BYTES + j * kstep_a, lbo_a, 1024);
                mma(d_tmem, ad2, bd, 1u);
              } else if (SPLIT == SPLIT_B) {
                const uint64_t bd2 =
                    smem_desc_sw128(b_base + C::B_BYTES + j * kstep_b, lbo_b, 1024);
                mma(d_tmem, ad, bd2, 1u);
              }
            }
          }
          commit(&empty[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        commit(&tfull[acc]);
      }
      if (!ok) {
        *vabort = 1;
        set_status(args.status, MOK_ERR_DEVICE_TIMEOUT);
        const int zero = 0;
        commit(drain);
        mbar_wait(drain, 0, &zero);
      }
    }
  } else {
    // ----------------------------------------------------------- epilogue --
    const int q = warp & 3;                // TMEM lane quarter this warp may read
    const int half = (warp - 2) >> 2;      // column half of the tile
    uint8_t* stage_buf = staging + (warp - 2) * C::STAGING_PER_WARP;
    const uint32_t tempty_leader = PAIR ? mapa_shared(smem_addr(tempty), 0) : 0u;
    // SwiGLU backward: g, u come by TMA (tmC maps them); `gu_chunks` counts
    // the chunks this warp has requested
    constexpr bool kGuTma = EPI == EPI_SWIGLU_BWD;
    // block-scaled pairs (one accumulator): free it before the stores
    constexpr bool kEarlyRelease = PAIR && block_scaled(SPLIT) && C::NACC == 1 &&
                                   SCHED == SCHED_MGROUP && BN == 256 &&
                                   (EPI == EPI_F32 || EPI == EPI_SWIGLU_FWD);
    uint64_t* wbar = gu_bar + 2 * (warp - 2);
    uint32_t gu_chunks = 0;
    uint32_t nst = 0;  // TMA-store blocks issued by this warp
    int it = 0;
    for (int t = first; t < total; t += step, ++it) {
      bool valid;
      const Tile tl = tile_at(t, &valid);
      const int acc = C::NACC == 2 ? (it & 1) : 0;
      const uint32_t acc_par = static_cast<uint32_t>(C::NACC == 2 ? ((it >> 1) & 1) : (it & 1));
      // this warp's 32 rows: none of them read by anything (args.coff)
      bool unread = false;
      if (SCHED == SCHED_MGROUP && args.coff != nullptr && valid) {
        const int used = (__ldg(args.coff + tl.e + 1) - __ldg(args.coff + tl.e) + 63) / 64 * 64;
        unread = tl.row0 + q * 32 - __ldg(args.poff + tl.e) >= used;
      }
      const bool work = valid && !unread;
      // the tile's first g, u chunk does not depend on the accumulator
      if (kGuTma && work)
        gu_issue<BN, kDbuf ? 2 : 1>(args, tl, q, lane, half, 0, stage_buf, wbar, gu_chunks,
                                    &tmC);
      if (!wait(&tfull[acc], acc_par)) {
        *vabort = 1;
        set_status(args.status, MOK_ERR_DEVICE_TIMEOUT);
        break;
      }
      tc_fence_after_sync();
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
      if constexpr (kEarlyRelease) {
        // the accumulator to registers, freed at once; the stores follow
        float accr[128];
        if (work) acc_to_regs<EPI>(taddr, half, accr);
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(tempty_leader + 8u * acc);
        if (work)
          epilogue_regs<EPI, SPLIT, kDbuf>(args, tl, accr, q, lane, half, stage_buf, nst, &tmC,
                                           &om.h);
        continue;
      }
      if constexpr (kGuTma) {
        if (work)
          gu_chunks = swiglu_bwd_tma<BN, kDbuf>(args, tl, taddr, q, lane, half, stage_buf, wbar,
                                         gu_chunks, &tmC, &om, vabort);
      } else if (work) {
        epilogue_tile<BN, SCHED, EPI, kDbuf, SPLIT>(args, tl, taddr, q, lane, half, stage_buf,
                                                    nst, &tmC, &om.h);
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if (PAIR) mbar_arrive_cluster(tempty_leader + 8u * acc);
        else mbar_arrive(&tempty[acc]);
      }
    }
    if (kTmaStore && lane == 0) bulk_wait_all<0>();  // stores complete before exit
    // after a failed wait, g/u copies may still be landing in staging
    if (kGuTma && *vabort) spin_ns(1000000ull);
  }

  // the leader's MMAs read the other CTA's shared memory: neither CTA of a
  // pair leaves (or frees TMEM) before both are done
  tc_fence_before_sync();
  if (PAIR) cluster_sync(); else __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    if (PAIR) tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    else tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// --------------------------------------------------------------------- host --

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D map over a row-major [outer, inner] array with row stride `row_elems`,
// box {box_inner, box_rows}, 128-byte swizzle, zero fill out of bounds.
static bool make_map_t(CUtensorMap* m, CUtensorMapDataType dt, int esz, const void* base,
                       uint64_t inner, uint64_t outer, uint64_t row_elems, uint32_t box_inner,
                       uint32_t box_rows,
                       CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  if (outer == 0) outer = 1;  // empty operand: the map exists but is never read
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_elems * esz};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tensor_map_2d(CUtensorMap* m, CUtensorMapDataType dt, int esz, const void* base,
                        uint64_t inner, uint64_t outer, uint64_t row_elems, uint32_t box_inner,
                        uint32_t box_rows, CUtensorMapSwizzle swz) {
  return make_map_t(m, dt, esz, base, inner, outer, row_elems, box_inner, box_rows, swz);
}

// bf16 operand map, box {64, box_rows}
static bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                     uint64_t row_elems, uint32_t box_rows) {
  return make_map_t(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, inner, outer, row_elems, 64,
                    box_rows);
}

// fp32 output map for the TMA-store epilogue, box {32, 32}
static bool make_out_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows) {
  return make_map_t(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, cols, rows, cols, 32, 32);
}
// bf16 C: 32-row x 64-column blocks (128-byte rows, 128-byte swizzle)
static bool make_out_map_bf16(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows) {
  return make_map_t(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, cols, rows, cols, 64, 32);
}
// bf16 [rows, cols] stored in 32 x 32 blocks (64-byte rows, 64-byte swizzle):
// C^T blocks of the transposed weight gradients, and h
static bool make_out_map_bf16_t(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows) {
  return make_map_t(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, cols, rows, cols, 32, 32,
                    CU_TENSOR_MAP_SWIZZLE_64B);
}

// max_units: an upper bound on the tiles (PAIR: tile pairs) of the launch;
// the kernel reads the exact count on the device.
template <int BN, bool A_MN, bool B_MN, int SCHED, int EPI, int SPLIT = SPLIT_NONE,
          bool PAIR = false, bool DB = false>
static cudaError_t launch(const char* name, const CUtensorMap& ta, const CUtensorMap& tb,
                          const CUtensorMap& tc, const GemmArgs& args, int max_units,
                          cudaStream_t st, const CUtensorMap* tl = nullptr,
                          const OutMaps* om = nullptr) {
  OutMaps om_v;
  if (om) om_v = *om;
  else memset(&om_v, 0, sizeof(om_v));
  auto kern = gemm_kernel<BN, A_MN, B_MN, SCHED, EPI, SPLIT, PAIR, DB>;
  constexpr int smem = Cfg<BN, SPLIT, PAIR, staging_bytes<EPI, SPLIT, SCHED, DB>()>::SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if (max_units <= 0) return cudaSuccess;
  // every GEMM launches as a programmatic dependent of the kernel before it:
  // its prologue (barriers, TMEM, descriptors) runs in that kernel's tail and
  // it waits for that kernel's results before its first global access
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (!PAIR) {
    int grid = num_sms_current_device();
    if (max_units < grid) grid = max_units;
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    ProfScope prof(name, st);
    e = cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, tl ? *tl : ta, args, om_v);
    count_launch();
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  // clusters of two CTAs, as many as can be resident at once (one per SM pair)
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.numAttrs = 2;
  cfg.gridDim = dim3(static_cast<unsigned>(num_sms_current_device() / 2 * 2), 1, 1);
  // per kernel instantiation and process (one device type); racing first
  // launches compute the same value
  static std::atomic<int> max_clusters_cache{-1};
  int max_clusters = max_clusters_cache.load(std::memory_order_relaxed);
  if (max_clusters < 0) {
    cudaLaunchConfig_t q = cfg;  // the cluster shape alone
    q.attrs = &attr[1];
    q.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &q);
    if (e != cudaSuccess) return e;
    max_clusters = n;
    max_clusters_cache.store(n, std::memory_order_relaxed);
  }
  if (max_clusters < 1) return cudaErrorInvalidConfiguration;
  int clusters = max_clusters < max_units ? max_clusters : max_units;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters), 1, 1);
  ProfScope prof(name, st);
  e = cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, tl ? *tl : ta, args, om_v);
  count_launch();
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

static GemmArgs blank_args(int* status) {
  GemmArgs a;
  memset(&a, 0, sizeof(a));
  a.status = status;
  return a;
}

static inline int max_mtiles(const Dims& D) { return static_cast<int>(D.rows_max / 128); }
// bound on the tile pairs: sum over experts of ceil(tiles_e / 2)
static inline int max_mpairs(const Dims& D) {
  const int64_t segs = D.R < D.E ? D.R : D.E;
  return static_cast<int>((D.rows_max / 128 + segs + 1) / 2);
}

cudaError_t gemm_fwd_gate_up(const Dims& D, const void* X_perm, const void* w_gate_up,
                             const int32_t* mtile_prefix, const int32_t* poff, void* GU, void* H,
                             int* status, cudaStream_t st) {
  CUtensorMap ta, tb, tc;
  if (!make_map(&ta, X_perm, D.d, D.rows_max, D.d, 128)) return cudaErrorInvalidValue;
  if (!make_map(&tb, w_gate_up, D.d, D.E * 2 * D.I, D.d, 128)) return cudaErrorInvalidValue;
  // without GU the C map is never used; it then describes the A operand so
  // that the kernel's descriptor prefetch still sees a valid map
  if (GU ? !make_out_map(&tc, GU, 2 * D.I, D.rows_max) : !make_map(&tc, X_perm, D.d, D.rows_max, D.d, 128))
    return cudaErrorInvalidValue;
  if (!GU && !H) return cudaErrorInvalidValue;
  GemmArgs a = blank_args(status);
  a.store_c = GU ? 1 : 0;
  a.evict_first = 1;  // g, u are read again only by the backward
  a.E = (int)D.E;
  a.n_tiles = (int)((D.I + 127) / 128);  // a ragged last tile: FFN columns past I unstored
  a.num_kb = (int)((D.d + 63) / 64);  // a ragged last K block reads zeros
  a.b_group_rows = (int)(2 * D.I);
  a.I = (int)D.I;
  a.mtile_prefix = mtile_prefix;
  a.poff = poff;
  a.coff = D.coff;  // unread padding rows: no epilogue
  a.out = GU;
  a.out2 = H;
  a.mx = D.mx ? 1 : 0;
  OutMaps om;  // h through TMA stores of 32 x 32 blocks
  memset(&om, 0, sizeof(om));
  if (H && !make_out_map_bf16_t(&om.h, H, D.I, D.rows_max)) return cudaErrorInvalidValue;
  if (D.pair)
    return launch<256, false, false, SCHED_MGROUP, EPI_SWIGLU_FWD, SPLIT_NONE, true>(
        "fwd_gate_up_swiglu", ta, tb, tc, a, max_mpairs(D) * a.n_tiles, st, nullptr, &om);
  return launch<256, false, false, SCHED_MGROUP, EPI_SWIGLU_FWD>(
      "fwd_gate_up_swiglu", ta, tb, tc, a, max_mtiles(D) * a.n_tiles, st, nullptr, &om);
}

// The tiled scales of a [rows, K] MXFP8 operand as a TMA map: 512-byte blocks
// viewed as pairs of 256-byte rows (box: one block).
static bool make_sf_map(CUtensorMap* m, const uint8_t* scales, int64_t rows, int64_t K) {
  const uint64_t blocks = static_cast<uint64_t>(rows / 128) * static_cast<uint64_t>(K / 128);
  return make_map_t(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, scales, 256, 2 * blocks, 256, 256, 2,
                    CU_TENSOR_MAP_SWIZZLE_NONE);
}

// MXFP8 operands (E4M3 codes, E8M0 scale bytes per 32 K values, K-major):
// the gate/up GEMM with g, u to GU (NULL: not stored) and h as MXFP8 codes
// and scales (NULL: not stored), single-CTA 128-wide tiles of 64 FFN columns.
cudaError_t gemm_fwd_gate_up_mx(const Dims& D, const uint8_t* x_codes, const uint8_t* x_scales,
                                const uint8_t* wgu_codes, const uint8_t* wgu_scales,
                                const int32_t* mtile_prefix, const int32_t* poff, void* GU,
                                uint8_t* h_codes, uint8_t* h_scales, int* status,
                                cudaStream_t st) {
  const auto u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  const bool pair = D.pair;  // 256-wide tiles (128 FFN columns) on CTA pairs
  CUtensorMap ta, tb, tc;
  if (!make_map_t(&ta, u8, 1, x_codes, D.d, D.rows_max, D.d, 128, 128, sw) ||
      !make_map_t(&tb, u8, 1, wgu_codes, D.d, D.E * 2 * D.I, D.d, 128, pair ? 128 : 64, sw))
    return cudaErrorInvalidValue;
  if (GU ? !make_out_map(&tc, GU, 2 * D.I, D.rows_max) : false) return cudaErrorInvalidValue;
  if (!GU) tc = ta;  // never used without GU; a valid map for the prefetch
  if (!GU && !h_codes) return cudaErrorInvalidValue;
  GemmArgs a = blank_args(status);
  a.store_c = GU ? 1 : 0;
  a.evict_first = 1;
  a.E = (int)D.E;
  a.n_tiles = (int)(D.I / 64);
  a.num_kb = (int)(D.d / 128);
  a.b_group_rows = (int)(2 * D.I);
  a.I = (int)D.I;
  a.mtile_prefix = mtile_prefix;
  a.poff = poff;
  a.coff = D.coff;  // unread padding rows: no epilogue
  a.out = GU;
  a.sa = x_scales;
  a.sb = wgu_scales;
  a.ks = (int)(D.d / 32);
  a.h_codes = h_codes;
  a.h_scales = h_scales;
  if (pair) {
    a.n_tiles = (int)(D.I / 128);
    OutMaps om;
    memset(&om, 0, sizeof(om));
    if (!make_sf_map(&om.sfa, x_scales, D.rows_max, D.d) ||
        !make_sf_map(&om.sfb, wgu_scales, D.E * 2 * D.I, D.d))
      return cudaErrorInvalidValue;
    return launch<256, false, false, SCHED_MGROUP, EPI_SWIGLU_FWD, SPLIT_MX, true>(
        "fwd_gate_up_swiglu", ta, tb, tc, a, max_mpairs(D) * a.n_tiles, st, nullptr, &om);
  }
  return launch<128, false, false, SCHED_MGROUP, EPI_SWIGLU_FWD, SPLIT_MX>(
      "fwd_gate_up_swiglu", ta, tb, tc, a, max_mtiles(D) * a.n_tiles, st);
}

// An M-grouped GEMM on MXFP8 operands with fp32 rows out: O[rows_max, d] =
// A[rows_max, K] B_e[d, K]^T per expert segment, A and B as E4M3 codes,
// K-major, with tiled scales.  The down projection (K = I) and the gate/up
// dgrad (K = 2I, B = W_gate_up transposed) are this GEMM.
static cudaError_t grouped_mx_f32(const char* name, const Dims& D, int64_t K,
                                  const uint8_t* a_codes, const uint8_t* a_scales,
                                  const uint8_t* b_codes, const uint8_t* b_scales,
                                  const int32_t* mtile_prefix, const int32_t* poff, void* O,
                                  int* status, cudaStream_t st) {
  const auto u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  CUtensorMap ta, tb, tc;
  if (!make_map_t(&ta, u8, 1, a_codes, K, D.rows_max, K, 128, 128, sw) ||
      !make_map_t(&tb, u8, 1, b_codes, K, D.E * D.d, K, 128, 128, sw) ||
      !make_out_map(&tc, O, D.d, D.rows_max))
    return cudaErrorInvalidValue;
  GemmArgs a = blank_args(status);
  a.E = (int)D.E;
  a.n_tiles = (int)(D.d / 128);
  a.num_kb = (int)(K / 128);
  a.b_group_rows = (int)D.d;
  a.mtile_prefix = mtile_prefix;
  a.poff = poff;
  a.coff = D.coff;  // unread padding rows: no epilogue
  a.out = O;  // fp32 [rows_max, d]
  a.ldo = D.d;
  a.sa = a_scales;
  a.sb = b_scales;
  a.ks = (int)(K / 32);
  if (D.pair && D.d % 256 == 0) {
    a.n_tiles = (int)(D.d / 256);
    OutMaps om;
    memset(&om, 0, sizeof(om));
    if (!make_sf_map(&om.sfa, a_scales, D.rows_max, K) ||
        !make_sf_map(&om.sfb, b_scales, D.E * D.d, K))
      return cudaErrorInvalidValue;
    return launch<256, false, false, SCHED_MGROUP, EPI_F32, SPLIT_MX, true>(
        name, ta, tb, tc, a, max_mpairs(D) * a.n_tiles, st, nullptr, &om);
  }
  return launch<128, false, false, SCHED_MGROUP, EPI_F32, SPLIT_MX>(
      name, ta, tb, tc, a, max_mtiles(D) * a.n_tiles, st);
}

cudaError_t gemm_fwd_down_mx(const Dims& D, const uint8_t* h_codes, const uint8_t* h_scales,
                             const uint8_t* wd_codes, const uint8_t* wd_scales,
                             const int32_t* mtile_prefix, const int32_t* poff, void* O,
                             int* status, cudaStream_t st) {
  return grouped_mx_f32("fwd_down", D, D.I, h_codes, h_scales, wd_codes, wd_scales, mtile_prefix,
                        poff, O, status, st);
}

// NVFP4 scales in the tiled layout (one 512-byte block per 128 rows x 64 K
// values, the four blocks of a 256-value stage consecutive) as a TMA map of
// 256-byte rows: one stage's blocks of a 128-row tile are a 2 KB box.
static bool make_nv_sf_map(CUtensorMap* m, const uint8_t* scales, int64_t rows, int64_t K) {
  const uint64_t blocks = static_cast<uint64_t>(rows / 128) * static_cast<uint64_t>(K / 64);
  return make_map_t(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, scales, 256, 2 * blocks, 256, 256, 8,
                    CU_TENSOR_MAP_SWIZZLE_NONE);
}

// NVFP4 operands (packed E2M1 codes [rows, K/2] K-major, tiled E4M3 scales,
// device tensor scales): the gate/up GEMM with fp32 g, u to GU and bf16 h to
// H, on CTA pairs (256 rows x 128 FFN columns of gate and of up per tile).
cudaError_t gemm_fwd_gate_up_nv(const Dims& D, const uint8_t* x_codes, const uint8_t* x_scales,
                                const float* x_g, const uint8_t* wgu_codes,
                                const uint8_t* wgu_scales, const float* wgu_g,
                                const int32_t* mtile_prefix, const int32_t* poff, void* GU,
                                void* H, int* status, cudaStream_t st) {
  const auto u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  if (D.d % 256 || D.I % 128 || !GU || !H) return cudaErrorInvalidValue;
  CUtensorMap ta, tb, tc;
  if (!make_map_t(&ta, u8, 1, x_codes, D.d / 2, D.rows_max, D.d / 2, 128, 128, sw) ||
      !make_map_t(&tb, u8, 1, wgu_codes, D.d / 2, D.E * 2 * D.I, D.d / 2, 128, 128, sw) ||
      !make_out_map(&tc, GU, 2 * D.I, D.rows_max))
    return cudaErrorInvalidValue;
  GemmArgs a = blank_args(status);
  a.store_c = 1;
  a.evict_first = 1;
  a.E = (int)D.E;
  a.n_tiles = (int)(D.I / 128);
  a.num_kb = (int)(D.d / 256);
  a.b_group_rows = (int)(2 * D.I);
  a.I = (int)D.I;
  a.mtile_prefix = mtile_prefix;
  a.poff = poff;
  a.coff = D.coff;  // unread padding rows: no epilogue
  a.out = GU;
  a.out2 = H;
  a.ks = (int)(D.d / 64);
  a.ga = x_g;
  a.gb = wgu_g;
  OutMaps om;
  memset(&om, 0, sizeof(om));
  if (!make_nv_sf_map(&om.sfa, x_scales, D.rows_max, D.d) ||
      !make_nv_sf_map(&om.sfb, wgu_scales, D.E * 2 * D.I, D.d) ||
      !make_out_map_bf16_t(&om.h, H, D.I, D.rows_max))
    return cudaErrorInvalidValue;
  return launch<256, false, false, SCHED_MGROUP, EPI_SWIGLU_FWD, SPLIT_NV, true>(
      "fwd_gate_up_swiglu", ta, tb, tc, a, max_mpairs(D) * a.n_tiles, st, nullptr, &om);
}

// An M-grouped GEMM on NVFP4 operands with fp32 rows out, on CTA pairs
// (256 x 256 tiles): O[rows_max, d] = A[rows_max, K] B_e[d, K]^T per expert
// segment, A and B packed E2M1 codes [.., K/2] with tiled scales.  The down
// projection (K = I) and the gate/up dgrad (K = 2I, B = W_gate_up transposed).
static cudaError_t grouped_nv_f32(const char* name, const Dims& D, int64_t K,
                                  const uint8_t* a_codes, const uint8_t* a_scales,
                                  const float* a_g, const uint8_t* b_codes,
                                  const uint8_t* b_scales, const float* b_g,
                                  const int32_t* mtile_prefix, const int32_t* poff, void* O,
                                  int* status, cudaStream_t st) {
  const auto u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  if (D.d % 256 || K % 256) return cudaErrorInvalidValue;
  CUtensorMap ta, tb, tc;
  if (!make_map_t(&ta, u8, 1, a_codes, K / 2, D.rows_max, K / 2, 128, 128, sw) ||
      !make_map_t(&tb, u8, 1, b_codes, K / 2, D.E * D.d, K / 2, 128, 128, sw) ||
      !make_out_map(&tc, O, D.d, D.rows_max))
    return cudaErrorInvalidValue;
  GemmArgs a = blank_args(status);
  a.E = (int)D.E;
  a.n_tiles = (int)(D.d / 256);
  a.num_kb = (int)(K / 256);
  a.b_group_rows = (int)D.d;
  a.mtile_prefix = mtile_prefix;
  a.poff = poff;
  a.coff = D.coff;  // unread padding rows: no epilogue
  a.out = O;
  a.ldo = D.d;
  a.ks = (int)(K / 64);
  a.ga = a_g;
  a.gb = b_g;
  OutMaps om;
  memset(&om, 0, sizeof(om));
  if (!make_nv_sf_map(&om.sfa, a_scales, D.rows_max, K) ||
      !make_nv_sf_map(&om.sfb, b_scales, D.E * D.d, K))
    return cudaErrorInvalidValue;
  return launch<256, false, false, SCHED_MGROUP, EPI_F32, SPLIT_NV, true>(
      name, ta, tb, tc, a, max_mpairs(D) * a.n_tiles, st, nullptr, &om);
}

cudaError_t gemm_fwd_down_nv(const Dims& D, const uint8_t* h_codes, const uint8_t* h_scales,
                             const float* h_g, const uint8_t* wd_codes, const uint8_t* wd_scales,
                             const float* wd_g, const int32_t* mtile_prefix, const int32_t* poff,
                             void* O, int* status, cudaStream_t st) {
  return grouped_nv_f32("fwd_down", D, D.I, h_codes, h_scales, h_g, wd_codes, wd_scales, wd_g,
                        mtile_prefix, poff, O, status, st);
}

cudaError_t gemm_bwd_gate_up_dgrad_nv(const Dims& D, const uint8_t* dgu_codes,
                                      const uint8_t* dgu_scales, const float* dgu_g,
                                      const uint8_t* wgu_t_codes, const uint8_t* wgu_t_scales,
                                      const float* wgu_g, const int32_t* mtile_prefix,
                                      const int32_t* poff, void* dX_perm, int* status,
                                      cudaStream_t st) {
  return grouped_nv_f32("bwd_gate_up_dgrad", D, 2 * D.I, dgu_codes, dgu_scales, dgu_g,
                        wgu_t_codes, wgu_t_scales, wgu_g, mtile_prefix, poff, dX_perm, status,
                        st);
}

cudaError_t gemm_bwd_gate_up_dgrad_mx(const Dims& D, const uint8_t* dgu_codes,
                                      const uint8_t* dgu_scales, const uint8_t* wgu_t_codes,
                                      const uint8_t* wgu_t_scales, const int32_t* mtile_prefix,
                                      const int32_t* poff, void* dX_perm, int* status,
                                      cudaStream_t st) {
  return grouped_mx_f32("bwd_gate_up_dgrad", D, 2 * D.I, dgu_codes, dgu_scales, wgu_t_codes,
                        wgu_t_scales, mtile_prefix, poff, dX_perm, status, st);
}

cudaError_t gemm_fwd_down(const Dims& D, const void* H, const void* w_down,
                          const int32_t* mtile_prefix, const int32_t* poff, void* O, int* status,
                          cudaStream_t st) {
  const int bn = (D.d % 256 == 0) ? 256 : 128;
  const bool pair = D.pair && bn == 256;
  CUtensorMap ta, tb, tc;
  if (!make_map(&ta, H, D.I, D.rows_max, D.I, 128)) return cudaErrorInvalidValue;
  if (!make_map(&tb, w_down, D.I, D.E * D.d, D.I, pair ? bn / 2 : bn))
    return cudaErrorInvalidValue;
  if (!make_out_map(&tc, O, D.d, D.rows_max)) return cudaErrorInvalidValue;
  GemmArgs a = blank_args(status);
  a.E = (int)D.E;
  a.n_tiles = (int)((D.d + bn - 1) / bn);
  a.n_valid = (int)D.d;
  a.num_kb = (int)((D.I + 63) / 64);
  a.b_group_rows = (int)D.d;
  a.mtile_prefix = mtile_prefix;
  a.poff = poff;
  a.coff = D.coff;  // unread padding rows: no epilogue
  a.out = O;  // fp32 [rows_max, d]
  a.ldo = D.d;
  const int mt = max_mtiles(D) * a.n_tiles;
  if (pair)
    return launch<256, false, false, SCHED_MGROUP, EPI_F32, SPLIT_NONE, true>(
        "fwd_down", ta, tb, tc, a, max_mpairs(D) * a.n_tiles, st);
  if (bn == 256)
    return launch<256, false, false, SCHED_MGROUP, EPI_F32>("fwd_down", ta, tb, tc, a, mt, st);
  return launch<128, false, false, SCHED_MGROUP, EPI_F32>("fwd_down", ta, tb, tc, a, mt, st);
}

cudaError_t gemm_bwd_down_dgrad(const Dims& D, const void* dY_perm, const void* w_down,
                                const int32_t* mtile_prefix, const int32_t* poff, const float* GU,
                                const float* row_w, void* dGU_hi, void* dGU_lo, void* P_hi,
                                void* P_lo, uint8_t* dgu_codes, uint8_t* dgu_scales,
                                float* dp_part, int* status,
                                cudaStream_t st) {
  const int bn = D.bn_dgrad;
  CUtensorMap ta, tb, tg;
  if (!make_map(&ta, dY_perm, D.d, D.rows_max, D.d, 128)) return cudaErrorInvalidValue;
  // fp32 g, u rows for the epilogue: boxes of 32 rows x 16 columns, 64-byte swizzle
  if (!make_map_t(&tg, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, GU, 2 * D.I, D.rows_max, 2 * D.I, 16,
                  32, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  // bf16 outputs: boxes of 32 rows x 16 columns, unswizzled
  OutMaps om;
  const auto bf16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto none = CU_TENSOR_MAP_SWIZZLE_NONE;
  if (!make_map_t(&om.dgu_hi, bf16, 2, dGU_hi, 2 * D.I, D.rows_max, 2 * D.I, 16, 32, none) ||
      !make_map_t(&om.dgu_lo, bf16, 2, dGU_lo, 2 * D.I, D.rows_max, 2 * D.I, 16, 32, none) ||
      !make_map_t(&om.p_hi, bf16, 2, P_hi, D.I, D.rows_max, D.I, 16, 32, none) ||
      !make_map_t(&om.p_lo, bf16, 2, P_lo, D.I, D.rows_max, D.I, 16, 32, none))
    return cudaErrorInvalidValue;
  // W_down_e viewed as [K = d rows, N = I columns]: N-major operand
  if (!make_map(&tb, w_down, D.I, D.E * D.d, D.I, 64)) return cudaErrorInvalidValue;
  GemmArgs a = blank_args(status);
  a.E = (int)D.E;
  a.n_tiles = (int)((D.I + bn - 1) / bn);  // columns past I: no outputs, no dp
  a.num_kb = (int)((D.d + 63) / 64);  // dY reads zeros past d
  a.b_group_rows = (int)D.d;
  a.I = (int)D.I;
  a.mtile_prefix = mtile_prefix;
  a.poff = poff;
  a.coff = D.coff;  // unread padding rows: no epilogue
  a.out = dGU_hi;
  a.out2 = P_hi;
  a.out3 = dGU_lo;
  a.out4 = P_lo;
  a.dgu_codes = dgu_codes;
  a.dgu_scales = dgu_scales;
  a.mx = D.mx ? 1 : 0;
  if (D.mx && (!dgu_codes || !dgu_scales)) return cudaErrorInvalidValue;
  a.in_gu = GU;
  a.row_w = row_w;
  a.dp_part = dp_part;
  a.np = D.np;
  const int mt = max_mtiles(D) * a.n_tiles;
  if (bn == 256 && D.pair && D.d >= kSwigluBwdDirectMinD)  // long K: operand stages first
    return launch<256, false, true, SCHED_MGROUP, EPI_SWIGLU_BWD, SPLIT_NONE, true, true>(
        "bwd_down_dgrad_swiglu", ta, tb, tg, a, max_mpairs(D) * a.n_tiles, st, nullptr, &om);
  if (bn == 256 && D.pair)
    return launch<256, false, true, SCHED_MGROUP, EPI_SWIGLU_BWD, SPLIT_NONE, true>(
        "bwd_down_dgrad_swiglu", ta, tb, tg, a, max_mpairs(D) * a.n_tiles, st, nullptr, &om);
  if (bn == 256)
    return launch<256, false, true, SCHED_MGROUP, EPI_SWIGLU_BWD>("bwd_down_dgrad_swiglu", ta, tb,
                                                                   tg, a, mt, st, nullptr, &om);
  return launch<128, false, true, SCHED_MGROUP, EPI_SWIGLU_BWD>("bwd_down_dgrad_swiglu", ta, tb,
                                                                 tg, a, mt, st, nullptr, &om);
}

cudaError_t gemm_bwd_gate_up_dgrad(const Dims& D, const void* dGU, const void* w_gate_up,
                                   const int32_t* mtile_prefix, const int32_t* poff,
                                   void* dX_perm, int* status, cudaStream_t st) {
  const int bn = (D.d % 256 == 0) ? 256 : 128;
  CUtensorMap ta, tb, tc;
  if (!make_map(&ta, dGU, 2 * D.I, D.rows_max, 2 * D.I, 128)) return cudaErrorInvalidValue;
  // W_gu_e viewed as [K = 2I rows, N = d columns]: N-major operand
  if (!make_map(&tb, w_gate_up, D.d, D.E * 2 * D.I, D.d, 64)) return cudaErrorInvalidValue;
  if (!make_out_map(&tc, dX_perm, D.d, D.rows_max)) return cudaErrorInvalidValue;
  GemmArgs a = blank_args(status);
  a.E = (int)D.E;
  a.n_tiles = (int)((D.d + bn - 1) / bn);
  a.n_valid = (int)D.d;
  a.num_kb = (int)((2 * D.I + 63) / 64);
  a.b_group_rows = (int)(2 * D.I);
  a.mtile_prefix = mtile_prefix;
  a.poff = poff;
  a.coff = D.coff;  // unread padding rows: no epilogue
  a.out = dX_perm;  // fp32 [rows_max, d]
  a.ldo = D.d;
  const int mt = max_mtiles(D) * a.n_tiles;
  if (bn == 256 && D.pair)
    return launch<256, false, true, SCHED_MGROUP, EPI_F32, SPLIT_NONE, true>(
        "bwd_gate_up_dgrad", ta, tb, tc, a, max_mpairs(D) * a.n_tiles, st);
  if (bn == 256)
    return launch<256, false, true, SCHED_MGROUP, EPI_F32>("bwd_gate_up_dgrad", ta, tb, tc, a, mt,
                                                           st);
  return launch<128, false, true, SCHED_MGROUP, EPI_F32>("bwd_gate_up_dgrad", ta, tb, tc, a, mt,
                                                         st);
}

// Double-buffered store staging for a weight gradient whose experts average at
// most 384 real rows over the launch's row spaces (six 64-row K blocks per
// output tile): a function of the shape only.
static bool short_k_wgrad(const Dims& D, int nseg) {
  const int64_t rows = D.R * (nseg > 1 ? nseg : 1);
  return rows <= 384 * D.E;
}

// K-grouped weight gradient C_e [M, N] = A_e^T B_e over the expert's padded
// rows, A_e = rows of `A_rows` (inner dim M), B_e = rows of `B_rows` (inner
// dim N).  One of the two operands comes as a hi/lo pair (`lo_is_a` selects
// which); fp32 output through TMA stores, or bf16 direct stores.
static cudaError_t wgrad(const Dims& D, const char* name, const void* A_rows, int64_t M,
                         const void* B_rows, int64_t N, const void* lo_rows, bool lo_is_a,
                         const int32_t* poff, void* out, bool accumulate, int* status,
                         cudaStream_t st, const WgradSegs& sg) {
  // B-split tiles are 128 wide so that four 48 KB stages fit
  const int bn = (!lo_is_a || N % 256 != 0) ? 128 : 256;
  const int64_t rows = D.rows_max * sg.nseg;  // operand rows of all row spaces
  CUtensorMap ta, tb, tc, tl;
  if (!make_map(&ta, A_rows, M, rows, M, 64)) return cudaErrorInvalidValue;
  if (!make_map(&tb, B_rows, N, rows, N, 64)) return cudaErrorInvalidValue;
  if (lo_is_a) {
    if (!make_map(&tl, lo_rows, M, rows, M, 64)) return cudaErrorInvalidValue;
  } else {
    if (!make_map(&tl, lo_rows, N, rows, N, 64)) return cudaErrorInvalidValue;
  }
  GemmArgs a = blank_args(status);
  a.nseg = sg.nseg;
  a.poff_stride = sg.poff_stride;
  a.seg_rows = (int)D.rows_max;
  a.coff = sg.coff;
  a.E = (int)D.E;
  a.m_tiles = (int)((M + 127) / 128);
  a.n_tiles = (int)((N + bn - 1) / bn);
  a.m_valid = (int)M;
  a.n_valid = (int)N;
  a.m_rows = (int)M;
  a.poff = poff;
  a.out = out;
  a.ldo = N;
  a.out_group_stride = M * N;
  a.accumulate = accumulate ? 1 : 0;
  // dW with the default L2 policy: evict-first measured 393 vs 383 us for the
  // fine workload's gate/up weight gradient
  a.evict_first = 0;
  const int mt = a.E * a.m_tiles * a.n_tiles;
  if (D.wgrad_bf16) {
    // bf16 dW: the fp32 accumulation rounded once, stored through TMA
    if (accumulate) return cudaErrorInvalidValue;  // accumulation is fp32 only
    if (!make_out_map_bf16(&tc, out, N, D.E * M)) return cudaErrorInvalidValue;
    if (!lo_is_a)
      return launch<128, true, true, SCHED_KGROUP, EPI_BF16_TMA, SPLIT_B>(name, ta, tb, tc, a, mt,
                                                                          st, &tl);
    if (bn == 256 && D.pair && a.m_tiles % 2 == 0)
      return launch<256, true, true, SCHED_KGROUP, EPI_BF16_TMA, SPLIT_A, true>(
          name, ta, tb, tc, a, mt / 2, st, &tl);
    if (bn == 256)
      return launch<256, true, true, SCHED_KGROUP, EPI_BF16_TMA, SPLIT_A>(name, ta, tb, tc, a, mt,
                                                                          st, &tl);
    return launch<128, true, true, SCHED_KGROUP, EPI_BF16_TMA, SPLIT_A>(name, ta, tb, tc, a, mt,
                                                                        st, &tl);
  }
  if (!make_out_map(&tc, out, N, D.E * M)) return cudaErrorInvalidValue;
  const bool db = short_k_wgrad(D, sg.nseg);
  if (!lo_is_a) {
    if (db)
      return launch<128, true, true, SCHED_KGROUP, EPI_F32, SPLIT_B, false, true>(
          name, ta, tb, tc, a, mt, st, &tl);
    return launch<128, true, true, SCHED_KGROUP, EPI_F32, SPLIT_B>(name, ta, tb, tc, a, mt, st,
                                                                   &tl);
  }
  if (bn == 256 && D.pair && a.m_tiles % 2 == 0) {
    if (db)
      return launch<256, true, true, SCHED_KGROUP, EPI_F32, SPLIT_A, true, true>(
          name, ta, tb, tc, a, mt / 2, st, &tl);
    return launch<256, true, true, SCHED_KGROUP, EPI_F32, SPLIT_A, true>(name, ta, tb, tc, a,
                                                                         mt / 2, st, &tl);
  }
  if (bn == 256) {
    if (db)
      return launch<256, true, true, SCHED_KGROUP, EPI_F32, SPLIT_A, false, true>(
          name, ta, tb, tc, a, mt, st, &tl);
    return launch<256, true, true, SCHED_KGROUP, EPI_F32, SPLIT_A>(name, ta, tb, tc, a, mt, st,
                                                                   &tl);
  }
  if (db)
    return launch<128, true, true, SCHED_KGROUP, EPI_F32, SPLIT_A, false, true>(
        name, ta, tb, tc, a, mt, st, &tl);
  return launch<128, true, true, SCHED_KGROUP, EPI_F32, SPLIT_A>(name, ta, tb, tc, a, mt, st, &tl);
}

cudaError_t gemm_wgrad_down(const Dims& D, const void* dY_perm, const void* P_hi,
                            const void* P_lo, const int32_t* poff, void* dw_down,
                            bool accumulate, int* status, cudaStream_t st, const WgradSegs& sg) {
  // dW_down_e [d, I] (+)= dY_e^T [d x rows] * (P_hi + P_lo)_e [rows x I],  P = p h
  if (D.d % 256 != 0)
    return wgrad(D, "bwd_down_wgrad", dY_perm, D.d, P_hi, D.I, P_lo, false, poff, dw_down,
                 accumulate, status, st, sg);
  // computed as its transpose, (P_hi + P_lo)_e^T [I x rows] * dY_e [rows x d],
  // so that the hi/lo pair is the A operand and the tile is 128 x 256 like
  // the gate/up wgrad's; the epilogue stores each block transposed
  const int64_t rows = D.rows_max * sg.nseg;
  CUtensorMap ta, tb, tc, tl;
  if (!make_map(&ta, P_hi, D.I, rows, D.I, 64)) return cudaErrorInvalidValue;
  if (!make_map(&tl, P_lo, D.I, rows, D.I, 64)) return cudaErrorInvalidValue;
  if (!make_map(&tb, dY_perm, D.d, rows, D.d, 64)) return cudaErrorInvalidValue;
  if (D.wgrad_bf16 && accumulate) return cudaErrorInvalidValue;  // accumulation is fp32 only
  if (!(D.wgrad_bf16 ? make_out_map_bf16_t(&tc, dw_down, D.I, D.E * D.d)
                     : make_out_map(&tc, dw_down, D.I, D.E * D.d)))
    return cudaErrorInvalidValue;
  GemmArgs a = blank_args(status);
  a.nseg = sg.nseg;
  a.poff_stride = sg.poff_stride;
  a.seg_rows = (int)D.rows_max;
  a.coff = sg.coff;
  a.E = (int)D.E;
  a.m_tiles = (int)((D.I + 127) / 128);
  a.m_valid = (int)D.I;
  a.n_tiles = (int)(D.d / 256);
  a.m_rows = (int)D.I;
  a.poff = poff;
  a.out = dw_down;
  a.ldo = D.d;  // rows of one expert's block in the [E*d, I] view
  a.accumulate = accumulate ? 1 : 0;
  // dW with the default L2 policy: evict-first measured 393 vs 383 us for the
  // fine workload's gate/up weight gradient
  a.evict_first = 0;
  const int mt = a.E * a.m_tiles * a.n_tiles;
  if (D.wgrad_bf16) {
    if (D.pair && a.m_tiles % 2 == 0)
      return launch<256, true, true, SCHED_KGROUP, EPI_BF16_T, SPLIT_A, true>(
          "bwd_down_wgrad", ta, tb, tc, a, mt / 2, st, &tl);
    return launch<256, true, true, SCHED_KGROUP, EPI_BF16_T, SPLIT_A>("bwd_down_wgrad", ta, tb,
                                                                      tc, a, mt, st, &tl);
  }
  const bool db = short_k_wgrad(D, sg.nseg);
  if (D.pair && a.m_tiles % 2 == 0) {
    if (db)
      return launch<256, true, true, SCHED_KGROUP, EPI_F32_T, SPLIT_A, true, true>(
          "bwd_down_wgrad", ta, tb, tc, a, mt / 2, st, &tl);
    return launch<256, true, true, SCHED_KGROUP, EPI_F32_T, SPLIT_A, true>(
        "bwd_down_wgrad", ta, tb, tc, a, mt / 2, st, &tl);
  }
  if (db)
    return launch<256, true, true, SCHED_KGROUP, EPI_F32_T, SPLIT_A, false, true>(
        "bwd_down_wgrad", ta, tb, tc, a, mt, st, &tl);
  return launch<256, true, true, SCHED_KGROUP, EPI_F32_T, SPLIT_A>("bwd_down_wgrad", ta, tb, tc,
                                                                   a, mt, st, &tl);
}

cudaError_t gemm_wgrad_gate_up(const Dims& D, const void* dGU_hi, const void* dGU_lo,
                               const void* X_perm, const int32_t* poff, void* dw_gate_up,
                               bool accumulate, int* status, cudaStream_t st,
                               const WgradSegs& sg) {
  // dW_gu_e [2I, d] (+)= (dGU_hi + dGU_lo)_e^T [2I x rows] * X_e [rows x d]
  return wgrad(D, "bwd_gate_up_wgrad", dGU_hi, 2 * D.I, X_perm, D.d, dGU_lo, true, poff,
               dw_gate_up, accumulate, status, st, sg);
}

cudaError_t gemm_router_wgrad(const Dims& D, const void* x, const void* dl_hi, const void* dl_lo,
                              const int32_t* rw_off, float* part, int* status, cudaStream_t st) {
  // partial s [E_pad, d] = (dl_hi + dl_lo)^T x over tokens rw_off[s] .. rw_off[s+1]
  // (the K-grouped schedule with one group per token chunk); tokens >= T of the
  // last chunk are zero-filled by the TMA on both operands
  if (D.T == 0) return cudaSuccess;
  const RwSplit rw = router_wgrad_split(D);
  const int64_t M = router_e_pad(D);
  const int bn = router_wgrad_bn(D);
  CUtensorMap ta, tb, tc, tl;
  if (!make_map(&ta, dl_hi, M, D.T, M, 64)) return cudaErrorInvalidValue;
  if (!make_map(&tl, dl_lo, M, D.T, M, 64)) return cudaErrorInvalidValue;
  if (!make_map(&tb, x, D.d, D.T, D.d, 64)) return cudaErrorInvalidValue;
  if (!make_out_map(&tc, part, D.d, rw.ks * M)) return cudaErrorInvalidValue;
  GemmArgs a = blank_args(status);
  a.E = rw.ks;
  a.m_tiles = (int)(M / 128);
  a.n_tiles = (int)((D.d + bn - 1) / bn);
  a.n_valid = (int)D.d;
  a.m_rows = (int)M;
  a.poff = rw_off;
  a.out = part;
  a.ldo = D.d;
  a.out_group_stride = M * D.d;
  const int mt = a.E * a.m_tiles * a.n_tiles;
  if (bn == 256)
    return launch<256, true, true, SCHED_KGROUP, EPI_F32, SPLIT_A>("router_wgrad", ta, tb, tc, a,
                                                                   mt, st, &tl);
  return launch<128, true, true, SCHED_KGROUP, EPI_F32, SPLIT_A>("router_wgrad", ta, tb, tc, a,
                                                                 mt, st, &tl);
}

cudaError_t launch_router_logits(const Dims& D, const void* x, const void* w_router,
                                 float* logits, int* status, cudaStream_t st) {
  // logits [T, E] fp32 = x [T,d] * W_r[E,d]^T; rows >= T and columns >= E
  // are zero-filled by the TMA and masked at the store.
  if (D.T == 0) return cudaSuccess;
  const int bn = (D.E > 128) ? 256 : 128;
  CUtensorMap ta, tb;
  if (!make_map(&ta, x, D.d, D.T, D.d, 128)) return cudaErrorInvalidValue;
  if (!make_map(&tb, w_router, D.d, D.E, D.d, bn)) return cudaErrorInvalidValue;
  GemmArgs a = blank_args(status);
  a.E = 1;
  a.m_tiles = (int)((D.T + 127) / 128);
  a.n_tiles = (int)((D.E + bn - 1) / bn);
  a.num_kb = (int)((D.d + 63) / 64);
  a.m_valid = (int)D.T;
  a.n_valid = (int)D.E;
  a.out = logits;
  a.ldo = D.E;
  // split K so that about 128 CTAs share the work; split s writes its
  // partial logits to logits + s*T*E and the top-k sums them in order
  a.k_splits = router_k_splits(D);
  a.num_kb /= a.k_splits;
  a.out_group_stride = D.T * D.E;
  const int mt = a.m_tiles * a.n_tiles * a.k_splits;
  if (bn == 256)
    return launch<256, false, false, SCHED_DENSE, EPI_F32>("router_logits", ta, tb, ta, a, mt, st);
  return launch<128, false, false, SCHED_DENSE, EPI_F32>("router_logits", ta, tb, ta, a, mt, st);
}

cudaError_t gemm_dense_bf16(int64_t M, int64_t N, int64_t K, const void* A, bool a_mn,
                            const void* B, bool b_mn, void* C, int* status, cudaStream_t st) {
  const int bn = (N % 256 == 0) ? 256 : 128;
  CUtensorMap ta, tb;
  if (!a_mn) {
    if (!make_map(&ta, A, K, M, K, 128)) return cudaErrorInvalidValue;
  } else {
    if (!make_map(&ta, A, M, K, M, 64)) return cudaErrorInvalidValue;
  }
  if (!b_mn) {
    if (!make_map(&tb, B, K, N, K, bn)) return cudaErrorInvalidValue;
  } else {
    if (!make_map(&tb, B, N, K, N, 64)) return cudaErrorInvalidValue;
  }
  GemmArgs a = blank_args(status);
  a.E = 1;
  a.m_tiles = (int)(M / 128);
  a.n_tiles = (int)(N / bn);
  a.num_kb = (int)(K / 64);
  a.m_valid = (int)M;
  a.n_valid = (int)N;
  a.out = C;
  a.ldo = N;
  const int mt = a.m_tiles * a.n_tiles;
  if (a_mn) {
    if (bn == 256)
      return launch<256, true, true, SCHED_DENSE, EPI_BF16>("dense_gemm", ta, tb, ta, a, mt, st);
    return launch<128, true, true, SCHED_DENSE, EPI_BF16>("dense_gemm", ta, tb, ta, a, mt, st);
  }
  if (b_mn) {
    if (bn == 256)
      return launch<256, false, true, SCHED_DENSE, EPI_BF16>("dense_gemm", ta, tb, ta, a, mt, st);
    return launch<128, false, true, SCHED_DENSE, EPI_BF16>("dense_gemm", ta, tb, ta, a, mt, st);
  }
  if (bn == 256)
    return launch<256, false, false, SCHED_DENSE, EPI_BF16>("dense_gemm", ta, tb, ta, a, mt, st);
  return launch<128, false, false, SCHED_DENSE, EPI_BF16>("dense_gemm", ta, tb, ta, a, mt, st);
}

}  // namespace mok
