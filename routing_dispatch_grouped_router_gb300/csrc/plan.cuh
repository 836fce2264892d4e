// Device bodies of the router's top-k selection and of the dispatch plan.
// The stand-alone kernels (route_dispatch.cu) and the fused front-end kernel
// (front.cu) both run these, so the two paths compute bit for bit the same.
//
// Sources (page title, section):
//   [gtnt] "MoK揭秘：NVL72上大规模MoE训练工程方案深度解读", §1.1: a router
//     picks the best few experts for every token.
//   [dothoosh] "Cursor Mixture-of-Kittens cuts MoE training latency by 5.8x",
//     "MoK technical details", bullet "Ring buffer logic": no token is
//     dropped; bullet "Hybrid communication": dispatch into expert order.
#pragma once

#include <cuda_runtime.h>

#include "mok_internal.h"
#include "ptx.cuh"

namespace mok {

// One warp selects token `token`'s experts: add the bias, pick the k largest
// logits (exact ties to the lower expert index; NaN counts as -inf and is
// reported), softmax over the chosen k.  Slots come out in descending logit
// order.  PER = logits per lane: ceil(E / 32) rounded up to a power of two.
// `logits` holds nsplit split-K partial products [nsplit][T][E], summed in
// split order.  block_counts (or NULL): lane 0 adds the token's experts to the
// counts of its kPlanBlock-token block, [T / kPlanBlock][E] (integer atomics:
// the totals do not depend on their order).
template <int PER>
__device__ __forceinline__ void topk_token(const float* __restrict__ logits,
                                           const float* __restrict__ bias, int T, int E, int k,
                                           int nsplit, int token, int lane,
                                           int32_t* __restrict__ topk_idx,
                                           float* __restrict__ topk_w,
                                           int32_t* __restrict__ block_counts, int* status) {
  float v[PER];
  bool nan_seen = false;
  const float* row = logits + static_cast<long long>(token) * E;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int e = j * 32 + lane;
    float x = -INFINITY;
    if (e < E) {
      // the split-K partial logits, summed in split order
      x = row[e];
      for (int sp = 1; sp < nsplit; ++sp) x += row[static_cast<long long>(sp) * T * E + e];
      if (bias) x += bias[e];
      if (x != x) {
        nan_seen = true;
        x = -INFINITY;
      }
    }
    v[j] = x;
  }
  if (__any_sync(0xffffffffu, nan_seen) && lane == 0) set_status(status, MOK_ERR_DEVICE_NONFINITE);
  // slot loops unrolled over kMaxTopK (guarded by k) so that the selected
  // values and experts stay in registers
  float sel_v[kMaxTopK];
  int sel_e[kMaxTopK];
#pragma unroll
  for (int s = 0; s < kMaxTopK; ++s) {
    if (s >= k) break;
    // best of this lane: experts are visited in increasing index order, so a
    // strict '>' keeps the lower index on equal values
    float bv = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int e = j * 32 + lane;
      if (e < E && (v[j] > bv || (v[j] == bv && e < be))) {
        bv = v[j];
        be = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oe = __shfl_xor_sync(0xffffffffu, be, off);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
      }
    }
    sel_v[s] = bv;
    sel_e[s] = be;
    // remove the winner
#pragma unroll
    for (int j = 0; j < PER; ++j)
      if (j * 32 + lane == be) v[j] = NAN;  // NaN never wins a comparison
  }
  if (lane == 0) {
    const float m = sel_v[0];
    float den = 0.f;
    float ex[kMaxTopK];
#pragma unroll
    for (int s = 0; s < kMaxTopK; ++s) {
      if (s >= k) break;
      ex[s] = (sel_v[s] == -INFINITY) ? (m == -INFINITY ? 1.f : 0.f) : expf(sel_v[s] - m);
      den += ex[s];
    }
    const float inv = 1.0f / den;
#pragma unroll
    for (int s = 0; s < kMaxTopK; ++s) {
      if (s >= k) break;
      topk_idx[static_cast<long long>(token) * k + s] = sel_e[s];
      topk_w[static_cast<long long>(token) * k + s] = ex[s] * inv;
    }
    if (block_counts) {
      int32_t* bc = block_counts + static_cast<long long>(token / kPlanBlock) * E;
#pragma unroll
      for (int s = 0; s < kMaxTopK; ++s) {
        if (s >= k) break;
        atomicAdd(bc + sel_e[s], 1);
      }
    }
  }
}

// A token's k experts, loaded once into registers, and the mask of its valid
// slots: bit s is set when slot s names an expert in range that no earlier
// slot of the token names (a router never repeats; a caller's table might).
__device__ __forceinline__ uint32_t load_row(const int32_t* row, int k, int E,
                                             int (&ids)[kMaxTopK]) {
#pragma unroll
  for (int s = 0; s < kMaxTopK; ++s) ids[s] = s < k ? row[s] : -1;
  uint32_t valid = 0;
#pragma unroll
  for (int s = 0; s < kMaxTopK; ++s) {
    bool ok = s < k && ids[s] >= 0 && ids[s] < E;
#pragma unroll
    for (int j = 0; j < s; ++j) ok = ok && ids[j] != ids[s];
    valid |= ok ? (1u << s) : 0u;
  }
  return valid;
}

// One CTA (any size that is a multiple of 32): per-expert totals and
// per-(block, expert) bases, then the exclusive scans (plain and padded to
// 128 rows), the 128-row tile prefix, and the padding rows of every expert
// segment (weight 0).  Padding rows up to the next multiple of 64 rows get
// token -1: the weight-gradient GEMMs read them (their K loops run in 64-row
// blocks), so they must hold zeros.  The rest, up to the 128-row boundary,
// get token -2: only whole-tile GEMMs read them, for output rows that nothing
// reads, so they are never written.
__device__ __forceinline__ void plan_scan_body(const int32_t* __restrict__ block_counts, int nb,
                                               int E, int32_t* __restrict__ block_base,
                                               int32_t* __restrict__ counts,
                                               int32_t* __restrict__ offsets,
                                               int32_t* __restrict__ poff,
                                               int32_t* __restrict__ mtile_prefix,
                                               int32_t* __restrict__ ptok,
                                               float* __restrict__ row_w) {
  __shared__ int s_cnt[kMaxExperts];
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_poff[kMaxExperts + 1];
  __shared__ int s_pair[kMaxExperts + 1];
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    // eight blocks' counts in flight at a time, then their running sum
    int run = 0;
    for (int b0 = 0; b0 < nb; b0 += 8) {
      int c[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        c[j] = b0 + j < nb ? block_counts[static_cast<long long>(b0 + j) * E + e] : 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (b0 + j < nb) block_base[static_cast<long long>(b0 + j) * E + e] = run;
        run += c[j];
      }
    }
    s_cnt[e] = run;
    counts[e] = run;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    // warp scan: lane owns experts [lane*PER, lane*PER+PER)
    const int lane = threadIdx.x;
    constexpr int PER = kMaxExperts / 32;
    // row tiles of an expert, and pairs of row tiles (an odd count rounds up)
    auto tiles = [](int c) { return (c + kRowPad - 1) / kRowPad; };
    int sum = 0, psum = 0, qsum = 0;
    for (int j = 0; j < PER; ++j) {
      const int e = lane * PER + j;
      if (e < E) {
        sum += s_cnt[e];
        psum += tiles(s_cnt[e]) * kRowPad;
        qsum += (tiles(s_cnt[e]) + 1) / 2;
      }
    }
    int incl = sum, pincl = psum, qincl = qsum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, incl, off);
      const int b = __shfl_up_sync(0xffffffffu, pincl, off);
      const int c = __shfl_up_sync(0xffffffffu, qincl, off);
      if (lane >= off) {
        incl += a;
        pincl += b;
        qincl += c;
      }
    }
    int run = incl - sum, prun = pincl - psum, qrun = qincl - qsum;
    for (int j = 0; j < PER; ++j) {
      const int e = lane * PER + j;
      if (e < E) {
        s_off[e] = run;
        s_poff[e] = prun;
        s_pair[e] = qrun;
        run += s_cnt[e];
        prun += tiles(s_cnt[e]) * kRowPad;
        qrun += (tiles(s_cnt[e]) + 1) / 2;
      }
    }
    if (lane == 31) {
      s_off[E] = run;
      s_poff[E] = prun;
      s_pair[E] = qrun;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    offsets[e] = s_off[e];
    poff[e] = s_poff[e];
    mtile_prefix[e] = s_poff[e] / kRowPad;
    mtile_prefix[E + 1 + e] = s_pair[e];  // prefix of tile pairs
  }
  // padding rows of each expert segment
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  for (int e = warp; e < E; e += nw) {
    const int a = s_poff[e] + s_cnt[e], b = s_poff[e + 1];
    const int z = s_poff[e] + (s_cnt[e] + 63) / 64 * 64;  // end of the zeroed rows
    for (int r = a + lane; r < b; r += 32) {
      ptok[r] = r < z ? -1 : -2;
      if (row_w) row_w[r] = 0.f;
    }
  }
}

// Stable placement of block `blk` (kPlanBlock tokens, one per thread of a
// kPlanBlock-thread CTA): the rank of token t among the tokens of its block
// routed to the same expert is the number of set bits below t in that
// expert's 256-bit membership mask.
__device__ __forceinline__ void plan_place_body(int blk, const int32_t* __restrict__ topk_idx,
                                                const float* __restrict__ topk_w, int T, int E,
                                                int k, const int32_t* __restrict__ block_base,
                                                const int32_t* __restrict__ offsets,
                                                const int32_t* __restrict__ poff,
                                                int32_t* __restrict__ pos,
                                                int32_t* __restrict__ token_of_row,
                                                int32_t* __restrict__ ppos,
                                                int32_t* __restrict__ ptok,
                                                float* __restrict__ row_w) {
  constexpr int W = kPlanBlock / 32;  // 8 mask words per expert
  __shared__ uint32_t mask[kMaxExperts * W];
  // per expert: first row of this block's tokens, plain and padded
  __shared__ int s_row[kMaxExperts], s_prow[kMaxExperts];
  for (int i = threadIdx.x; i < E * W; i += blockDim.x) mask[i] = 0u;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int b = block_base[static_cast<long long>(blk) * E + e];
    s_row[e] = offsets[e] + b;
    s_prow[e] = poff[e] + b;
  }
  __syncthreads();
  const int t = blk * kPlanBlock + threadIdx.x;
  const int word = threadIdx.x >> 5, bit = threadIdx.x & 31;
  int ids[kMaxTopK];
  uint32_t valid = 0;
  if (t < T) {
    valid = load_row(topk_idx + static_cast<long long>(t) * k, k, E, ids);
#pragma unroll
    for (int s = 0; s < kMaxTopK; ++s)
      if (valid & (1u << s)) atomicOr(&mask[ids[s] * W + word], 1u << bit);
  }
  __syncthreads();
  if (t < T) {
#pragma unroll
    for (int s = 0; s < kMaxTopK; ++s) {
      if (s >= k) break;
      const long long ts = static_cast<long long>(t) * k + s;
      if (!(valid & (1u << s))) {
        if (pos) pos[ts] = -1;
        ppos[ts] = -1;
        continue;
      }
      const int e = ids[s];
      int rank = __popc(mask[e * W + word] & ((1u << bit) - 1u));
      for (int w = 0; w < word; ++w) rank += __popc(mask[e * W + w]);
      const int p = s_row[e] + rank;
      const int pp = s_prow[e] + rank;
      if (pos) pos[ts] = p;
      if (token_of_row) token_of_row[p] = t;
      ppos[ts] = pp;
      ptok[pp] = t;
      if (row_w) row_w[pp] = topk_w[ts];
    }
  }
  // the block's shared masks are reused by the CTA's next block
  __syncthreads();
}

}  // namespace mok
