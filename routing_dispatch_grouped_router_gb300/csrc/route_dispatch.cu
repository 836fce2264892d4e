// Router top-k, dispatch plan, row dispatch (dispatch / reverse-combine),
// combine, reverse-dispatch with the router backward, router weight grad.
//
// Sources (page title, section):
//   [gtnt] "MoK揭秘：NVL72上大规模MoE训练工程方案深度解读", §1.1: a gating
//     network (router) picks the best few experts for every token.
//   [dothoosh] "Cursor Mixture-of-Kittens cuts MoE training latency by 5.8x",
//     "MoK technical details", bullet "Hybrid communication": forward =
//     dispatch then combine; backward = reverse-combine then
//     reverse-dispatch (across GPUs the pages pull the dispatch; within one
//     HBM the dispatch here is driven by the token so that each token row is
//     read once); bullet "Ring buffer logic": no token is dropped and no
//     buffer is sized by the CPU.
//   [aikraft] "Cursor MoK: revolution in MoE model training on NVL72", §03:
//     the CPU is kept off the critical path (no host synchronisation).
//
// Every kernel here is deterministic: integer atomics only where their order
// cannot change the result (counts, bit sets), and every floating-point sum
// runs in a fixed order.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mok_internal.h"
#include "plan.cuh"
#include "ptx.cuh"

namespace mok {

// ------------------------------------------------------------------ router --

// One warp per token (the body is topk_token in plan.cuh).
template <int PER>
__global__ void router_topk_kernel(const float* __restrict__ logits, const float* __restrict__ bias,
                                   int T, int E, int k, int nsplit,
                                   int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                                   int* status) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= T) return;
  topk_token<PER>(logits, bias, T, E, k, nsplit, warp, lane, topk_idx, topk_w, nullptr, status);
}

cudaError_t launch_router_topk(const Dims& D, const float* logits, const float* bias,
                               int32_t* topk_idx, float* topk_w, int* status, cudaStream_t st) {
  if (D.T == 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks = (D.T * 32 + threads - 1) / threads;
  ProfScope prof("router_topk", st);
  const int T = static_cast<int>(D.T), E = static_cast<int>(D.E), ns = router_k_splits(D);
  const unsigned g = static_cast<unsigned>(blocks);
  if (E <= 32)
    router_topk_kernel<1><<<g, threads, 0, st>>>(logits, bias, T, E, D.k, ns, topk_idx, topk_w, status);
  else if (E <= 64)
    router_topk_kernel<2><<<g, threads, 0, st>>>(logits, bias, T, E, D.k, ns, topk_idx, topk_w, status);
  else if (E <= 128)
    router_topk_kernel<4><<<g, threads, 0, st>>>(logits, bias, T, E, D.k, ns, topk_idx, topk_w, status);
  else if (E <= 256)
    router_topk_kernel<8><<<g, threads, 0, st>>>(logits, bias, T, E, D.k, ns, topk_idx, topk_w, status);
  else
    router_topk_kernel<16><<<g, threads, 0, st>>>(logits, bias, T, E, D.k, ns, topk_idx, topk_w,
                                                  status);
  count_launch();
  return cudaGetLastError();
}

// ----------------------------------------------------------- dispatch plan --

__global__ void plan_hist_kernel(const int32_t* __restrict__ topk_idx, int T, int E, int k,
                                 int32_t* __restrict__ block_counts, int* status) {
  __shared__ int cnt[kMaxExperts];
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int t = blockIdx.x * kPlanBlock + threadIdx.x;
  if (t < T) {
    int ids[kMaxTopK];
    const uint32_t valid = load_row(topk_idx + static_cast<long long>(t) * k, k, E, ids);
#pragma unroll
    for (int s = 0; s < kMaxTopK; ++s)
      if (valid & (1u << s)) atomicAdd(&cnt[ids[s]], 1);
    if (valid != (1u << k) - 1u) set_status(status, MOK_ERR_DEVICE_INDEX);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    block_counts[static_cast<long long>(blockIdx.x) * E + e] = cnt[e];
}

// One CTA (the body is plan_scan_body in plan.cuh).
__global__ void plan_scan_kernel(const int32_t* __restrict__ block_counts, int nb, int E,
                                 int32_t* __restrict__ block_base, int32_t* __restrict__ counts,
                                 int32_t* __restrict__ offsets, int32_t* __restrict__ poff,
                                 int32_t* __restrict__ mtile_prefix, int32_t* __restrict__ ptok,
                                 float* __restrict__ row_w) {
  plan_scan_body(block_counts, nb, E, block_base, counts, offsets, poff, mtile_prefix, ptok,
                 row_w);
}

// One CTA of kPlanBlock threads per block of tokens (the body is
// plan_place_body in plan.cuh).
__global__ void plan_place_kernel(const int32_t* __restrict__ topk_idx,
                                  const float* __restrict__ topk_w, int T, int E, int k,
                                  const int32_t* __restrict__ block_base,
                                  const int32_t* __restrict__ offsets,
                                  const int32_t* __restrict__ poff, int32_t* __restrict__ pos,
                                  int32_t* __restrict__ token_of_row, int32_t* __restrict__ ppos,
                                  int32_t* __restrict__ ptok, float* __restrict__ row_w) {
  plan_place_body(blockIdx.x, topk_idx, topk_w, T, E, k, block_base, offsets, poff, pos,
                  token_of_row, ppos, ptok, row_w);
}

cudaError_t launch_plan(const Dims& D, const int32_t* topk_idx, const float* topk_w,
                        int32_t* block_counts, int32_t* block_base, const PlanOut& o, int* status,
                        cudaStream_t st) {
  const int nb = static_cast<int>(D.nb);
  const int E = static_cast<int>(D.E), T = static_cast<int>(D.T);
  if (nb > 0) {
    ProfScope prof("plan_hist", st);
    plan_hist_kernel<<<nb, kPlanBlock, 0, st>>>(topk_idx, T, E, D.k, block_counts, status);
    count_launch();
  }
  {
    ProfScope prof("plan_scan", st);
    plan_scan_kernel<<<1, 1024, 0, st>>>(block_counts, nb, E, block_base, o.counts, o.offsets,
                                         o.padded_offsets, o.mtile_prefix, o.ptok, o.row_w);
    count_launch();
  }
  if (nb > 0) {
    ProfScope prof("plan_place", st);
    plan_place_kernel<<<nb, kPlanBlock, 0, st>>>(topk_idx, topk_w, T, E, D.k, block_base,
                                                 o.offsets, o.padded_offsets, o.pos,
                                                 o.token_of_row, o.ppos, o.ptok, o.row_w);
    count_launch();
  }
  return cudaGetLastError();
}

// ----------------------------------------------------------- row dispatch --

// Dispatch of token rows into the padded expert-major row space, staged
// through TMA and driven by the token: padded row r < padded_offsets[E]
// receives src[t] where r is one of t's k padded positions (ppos[t, s]), and
// zeros if r is a padding row.  Each token row is read from HBM once (one bulk
// copy global -> shared completing on its slot's mbarrier) and stored to its
// k rows from the same slot (k bulk stores, one bulk group).  CTA b (one
// warp) takes tokens b, b + G, b + 2G, ... (G CTAs) through a ring of `nslot`
// row-sized slots; a slot is refilled kDispatchLag tokens after its stores
// were issued.  The k positions of each token come through a 128-token shared
// ring that the warp refills 32 tokens at a time (each lane loads one token's
// positions), each refill's loads issued 16 tokens before they are written,
// so the issuing lane never waits on an index load.  Afterwards the CTA
// stores a zeroed slot to the padding rows among rows b, b + G, ... that the
// plan marks as read (token -1: up to each expert's next 64-row boundary);
// rows marked -2 are left as they are.
constexpr int kDispatchLag = 2;
constexpr int kDispatchMaxSlots = 32;
constexpr int kDispatchIdx = 128;

__global__ void __launch_bounds__(32) dispatch_rows_kernel(
    const uint8_t* __restrict__ src, const int32_t* __restrict__ ppos, int k,
    const int32_t* __restrict__ ptok, const int32_t* __restrict__ poff_end, int T,
    uint32_t row_bytes, int nslot, uint8_t* __restrict__ dst, int* status) {
  grid_dep_launch();  // a GEMM after this kernel may start its prologue
  extern __shared__ __align__(128) uint8_t gsm[];
  __shared__ __align__(8) uint64_t full[kDispatchMaxSlots];
  __shared__ int s_pos[kDispatchIdx][kMaxTopK];
  const int lane = threadIdx.x;
  const long long G = gridDim.x;
  const long long first = blockIdx.x;
  const long long n = (T > first) ? (T - first + G - 1) / G : 0;  // tokens of this CTA
  const int never = 0;
  if (lane == 0) {
    for (int s = 0; s < nslot; ++s) mbar_init(&full[s], 1);
    fence_barrier_init();
  }
  // positions of this CTA's tokens 0..95; tokens 96..127 come with the first refill
  for (int i = lane; i < kDispatchIdx - 32; i += 32)
#pragma unroll
    for (int p = 0; p < kMaxTopK; ++p)
      s_pos[i][p] = (i < n && p < k) ? ppos[(first + i * G) * k + p] : -1;
  __syncwarp();
  const uint64_t keep = l2_policy_evict_last(), stream = l2_policy_evict_first();
  auto issue = [&](long long j) {  // lane 0: token j's row into its slot
    const int s = static_cast<int>(j % nslot);
    mbar_arrive_expect_tx(&full[s], row_bytes);
    bulk_load_hint(gsm + static_cast<size_t>(s) * row_bytes,
                   src + (first + j * G) * static_cast<long long>(row_bytes), row_bytes, &full[s],
                   keep);
  };
  if (lane == 0) {
    const long long pro = n < nslot ? n : nslot;
    for (long long j = 0; j < pro; ++j) issue(j);
  }
  int pend[kMaxTopK];  // the position refill in flight (lane's token)
#pragma unroll
  for (int p = 0; p < kMaxTopK; ++p) pend[p] = -1;
  for (long long j = 0; j < n; ++j) {
    __syncwarp();
    if ((j & 31) == 0) {
      const long long jj = j + (kDispatchIdx - 32) + lane;
#pragma unroll
      for (int p = 0; p < kMaxTopK; ++p)
        pend[p] = (jj < n && p < k) ? ppos[(first + jj * G) * k + p] : -1;
    } else if ((j & 31) == 16) {
      const int e = static_cast<int>((j - 16 + (kDispatchIdx - 32) + lane) % kDispatchIdx);
#pragma unroll
      for (int p = 0; p < kMaxTopK; ++p) s_pos[e][p] = pend[p];
    }
    __syncwarp();
    if (lane == 0) {
      const int s = static_cast<int>(j % nslot);
      const uint32_t par = static_cast<uint32_t>((j / nslot) & 1);
      if (!mbar_wait(&full[s], par, &never)) set_status(status, MOK_ERR_DEVICE_TIMEOUT);
      const uint8_t* slot = gsm + static_cast<size_t>(s) * row_bytes;
      for (int p = 0; p < k; ++p) {
        const int r = s_pos[j % kDispatchIdx][p];
        if (r >= 0) bulk_store_hint(dst + static_cast<long long>(r) * row_bytes, slot, row_bytes,
                                    stream);
      }
      bulk_commit();
      // token j - lag's stores have read their slot: refill it with token j - lag + nslot
      const long long jr = j - kDispatchLag + nslot;
      if (j >= kDispatchLag && jr < n) {
        bulk_wait_read<kDispatchLag>();
        issue(jr);
      }
    }
  }
  // padding rows that are read: a zeroed slot stored to every row
  // r = first + i G marked -1
  if (lane == 0) bulk_wait_read<0>();  // every slot has been read out
  __syncwarp();
  for (uint32_t i = lane * 16; i < row_bytes; i += 32 * 16)
    *reinterpret_cast<uint4*>(gsm + i) = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  __syncwarp();
  const long long P = *poff_end;
  const long long m = (P > first) ? (P - first + G - 1) / G : 0;
  for (long long i0 = 0; i0 < m; i0 += 32) {
    const long long i = i0 + lane;
    const int t = i < m ? ptok[first + i * G] : 0;
    const unsigned pad = __ballot_sync(0xffffffffu, i < m && t == -1);
    if (lane == 0 && pad) {
      for (int l = 0; l < 32; ++l)
        if (pad & (1u << l))
          bulk_store_hint(dst + (first + (i0 + l) * G) * static_cast<long long>(row_bytes), gsm,
                          row_bytes, stream);
      bulk_commit();
    }
  }
  if (lane == 0) bulk_wait_all<0>();
}

cudaError_t launch_dispatch_rows(const Dims& D, const void* src, const int32_t* ppos,
                                 const int32_t* ptok, const int32_t* padded_offsets, void* dst,
                                 int* status, cudaStream_t st) {
  if (D.T == 0) return cudaSuccess;
  if (D.k > kMaxTopK) return cudaErrorInvalidValue;
  const uint32_t row_bytes = static_cast<uint32_t>(D.d * 2);
  // about 200 KB of slots per SM, split over up to four CTAs of at least six
  // slots each (d <= 16384: one CTA of six 32 KB slots at the largest)
  constexpr int kSmemPerSm = 200 * 1024;
  int per_sm = static_cast<int>(kSmemPerSm / (6 * row_bytes));
  per_sm = per_sm > 4 ? 4 : (per_sm < 1 ? 1 : per_sm);
  int nslot = static_cast<int>((kSmemPerSm / per_sm) / row_bytes);
  nslot = nslot > kDispatchMaxSlots ? kDispatchMaxSlots : nslot;
  if (nslot < kDispatchLag + 2) return cudaErrorInvalidValue;
  const int smem = nslot * static_cast<int>(row_bytes);
  // set on every launch: the attribute belongs to the current device
  cudaError_t e = cudaFuncSetAttribute(dispatch_rows_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  long long grid = static_cast<long long>(num_sms_current_device()) * per_sm;
  if (grid > D.T) grid = D.T;
  ProfScope prof("dispatch_rows", st);
  dispatch_rows_kernel<<<static_cast<unsigned>(grid), 32, smem, st>>>(
      static_cast<const uint8_t*>(src), ppos, static_cast<int>(D.k), ptok, padded_offsets + D.E,
      static_cast<int>(D.T), row_bytes, nslot, static_cast<uint8_t*>(dst), status);
  count_launch();
  return cudaGetLastError();
}

// ----------------------------------------------------------------- combine --

__device__ __forceinline__ void axpy4(float (&acc)[4], float w, float4 v) {
  acc[0] = fmaf(w, v.x, acc[0]);
  acc[1] = fmaf(w, v.y, acc[1]);
  acc[2] = fmaf(w, v.z, acc[2]);
  acc[3] = fmaf(w, v.w, acc[3]);
}

__device__ __forceinline__ void add4(float (&acc)[4], float4 v) {
  acc[0] += v.x;
  acc[1] += v.y;
  acc[2] += v.z;
  acc[3] += v.w;
}

__device__ __forceinline__ float4 ld_nc_f4(const float4* p) {
  float4 v;
  asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float4 bf16x4_to_f4(uint2 w) {
  return make_float4(bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y));
}

// Stores 4 consecutive values of row `row` (fp32 or bf16 output).
template <bool BF16_OUT>
__device__ __forceinline__ void store4(void* out, long long row, int dq, int c,
                                       const float (&a)[4]) {
  if (BF16_OUT) {
    reinterpret_cast<uint2*>(out)[row * dq + c] =
        make_uint2(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]));
  } else {
    reinterpret_cast<float4*>(out)[row * dq + c] = make_float4(a[0], a[1], a[2], a[3]);
  }
}

// One CTA per token: y_t = sum_{s=0..k-1} p[t,s] * O[ppos[t,s]], fp32 in slot
// order (O is fp32).
template <bool BF16_OUT>
__global__ void combine_kernel(const float4* __restrict__ O, const int32_t* __restrict__ ppos,
                               const float* __restrict__ topk_w, int k, int dq, void* y) {
  grid_dep_launch();  // a GEMM after this kernel may start its prologue
  __shared__ int s_row[kMaxTopK];
  __shared__ float s_w[kMaxTopK];
  const long long t = blockIdx.x;
  if (threadIdx.x < k) {
    s_row[threadIdx.x] = ppos[t * k + threadIdx.x];
    s_w[threadIdx.x] = topk_w[t * k + threadIdx.x];
  }
  __syncthreads();
  for (int c = threadIdx.x; c < dq; c += blockDim.x) {
    float4 v[kMaxTopK];
#pragma unroll
    for (int s = 0; s < kMaxTopK; ++s)
      if (s < k && s_row[s] >= 0) v[s] = ld_nc_f4(O + static_cast<long long>(s_row[s]) * dq + c);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int s = 0; s < kMaxTopK; ++s)
      if (s < k && s_row[s] >= 0) axpy4(acc, s_w[s], v[s]);
    store4<BF16_OUT>(y, t, dq, c, acc);
  }
}

static int row_threads(int nvec) {
  int th = nvec < 256 ? nvec : 256;
  th = (th + 31) / 32 * 32;
  return th < 32 ? 32 : th;
}

cudaError_t launch_combine(const Dims& D, const float* O, const int32_t* ppos, const float* topk_w,
                           void* y, cudaStream_t st) {
  if (D.T == 0) return cudaSuccess;
  const int dq = static_cast<int>(D.d / 4);
  ProfScope prof("combine", st);
  if (D.act_bf16)
    combine_kernel<true><<<static_cast<unsigned>(D.T), row_threads(dq), 0, st>>>(
        reinterpret_cast<const float4*>(O), ppos, topk_w, D.k, dq, y);
  else
    combine_kernel<false><<<static_cast<unsigned>(D.T), row_threads(dq), 0, st>>>(
        reinterpret_cast<const float4*>(O), ppos, topk_w, D.k, dq, y);
  count_launch();
  return cudaGetLastError();
}

// -------------------------------------------------------- reverse dispatch --

// One CTA per token.  Router backward first:
//   dp_s = sum_j dp_part[row_s, j]            (fixed j order; = <dy, O_s>)
//   dl_s = p_s (dp_s - sum_i p_i dp_i)        (softmax over the chosen k)
// then dx_t = sum_s (dX_perm[row_s] + dl_s * W_r[e_s])   in slot order.
template <bool BF16_OUT>
__global__ void reverse_dispatch_kernel(const float4* __restrict__ dXp,
                                        const int32_t* __restrict__ ppos,
                                        const int32_t* __restrict__ topk_idx,
                                        const float* __restrict__ topk_w,
                                        const float* __restrict__ dp_part, int np,
                                        const uint2* __restrict__ Wr, int k, int dq, void* dx,
                                        __nv_bfloat16* __restrict__ dl_hi,
                                        __nv_bfloat16* __restrict__ dl_lo, int e_pad,
                                        int32_t* __restrict__ rw_off, int rw_chunks,
                                        int rw_chunk_rows) {
  grid_dep_launch();  // a GEMM after this kernel may start its prologue
  __shared__ int s_row[kMaxTopK];
  __shared__ int s_e[kMaxTopK];
  __shared__ float s_dl[kMaxTopK];
  const long long t = blockIdx.x;
  const int s = threadIdx.x;  // slot, for the first k threads
  int row = -1;
  if (s < k) {
    row = ppos[t * k + s];
    s_row[s] = row;
    s_e[s] = topk_idx[t * k + s];
  }
  __syncthreads();
  // the k rows' loads of one column all in flight, then the sum in slot order
  float4 xr[kMaxTopK];
  uint2 wr[kMaxTopK];
  auto load_rows = [&](int c) {
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j < k && s_row[j] >= 0) {
        xr[j] = ld_nc_f4(dXp + static_cast<long long>(s_row[j]) * dq + c);
        asm volatile("ld.global.nc.v2.b32 {%0, %1}, [%2];"
                     : "=r"(wr[j].x), "=r"(wr[j].y)
                     : "l"(Wr + static_cast<long long>(s_e[j]) * dq + c));
      }
    }
  };
  // the first column's loads go out before the routing-weight gradient is known
  const int c0 = threadIdx.x;
  if (c0 < dq) load_rows(c0);
  if (threadIdx.x < 32) {
    float p = 0.f, dp = 0.f;
    if (s < k) {
      p = topk_w[t * k + s];
      if (row >= 0) {
        const float* q = dp_part + static_cast<long long>(row) * np;
#pragma unroll 4
        for (int j = 0; j < np; ++j) dp += q[j];
      }
    }
    // sum_i p_i dp_i, summed in slot order by every lane
    float pdp = 0.f;
    for (int i = 0; i < kMaxTopK; ++i) {
      const float pi = __shfl_sync(0xffffffffu, p, i);
      const float di = __shfl_sync(0xffffffffu, dp, i);
      if (i < k) pdp = fmaf(pi, di, pdp);
    }
    if (s < k) s_dl[s] = (row >= 0) ? p * (dp - pdp) : 0.f;
  }
  if (blockIdx.x == 0)
    for (int j = threadIdx.x; j <= rw_chunks; j += blockDim.x) rw_off[j] = j * rw_chunk_rows;
  __syncthreads();
  // dense dl row of the router-weight gradient, as a bf16 hi/lo pair
  for (int j = threadIdx.x; j < e_pad; j += blockDim.x) {
    float v = 0.f;
    for (int i = 0; i < k; ++i)
      if (s_e[i] == j) v = s_dl[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    dl_hi[t * e_pad + j] = hi;
    dl_lo[t * e_pad + j] = __float2bfloat16_rn(v - __bfloat162float(hi));
  }
  for (int c = c0; c < dq; c += blockDim.x) {
    if (c != c0) load_rows(c);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j < k && s_row[j] >= 0) {
        add4(acc, xr[j]);
        axpy4(acc, s_dl[j], bf16x4_to_f4(wr[j]));
      }
    }
    store4<BF16_OUT>(dx, t, dq, c, acc);
  }
}

cudaError_t launch_reverse_dispatch(const Dims& D, const float* dX_perm, const int32_t* ppos,
                                    const int32_t* topk_idx, const float* topk_w,
                                    const float* dp_part, const void* w_router, void* dx,
                                    void* dl_hi, void* dl_lo, int32_t* rw_off, cudaStream_t st) {
  if (D.T == 0) return cudaSuccess;
  const int dq = static_cast<int>(D.d / 4);
  const int th = row_threads(dq);
  const RwSplit rw = router_wgrad_split(D);
  const int e_pad = static_cast<int>(router_e_pad(D));
  auto* hi = static_cast<__nv_bfloat16*>(dl_hi);
  auto* lo = static_cast<__nv_bfloat16*>(dl_lo);
  ProfScope prof("reverse_dispatch", st);
  if (D.act_bf16)
    reverse_dispatch_kernel<true><<<static_cast<unsigned>(D.T), th, 0, st>>>(
        reinterpret_cast<const float4*>(dX_perm), ppos, topk_idx, topk_w, dp_part, D.np,
        static_cast<const uint2*>(w_router), D.k, dq, dx, hi, lo, e_pad, rw_off, rw.ks,
        rw.kb * 64);
  else
    reverse_dispatch_kernel<false><<<static_cast<unsigned>(D.T), th, 0, st>>>(
        reinterpret_cast<const float4*>(dX_perm), ppos, topk_idx, topk_w, dp_part, D.np,
        static_cast<const uint2*>(w_router), D.k, dq, dx, hi, lo, e_pad, rw_off, rw.ks,
        rw.kb * 64);
  count_launch();
  return cudaGetLastError();
}

// ------------------------------------------------------ router weight grad --

// dW_r = the sum of the ks partial products of the router-weight gradient
// GEMM, added in chunk order (then + the previous dW_r with accumulate); ks = 0
// (no tokens) gives zeros.  The
// partial of chunk s holds rows e < E of an [E padded to 128, d] block at
// part + s * split4 float4s; thread i takes float4 i of dW_r [E, d].
template <bool BF16_OUT>
__global__ void router_wgrad_reduce_kernel(const float4* __restrict__ part, int ks,
                                           long long split4, long long n4, void* dw,
                                           int accumulate) {
  grid_dep_launch();  // a GEMM after this kernel may start its prologue
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    float4 acc = ks > 0 ? ld_nc_f4(part + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 1; s < ks; ++s) {
      const float4 v = ld_nc_f4(part + s * split4 + i);
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    if (BF16_OUT) {
      reinterpret_cast<uint2*>(dw)[i] =
          make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
    } else {
      float4* q = reinterpret_cast<float4*>(dw) + i;
      if (accumulate) {
        const float4 a = *q;
        acc.x += a.x; acc.y += a.y; acc.z += a.z; acc.w += a.w;
      }
      *q = acc;
    }
  }
}

cudaError_t launch_router_wgrad_reduce(const Dims& D, const float* part, void* dw_router,
                                       bool accumulate, cudaStream_t st) {
  if (accumulate && D.wgrad_bf16) return cudaErrorInvalidValue;
  // no tokens: no partials, dW_r = 0 (or unchanged with accumulate)
  const int ks = D.T == 0 ? 0 : router_wgrad_split(D).ks;
  const long long n4 = D.E * D.d / 4;
  const long long split4 = router_e_pad(D) * D.d / 4;
  long long blocks = (n4 + 255) / 256;
  const long long cap = static_cast<long long>(num_sms_current_device()) * 8;
  if (blocks > cap) blocks = cap;
  const auto* p4 = reinterpret_cast<const float4*>(part);
  ProfScope prof("router_wgrad_reduce", st);
  if (D.wgrad_bf16)
    router_wgrad_reduce_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, st>>>(
        p4, ks, split4, n4, dw_router, 0);
  else
    router_wgrad_reduce_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, st>>>(
        p4, ks, split4, n4, dw_router, accumulate ? 1 : 0);
  count_launch();
  return cudaGetLastError();
}

// -------------------------------------------------------------- zero fill --

constexpr int kFillChunk = 16384;  // bytes per bulk store

// Zeroes [dst, dst + bytes) with bulk asynchronous stores from a zeroed
// shared-memory chunk, the store path of dispatch_rows_kernel: chunk c is
// written by CTA c % gridDim.x, the ragged tail (a multiple of 16 bytes) by
// the last CTA.  At most 9 stores per CTA are in flight.
__global__ void __launch_bounds__(32) fill_zero_kernel(uint8_t* __restrict__ dst,
                                                       unsigned long long bytes) {
  extern __shared__ __align__(128) uint8_t s_zero[];
  grid_dep_launch();
  for (int i = threadIdx.x; i < kFillChunk / 16; i += 32)
    reinterpret_cast<uint4*>(s_zero)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  __syncwarp();
  if (threadIdx.x != 0) return;
  const unsigned long long n = bytes / kFillChunk;
  for (unsigned long long c = blockIdx.x; c < n; c += gridDim.x) {
    bulk_store(dst + c * kFillChunk, s_zero, kFillChunk);
    bulk_commit();
    bulk_wait_read<8>();
  }
  const uint32_t rem = static_cast<uint32_t>(bytes - n * kFillChunk);
  if (rem != 0 && blockIdx.x == gridDim.x - 1) {
    bulk_store(dst + n * kFillChunk, s_zero, rem);
    bulk_commit();
  }
  bulk_wait_all<0>();
}

cudaError_t launch_fill_zero(void* dst, size_t bytes, cudaStream_t st) {
  if (bytes == 0) return cudaSuccess;
  const unsigned long long chunks = bytes / kFillChunk;
  const unsigned long long cap = static_cast<unsigned long long>(num_sms_current_device()) * 8;
  const unsigned grid = static_cast<unsigned>(chunks == 0 ? 1 : (chunks < cap ? chunks : cap));
  ProfScope prof("fill_zero", st);
  fill_zero_kernel<<<grid, 32, kFillChunk, st>>>(static_cast<uint8_t*>(dst),
                                                  static_cast<unsigned long long>(bytes));
  count_launch();
  return cudaGetLastError();
}

// --------------------------------------------------------- bounded waits --

// Waits on an mbarrier phase that nothing completes: the bounded wait gives up
// after its limit and records MOK_ERR_DEVICE_TIMEOUT, as a GEMM would.
__global__ void bounded_wait_selftest_kernel(int* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_barrier_init();
  const int never = 0;
  if (!mbar_wait(&bar, 0, &never)) set_status(status, MOK_ERR_DEVICE_TIMEOUT);
  // complete the phase so the barrier is left consistent
  mbar_arrive(&bar);
}

cudaError_t launch_bounded_wait_selftest(int* status, cudaStream_t st) {
  bounded_wait_selftest_kernel<<<1, 32, 0, st>>>(status);
  count_launch();
  return cudaGetLastError();
}

}  // namespace mok
