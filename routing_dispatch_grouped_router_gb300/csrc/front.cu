// The router's top-k selection and the whole dispatch plan in one persistent
// kernel, driven by a schedule table.
//
// Sources (page title, section):
//   [dothoosh] "Cursor Mixture-of-Kittens cuts MoE training latency by 5.8x",
//     "MoK technical details", bullet "Hybrid communication": one schedule
//     table drives the phases of the MoE layer inside a single persistent
//     kernel, at a small share of its time; here it covers the steps between
//     the router's logit GEMM and the row dispatch.
//   [gtnt] "MoK揭秘：NVL72上大规模MoE训练工程方案深度解读", §1.1 (the router).
//
// The table lists steps in order; every CTA of a cooperative grid walks it:
//   TOPK   items = tokens: one warp per token (topk_token), every warp of the
//          grid striding over the tokens; each token's experts are added to
//          its 256-token block's counts with integer atomics.  A CTA that
//          finishes its tokens arrives on a counter; the last to arrive is the
//          one that runs the next step.
//   SCAN   one item, run by the last CTA of TOPK (plan_scan_body); it then
//          raises a flag.
//   PLACE  items = 256-token blocks (plan_place_body), after the flag.
// Only PLACE waits (on the flag, bounded by the library's wait limit; a wait
// that gives up reports MOK_ERR_DEVICE_TIMEOUT).  The grid is launched
// cooperatively, so every CTA is resident and the last one always runs.
// The steps run the same device bodies as the stand-alone kernels, in an
// order that gives each the same inputs, so every result is bitwise equal to
// the four-launch path (the block counts are integer sums).
#include <cuda_runtime.h>

#include "mok_internal.h"
#include "plan.cuh"
#include "ptx.cuh"

namespace mok {

enum FrontStepKind : int { FRONT_TOPK = 0, FRONT_SCAN = 1, FRONT_PLACE = 2 };
constexpr int kFrontMaxSteps = 4;
struct FrontStep {
  int kind;
  int items;
};
struct FrontTable {
  int n;
  FrontStep step[kFrontMaxSteps];
};

struct FrontArgs {
  const float* logits;  // [nsplit][T][E] split-K partial logits
  const float* bias;    // [E] or NULL
  int T, E, k, nsplit, nb;
  int32_t* topk_idx;
  float* topk_w;
  int32_t* block_counts;  // [nb][E], zero at launch
  int32_t* block_base;    // [nb][E]
  PlanOut o;
  unsigned* sync;  // [0]: CTAs past TOPK, [1]: SCAN written; zero at launch
  int* status;
  FrontTable table;
};

// Thread-0 wait until *flag == 1 (acquire), bounded by the wait limit.
__device__ __forceinline__ bool wait_flag_acquire(const unsigned* flag) {
  const uint64_t t0 = global_timer_ns();
  uint32_t spins = 0;
  while (true) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    if (v == 1u) return true;
    if ((++spins & 63u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

template <int PER>
__global__ void __launch_bounds__(kPlanBlock) front_kernel(FrontArgs a) {
  __shared__ int s_last, s_ok;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kWarps = kPlanBlock / 32;
  for (int i = 0; i < a.table.n; ++i) {
    const FrontStep st = a.table.step[i];
    if (st.kind == FRONT_TOPK) {
      const long long nw = static_cast<long long>(gridDim.x) * kWarps;
      for (long long t = static_cast<long long>(blockIdx.x) * kWarps + warp; t < st.items;
           t += nw)
        topk_token<PER>(a.logits, a.bias, a.T, a.E, a.k, a.nsplit, static_cast<int>(t), lane,
                        a.topk_idx, a.topk_w, a.block_counts, a.status);
      __syncthreads();
      if (threadIdx.x == 0) {
        __threadfence();  // this CTA's selections and counts, before its arrival
        const unsigned prev = atomicAdd(&a.sync[0], 1u);
        s_last = prev == gridDim.x - 1;
        if (s_last) __threadfence();  // every other CTA's, before the scan reads them
      }
      __syncthreads();
    } else if (st.kind == FRONT_SCAN) {
      if (s_last) {
        plan_scan_body(a.block_counts, a.nb, a.E, a.block_base, a.o.counts, a.o.offsets,
                       a.o.padded_offsets, a.o.mtile_prefix, a.o.ptok, a.o.row_w);
        __syncthreads();
        if (threadIdx.x == 0) {
          __threadfence();
          atomicExch(&a.sync[1], 1u);
        }
      }
    } else {  // FRONT_PLACE
      if (threadIdx.x == 0) {
        s_ok = wait_flag_acquire(&a.sync[1]);
        if (!s_ok) set_status(a.status, MOK_ERR_DEVICE_TIMEOUT);
        __threadfence();
      }
      __syncthreads();
      if (!s_ok) return;
      for (int b = blockIdx.x; b < st.items; b += gridDim.x)
        plan_place_body(b, a.topk_idx, a.topk_w, a.T, a.E, a.k, a.block_base, a.o.offsets,
                        a.o.padded_offsets, a.o.pos, a.o.token_of_row, a.o.ppos, a.o.ptok,
                        a.o.row_w);
    }
  }
}

template <int PER>
static cudaError_t launch_front(const FrontArgs& a, int max_grid, cudaStream_t st) {
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, front_kernel<PER>,
                                                                kPlanBlock, 0);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorLaunchOutOfResources;
  long long grid = static_cast<long long>(num_sms_current_device()) * (per_sm < 2 ? per_sm : 2);
  if (grid > max_grid) grid = max_grid;
  if (grid < 1) grid = 1;
  FrontArgs args = a;
  void* params[] = {&args};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(front_kernel<PER>),
                                     dim3(static_cast<unsigned>(grid)), dim3(kPlanBlock), params,
                                     0, st);
}

cudaError_t launch_route_plan(const Dims& D, const float* logits, const float* bias,
                              int32_t* topk_idx, float* topk_w, int32_t* block_counts,
                              int32_t* block_base, unsigned* sync, const PlanOut& o, int* status,
                              cudaStream_t st) {
  if (D.k > kMaxTopK || D.E > kMaxExperts) return cudaErrorInvalidValue;
  const int nb = static_cast<int>(D.nb), E = static_cast<int>(D.E);
  // the arrival counter, the flag and the block counts start at zero: one
  // memset when the counts follow the 256-byte sync block, as the layer lays
  // them out
  const size_t counts_bytes = static_cast<size_t>(nb) * E * 4;
  cudaError_t e;
  if (reinterpret_cast<char*>(block_counts) == reinterpret_cast<char*>(sync) + 256) {
    e = cudaMemsetAsync(sync, 0, 256 + counts_bytes, st);
  } else {
    e = cudaMemsetAsync(sync, 0, 256, st);
    if (e == cudaSuccess && counts_bytes) e = cudaMemsetAsync(block_counts, 0, counts_bytes, st);
  }
  if (e != cudaSuccess) return e;
  FrontArgs a;
  a.logits = logits;
  a.bias = bias;
  a.T = static_cast<int>(D.T);
  a.E = E;
  a.k = D.k;
  a.nsplit = router_k_splits(D);
  a.nb = nb;
  a.topk_idx = topk_idx;
  a.topk_w = topk_w;
  a.block_counts = block_counts;
  a.block_base = block_base;
  a.o = o;
  a.sync = sync;
  a.status = status;
  // the schedule table of this shape
  a.table.n = 3;
  a.table.step[0] = {FRONT_TOPK, static_cast<int>(D.T)};
  a.table.step[1] = {FRONT_SCAN, 1};
  a.table.step[2] = {FRONT_PLACE, nb};
  // enough CTAs for one warp per token (and at least one per 256-token block)
  const long long want_tok = (D.T + kPlanBlock / 32 - 1) / (kPlanBlock / 32);
  const int max_grid = static_cast<int>(want_tok > nb ? (want_tok > (1 << 20) ? (1 << 20) : want_tok)
                                                      : (nb > 0 ? nb : 1));
  ProfScope prof("route_plan", st);
  if (E <= 32) e = launch_front<1>(a, max_grid, st);
  else if (E <= 64) e = launch_front<2>(a, max_grid, st);
  else if (E <= 128) e = launch_front<4>(a, max_grid, st);
  else if (E <= 256) e = launch_front<8>(a, max_grid, st);
  else e = launch_front<16>(a, max_grid, st);
  count_launch();
  return e;
}

}  // namespace mok
