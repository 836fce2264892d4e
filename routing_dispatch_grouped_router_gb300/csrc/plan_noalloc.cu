// Dispatch plan for callers that cannot hand the library any scratch memory.
//
// The regular mok_moe_dispatch_plan takes a caller-allocated workspace for
// its per-block counts, padded offsets and padded positions.  This variant
// keeps that scratch in one fixed device array defined in this file, so the
// caller passes only the inputs and outputs.  Every device that loads the
// library holds the array (kNoAllocScratchBytes) until the process exits.
#include <cuda_runtime.h>
#include <string.h>

#include "mok_internal.h"

namespace mok {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB

// File-scope device scratch.  In host code `g_noalloc_scratch` names a host
// stand-in, not device memory: its device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The array's device address in the current device's context.  Resolved on
// every call (cudaGetSymbolAddress allocates nothing): an address cached per
// device would go stale if the caller's framework tore the context down and
// built a new one.
static mok_status noalloc_scratch(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MOK_ERR_CUDA;
  *out = p;
  return MOK_OK;
}

}  // namespace mok

using namespace mok;

extern "C" mok_status mok_moe_dispatch_plan_noalloc(const mok_moe_desc* desc,
                                                    const int32_t* topk_idx, int32_t* counts,
                                                    int32_t* offsets, int32_t* pos,
                                                    int32_t* token_of_row, int32_t* status,
                                                    void* stream) {
  Dims D;
  mok_status s = make_dims(desc, &D);
  if (s != MOK_OK) return s;
  if (D.nmb != 1) return MOK_ERR_UNSUPPORTED;
  if ((!topk_idx && D.T > 0) || !counts || !offsets || (!pos && D.T > 0) ||
      (!token_of_row && D.T > 0))
    return MOK_ERR_INVALID_ARG;
  StageWs W;
  stage_layout(D, &W);
  // this entry point needs no router logits: the scratch ends where they start
  const size_t need = W.logits;
  if (need > kNoAllocScratchBytes) return MOK_ERR_SCRATCH_LIMIT;
  s = mok_check_device();
  if (s != MOK_OK) return s;
  void* scratch = nullptr;
  s = noalloc_scratch(&scratch);
  if (s != MOK_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(scratch);
  int* dstatus = status ? status : reinterpret_cast<int*>(base + W.status);
  if (cudaMemsetAsync(dstatus, 0, sizeof(int), st) != cudaSuccess) return MOK_ERR_CUDA;
  // slots skipped as invalid keep pos = -1; the rows they would have taken
  // stay unwritten, so the inverse map starts at -1
  if (D.R > 0 &&
      cudaMemsetAsync(token_of_row, 0xFF, static_cast<size_t>(D.R) * 4, st) != cudaSuccess)
    return MOK_ERR_CUDA;
  PlanOut o;
  o.counts = counts;
  o.offsets = offsets;
  o.pos = pos;
  o.token_of_row = token_of_row;
  o.padded_offsets = reinterpret_cast<int32_t*>(base + W.padded_offsets);
  o.mtile_prefix = reinterpret_cast<int32_t*>(base + W.mtile_prefix);
  o.ppos = reinterpret_cast<int32_t*>(base + W.ppos);
  o.ptok = reinterpret_cast<int32_t*>(base + W.ptok);
  o.row_w = nullptr;
  if (launch_plan(D, topk_idx, nullptr, reinterpret_cast<int32_t*>(base + W.block_counts),
                  reinterpret_cast<int32_t*>(base + W.block_base), o, dstatus,
                  st) != cudaSuccess)
    return MOK_ERR_CUDA;
  return MOK_OK;
}
