// C ABI of the MoE layer (declared in include/mok.h): argument checks, buffer
// layouts, and the order of kernels of the forward and the backward.
//
// Sources (page title, section):
//   [dothoosh] "Cursor Mixture-of-Kittens cuts MoE training latency by 5.8x",
//     "MoK technical details", bullet "Hybrid communication": forward =
//     dispatch -> expert GEMMs -> combine; backward = reverse-combine ->
//     grouped dgrad/wgrad -> reverse-dispatch; bullet "Ring buffer logic":
//     fixed-size buffers, nothing sized by the CPU from routing results.
//   [aikraft] "Cursor MoK: revolution in MoE model training on NVL72", §03:
//     no CPU-GPU synchronisation on the critical path.  Every buffer and grid
//     here is sized from (T, k, E, d, I) bounds; no count is read back.
#include <nvtx3/nvToolsExt.h>
#include <cuda_runtime.h>
#include <string.h>

#include <atomic>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "mok_internal.h"

namespace mok {

static std::atomic<int32_t> g_launches{0};
void count_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
void reset_launch_count() { g_launches.store(0, std::memory_order_relaxed); }
int32_t launch_count() { return g_launches.load(std::memory_order_relaxed); }

// ---------------------------------------------------------------- profiling --
struct ProfRec {
  const char* name;
  cudaEvent_t a, b;
};
static bool g_prof = false;
static std::vector<ProfRec> g_recs;
static std::vector<cudaEvent_t> g_pool;
static size_t g_pool_used = 0;

static cudaEvent_t pool_event() {
  if (g_pool_used == g_pool.size()) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    g_pool.push_back(e);
  }
  return g_pool[g_pool_used++];
}

// Every kernel launch is also an NVTX range (domain-less, named as the kernel
// step), and each forward / backward call one around them, so a system
// profiler's timeline shows the layer's steps; without a tool attached the
// NVTX calls return at once.
void prof_begin(const char* name, cudaStream_t st) {
  nvtxRangePushA(name);
  if (!g_prof) return;
  ProfRec r{name, pool_event(), pool_event()};
  if (!r.a || !r.b) return;
  cudaEventRecord(r.a, st);
  g_recs.push_back(r);
}

void prof_end(cudaStream_t st) {
  nvtxRangePop();
  if (!g_prof || g_recs.empty()) return;
  cudaEventRecord(g_recs.back().b, st);
}

// An NVTX range for the span of a scope (one forward or backward call).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

int num_sms_current_device() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 148;
  }
  return cache[dev];
}

mok_status mok_check_device() {
  static int ok_cache[64] = {0};  // 0 unknown, 1 ok, 2 bad
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOK_ERR_NO_DEVICE;
  if (ok_cache[dev] == 0) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    ok_cache[dev] = (major == 10 && minor == 3) ? 1 : 2;
  }
  return ok_cache[dev] == 1 ? MOK_OK : MOK_ERR_NO_DEVICE;
}

static inline size_t al(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

mok_status make_dims(const mok_moe_desc* desc, Dims* out) {
  if (!desc || !out) return MOK_ERR_INVALID_ARG;
  const mok_moe_desc& d = *desc;
  if (d.T < 0 || d.d <= 0 || d.E <= 0 || d.I <= 0 || d.k <= 0) return MOK_ERR_INVALID_ARG;
  if (d.dtype != MOK_BF16 && d.dtype != MOK_MXFP8 && d.dtype != MOK_NVFP4)
    return MOK_ERR_UNSUPPORTED;
  if (d.dtype == MOK_NVFP4 &&
      ((d.flags & (MOK_FLAG_SINGLE_CTA_GEMM | MOK_FLAG_RECOMPUTE_GATE_UP)) || d.d % 256 ||
       d.I % 256))
    return MOK_ERR_UNSUPPORTED;
  if (d.mb_tokens < 0 || d.ring_slots < 0) return MOK_ERR_INVALID_ARG;
  if (d.flags & ~(MOK_FLAG_BF16_ACT_OUT | MOK_FLAG_BF16_WGRAD_OUT | MOK_FLAG_ACCUMULATE_WGRAD |
                  MOK_FLAG_RECOMPUTE_GATE_UP | MOK_FLAG_SINGLE_CTA_GEMM |
                  MOK_FLAG_RECOMPUTE_DISPATCH))
    return MOK_ERR_UNSUPPORTED;
  if ((d.flags & MOK_FLAG_ACCUMULATE_WGRAD) && (d.flags & MOK_FLAG_BF16_WGRAD_OUT))
    return MOK_ERR_UNSUPPORTED;  // accumulation is fp32 only
  if (d.E > kMaxExperts || d.k > kMaxTopK || d.k > d.E) return MOK_ERR_UNSUPPORTED;
  // d and I: multiples of 32 from 128 on (ragged GEMM tiles: zero-filled loads,
  // unstored columns); MXFP8 operands: multiples of 128 (its code tiles)
  if (d.d % 32 != 0 || d.d < 128 || d.I % 32 != 0 || d.I < 128) return MOK_ERR_UNSUPPORTED;
  if (d.dtype == MOK_MXFP8 && (d.d % 128 != 0 || d.I % 128 != 0)) return MOK_ERR_UNSUPPORTED;
  if (d.d > 16384 || d.I > 16384) return MOK_ERR_UNSUPPORTED;
  if (d.T * d.k >= (1LL << 31) / 2) return MOK_ERR_UNSUPPORTED;
  Dims D;
  D.T_total = d.T;
  D.nmb = 1;
  D.ring = 1;
  int64_t mb = d.T;
  if (d.mb_tokens > 0 && d.T > 0) {
    if (d.T % d.mb_tokens != 0) return MOK_ERR_UNSUPPORTED;
    if (d.flags & MOK_FLAG_BF16_WGRAD_OUT) return MOK_ERR_UNSUPPORTED;  // fp32 accumulation
    mb = d.mb_tokens;
    D.nmb = static_cast<int>(d.T / d.mb_tokens);
    if (d.ring_slots > D.nmb) return MOK_ERR_UNSUPPORTED;
    D.ring = d.ring_slots > 0 ? d.ring_slots : D.nmb;
  } else if (d.ring_slots > 1) {
    return MOK_ERR_UNSUPPORTED;
  }
  D.T = mb;
  D.d = d.d;
  D.E = d.E;
  D.I = d.I;
  D.k = d.k;
  D.R = D.T * d.k;
  const int64_t segs = D.R < D.E ? D.R : D.E;
  D.rows_max = (D.R + (kRowPad - 1) * segs + kRowPad - 1) / kRowPad * kRowPad;
  D.nb = (D.T + kPlanBlock - 1) / kPlanBlock;
  D.bn_dgrad = (D.I % 256 == 0) ? 256 : 128;
  D.np = static_cast<int>((D.I + D.bn_dgrad - 1) / D.bn_dgrad) * 2;
  D.act_bf16 = (d.flags & MOK_FLAG_BF16_ACT_OUT) != 0;
  D.wgrad_bf16 = (d.flags & MOK_FLAG_BF16_WGRAD_OUT) != 0;
  D.mx = d.dtype == MOK_MXFP8;
  D.accumulate = (d.flags & MOK_FLAG_ACCUMULATE_WGRAD) != 0;
  D.recompute_gu = (d.flags & MOK_FLAG_RECOMPUTE_GATE_UP) != 0;
  D.pair = (d.flags & MOK_FLAG_SINGLE_CTA_GEMM) == 0;
  D.nv = d.dtype == MOK_NVFP4;
  // NVFP4 quantises the token rows through the row map and keeps no
  // dispatched rows; its BF16 backward gathers them again
  D.recompute_dispatch = ((d.flags & MOK_FLAG_RECOMPUTE_DISPATCH) != 0 && !D.mx) || D.nv;
  // every row index and element offset used in 32-bit arithmetic must fit
  if (D.rows_max * 2 * D.I >= (1LL << 40)) return MOK_ERR_UNSUPPORTED;
  if (D.rows_max >= (1LL << 31) / 2) return MOK_ERR_UNSUPPORTED;
  *out = D;
  return MOK_OK;
}

namespace {
struct Bump {
  size_t o = 0;
  size_t take(size_t bytes) {
    const size_t at = o;
    o += (bytes + 255) & ~static_cast<size_t>(255);
    return at;
  }
};
}  // namespace

void block_layout(const Dims& D, BlockL* B) {
  Bump b;
  const size_t Tk = static_cast<size_t>(D.T) * D.k;
  const size_t E = static_cast<size_t>(D.E);
  const size_t rows = static_cast<size_t>(D.rows_max);
  B->topk_idx = b.take(Tk * 4);
  B->topk_w = b.take(Tk * 4);
  B->counts = b.take(E * 4);
  B->offsets = b.take((E + 1) * 4);
  B->pos = b.take(Tk * 4);
  B->token_of_row = b.take(Tk * 4);
  B->padded_offsets = b.take((E + 1) * 4);
  B->mtile_prefix = b.take((E + 1) * 8);  // tiles, then tile pairs
  B->padded_pos = b.take(Tk * 4);
  B->padded_token = b.take(rows * 4);
  B->row_weight = b.take(rows * 4);
  B->gate_up = D.recompute_gu ? 0 : b.take(rows * 2 * D.I * 4);  // fp32
  B->total = b.o;
}

// saved = status | nmb micro-batch blocks | ring slots of dispatched rows
void saved_layout(const Dims& D, mok_saved_layout* L, size_t* mtile_prefix_off) {
  BlockL B;
  block_layout(D, &B);
  const size_t base = 256;
  // MXFP8 keeps no dispatched bf16 rows (its quantisers read the token rows
  // through the row -> token map), nor does the dispatch-recompute mode
  const bool keep_rows = !D.mx && !D.recompute_dispatch;
  const size_t slot = keep_rows ? static_cast<size_t>(D.rows_max) * D.d * 2 : 0;
  const size_t slot_al = (slot + 255) & ~static_cast<size_t>(255);
  const size_t ring0 = base + B.total * D.nmb;
  L->status = 0;
  L->topk_idx = base + B.topk_idx;
  L->topk_w = base + B.topk_w;
  L->counts = base + B.counts;
  L->offsets = base + B.offsets;
  L->pos = base + B.pos;
  L->token_of_row = base + B.token_of_row;
  L->padded_offsets = base + B.padded_offsets;
  if (mtile_prefix_off) *mtile_prefix_off = base + B.mtile_prefix;
  L->padded_pos = base + B.padded_pos;
  L->padded_token = base + B.padded_token;
  L->row_weight = base + B.row_weight;
  L->gate_up = D.recompute_gu ? MOK_NOT_KEPT : base + B.gate_up;
  L->nv_weight_scales = D.nv ? 16 : MOK_NOT_KEPT;  // inside the status block
  L->x_perm = keep_rows ? ring0 : MOK_NOT_KEPT;
  L->rows_max = static_cast<size_t>(D.rows_max);
  L->mb_count = static_cast<size_t>(D.nmb);
  L->mb_stride = B.total;
  L->ring_slots = static_cast<size_t>(D.ring);
  L->ring_slot_bytes = slot_al;
  L->total = ring0 + slot_al * D.ring;
  // block-scaled weights in the backward's orientations, written by the
  // forward from the same reads as its own codes: W_gate_up along 2I (the
  // gate/up dgrad's operand: codes, then tiled scales) and, for MXFP8,
  // W_down along d (the down dgrad's bf16 operand on MX values)
  auto al = [](size_t v) { return (v + 255) & ~static_cast<size_t>(255); };
  const size_t n = static_cast<size_t>(D.E) * 2 * D.I * D.d;
  L->w_gate_up_t = MOK_NOT_KEPT;
  L->w_down_col = MOK_NOT_KEPT;
  if (D.nv || D.mx) {
    L->w_gate_up_t = L->total;
    L->total += al(D.nv ? n / 2 + n / 16 : n + n / 32);
  }
  if (D.mx) {
    L->w_down_col = L->total;
    L->total += al(static_cast<size_t>(D.E) * D.d * D.I * 2);
  }
}

void fwd_layout(const Dims& D, FwdWs* W) {
  Bump b;
  const size_t rows = static_cast<size_t>(D.rows_max);
  W->front_sync = b.take(256);  // directly before the block counts (one memset)
  W->block_counts = b.take(static_cast<size_t>(D.nb) * D.E * 4);
  W->block_base = b.take(static_cast<size_t>(D.nb) * D.E * 4);
  W->h = D.mx ? 0 : b.take(rows * D.I * 2);  // bf16 h (MXFP8: codes below)
  W->x_perm = (D.recompute_dispatch && !D.nv) ? b.take(rows * D.d * 2) : 0;
  W->o = b.take(rows * D.d * 4);  // fp32 expert outputs
  W->logits = b.take(static_cast<size_t>(D.T) * D.E * 4 * router_k_splits(D));
  const size_t wgu = static_cast<size_t>(D.E) * 2 * D.I * D.d;  // elements
  const size_t wd = static_cast<size_t>(D.E) * D.d * D.I;
  auto mx = [&](size_t elems, size_t* codes, size_t* scales) {
    *codes = D.mx ? b.take(elems) : 0;
    *scales = D.mx ? b.take(elems / 32) : 0;
  };
  mx(rows * D.d, &W->xq_codes, &W->xq_scales);
  mx(rows * D.I, &W->h_codes, &W->h_scales);
  mx(wgu, &W->wgu_codes, &W->wgu_scales);
  mx(wd, &W->wd_codes, &W->wd_scales);
  auto nv = [&](size_t elems, size_t* codes, size_t* scales) {
    *codes = D.nv ? b.take(elems / 2) : 0;
    *scales = D.nv ? b.take(elems / 16) : 0;
  };
  nv(rows * D.d, &W->nxq_codes, &W->nxq_scales);
  nv(rows * D.I, &W->nh_codes, &W->nh_scales);
  nv(wgu, &W->nwgu_codes, &W->nwgu_scales);
  nv(wd, &W->nwd_codes, &W->nwd_scales);
  W->nv_g = D.nv ? b.take(256) : 0;
  W->total = b.o;
}

// With micro-batches the weight-gradient GEMMs run once after the loop over
// every micro-batch's rows, so their operands keep one slot per micro-batch
// (ns slots): dG/dU and p*h hi/lo, and the dY and x operands along the rows.
void bwd_layout(const Dims& D, BwdWs* W) {
  Bump b;
  const size_t rows = static_cast<size_t>(D.rows_max);
  const size_t ns = D.nmb > 1 ? static_cast<size_t>(D.nmb) : 1;
  W->dy_perm = b.take(rows * D.d * 2 * (D.mx ? 1 : ns));
  W->dgu_hi = b.take(ns * rows * 2 * D.I * 2);
  W->dgu_lo = b.take(ns * rows * 2 * D.I * 2);
  W->p_hi = b.take(ns * rows * D.I * 2);
  W->p_lo = b.take(ns * rows * D.I * 2);
  W->dp_part = b.take(rows * D.np * 4);
  W->dx_perm = b.take(rows * D.d * 4);  // fp32
  // router-weight gradient: dense dl as a bf16 hi/lo pair [T, E padded to
  // 128], its K-chunk offsets, and the chunks' fp32 partial products
  const size_t epad = static_cast<size_t>(router_e_pad(D));
  const RwSplit rw = router_wgrad_split(D);
  W->dl_hi = b.take(static_cast<size_t>(D.T) * epad * 2);
  W->dl_lo = b.take(static_cast<size_t>(D.T) * epad * 2);
  W->rw_off = b.take(static_cast<size_t>(rw.ks + 1) * 4);
  W->rw_part = b.take(static_cast<size_t>(rw.ks) * epad * D.d * 4);
  const size_t wgu = static_cast<size_t>(D.E) * 2 * D.I * D.d * 2;
  W->dyq_row = D.mx ? b.take(rows * D.d * 2) : 0;  // MXFP8 copies
  W->dyq_col = D.mx ? b.take(ns * rows * D.d * 2) : 0;
  W->xq_col = D.mx ? b.take(ns * rows * D.d * 2) : 0;
  // BF16 with micro-batches: each micro-batch's dispatched x rows
  W->x_def = (!D.mx && ns > 1) ? b.take(ns * rows * D.d * 2) : 0;
  // without micro-batches and with the dispatch recompute: x rows again
  W->x_rd = (D.recompute_dispatch && ns == 1) ? b.take(rows * D.d * 2) : 0;
  // block-scaled dG, dU (the gate/up dgrad's A operand; its B, W_gate_up
  // along 2I, is in saved): codes with tiled scales -- MXFP8 one byte and a
  // scale per 32 values, NVFP4 half a byte and a scale per 16
  const size_t dgu_n = rows * 2 * D.I;
  W->dgu_codes = D.mx ? b.take(dgu_n) : D.nv ? b.take(dgu_n / 2) : 0;
  W->dgu_scales = D.mx ? b.take(dgu_n / 32) : D.nv ? b.take(dgu_n / 16) : 0;
  W->nv_g = D.nv ? b.take(256) : 0;  // NVFP4: dG/dU's tensor scale
  // recompute of g, u: their fp32 rows, and the forward's MXFP8 operands
  W->gu = D.recompute_gu ? b.take(rows * 2 * D.I * 4) : 0;
  const bool rmx = D.recompute_gu && D.mx;  // MXFP8 operands of the recomputed gate/up GEMM
  W->xq_codes = rmx ? b.take(rows * D.d) : 0;
  W->xq_scales = rmx ? b.take(rows * D.d / 32) : 0;
  W->wgu_codes = rmx ? b.take(wgu / 2) : 0;
  W->wgu_scales = rmx ? b.take(wgu / 64) : 0;
  W->total = b.o;
}

void stage_layout(const Dims& D, StageWs* W) {
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += al(bytes);
    return at;
  };
  const size_t rows = static_cast<size_t>(D.rows_max);
  W->status = take(256);
  W->block_counts = take(static_cast<size_t>(D.nb) * D.E * 4);
  W->block_base = take(static_cast<size_t>(D.nb) * D.E * 4);
  W->padded_offsets = take((D.E + 1) * 4);
  W->mtile_prefix = take((D.E + 1) * 8);
  W->ppos = take(static_cast<size_t>(D.T) * D.k * 4);
  W->ptok = take(rows * 4);
  W->row_w = 0;
  W->logits = take(static_cast<size_t>(D.T) * D.E * 4 * router_k_splits(D));
  W->total = o;
}

}  // namespace mok

using namespace mok;

#define MOK_CUDA(call)                          \
  do {                                          \
    if ((call) != cudaSuccess) return MOK_ERR_CUDA; \
  } while (0)

static inline bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

template <typename T>
static inline T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}
template <typename T>
static inline const T* at(const void* base, size_t off) {
  return reinterpret_cast<const T*>(static_cast<const char*>(base) + off);
}

extern "C" {

mok_status mok_moe_workspace_size(const mok_moe_desc* desc, size_t* fwd_ws_bytes,
                                  size_t* saved_bytes, size_t* bwd_ws_bytes) {
  Dims D;
  mok_status s = make_dims(desc, &D);
  if (s != MOK_OK) return s;
  mok_saved_layout L;
  saved_layout(D, &L, nullptr);
  FwdWs F;
  fwd_layout(D, &F);
  BwdWs B;
  bwd_layout(D, &B);
  if (fwd_ws_bytes) *fwd_ws_bytes = F.total;
  if (saved_bytes) *saved_bytes = L.total;
  if (bwd_ws_bytes) *bwd_ws_bytes = B.total;
  return MOK_OK;
}

mok_status mok_moe_saved_layout(const mok_moe_desc* desc, mok_saved_layout* out) {
  if (!out) return MOK_ERR_INVALID_ARG;
  Dims D;
  mok_status s = make_dims(desc, &D);
  if (s != MOK_OK) return s;
  saved_layout(D, out, nullptr);
  return MOK_OK;
}

mok_status mok_moe_forward(const mok_moe_desc* desc, const void* x, const void* w_router,
                           const float* router_bias, const void* w_gate_up, const void* w_down,
                           void* y, void* saved, size_t saved_bytes, void* workspace,
                           size_t ws_bytes, void* stream) {
  NvtxRange nvtx("mok_moe_forward");
  Dims D;
  mok_status s = make_dims(desc, &D);
  if (s != MOK_OK) return s;
  const bool empty = D.T == 0;  // no token rows: x and y may be NULL
  if ((!x && !empty) || !w_router || !w_gate_up || !w_down || (!y && !empty) || !saved ||
      !workspace)
    return MOK_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(w_gate_up) || !aligned16(w_down) ||
      !aligned16(y) || !aligned16(saved) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(router_bias) & 3u))
    return MOK_ERR_INVALID_ARG;
  mok_saved_layout L;
  size_t mt_off;
  saved_layout(D, &L, &mt_off);
  FwdWs F;
  fwd_layout(D, &F);
  if (saved_bytes < L.total || ws_bytes < F.total) return MOK_ERR_WORKSPACE;
  s = mok_check_device();
  if (s != MOK_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  reset_launch_count();

  int* status = at<int>(saved, L.status);
  MOK_CUDA(cudaMemsetAsync(status, 0, sizeof(int), st));
  // MXFP8: E4M3 codes and E8M0 scales (blocks of 32 along K) of the weights,
  // once per call: W_gate_up along d, W_down along I
  uint8_t* wgu_c = at<uint8_t>(workspace, F.wgu_codes);
  uint8_t* wgu_s = at<uint8_t>(workspace, F.wgu_scales);
  uint8_t* wd_c = at<uint8_t>(workspace, F.wd_codes);
  uint8_t* wd_s = at<uint8_t>(workspace, F.wd_scales);
  uint8_t* xq_c = at<uint8_t>(workspace, F.xq_codes);
  uint8_t* xq_s = at<uint8_t>(workspace, F.xq_scales);
  uint8_t* h_c = at<uint8_t>(workspace, F.h_codes);
  uint8_t* h_s = at<uint8_t>(workspace, F.h_scales);
  if (D.mx) {
    // each weight read once for both orientations: the backward's forms go
    // to saved (W_gate_up along 2I as codes, W_down along d as bf16 values)
    uint8_t* wt = at<uint8_t>(saved, L.w_gate_up_t);
    MOK_CUDA(launch_mx_quant_2d(w_gate_up, D.E, 2 * D.I, D.d, wgu_c, wgu_s, wt,
                                wt + D.E * 2 * D.I * D.d, nullptr, st));
    MOK_CUDA(launch_mx_quant_2d(w_down, D.E, D.d, D.I, wd_c, wd_s, nullptr, nullptr,
                                at<char>(saved, L.w_down_col), st));
  }
  // NVFP4: tensor scales [x, h] in the workspace; the weights', once per
  // call, in `saved` [W_gate_up, W_down] (the backward reuses W_gate_up's)
  float* nvg = D.nv ? at<float>(workspace, F.nv_g) : nullptr;
  float* nvw = D.nv ? at<float>(saved, L.nv_weight_scales) : nullptr;
  uint8_t* nxq_c = at<uint8_t>(workspace, F.nxq_codes);
  uint8_t* nxq_s = at<uint8_t>(workspace, F.nxq_scales);
  uint8_t* nh_c = at<uint8_t>(workspace, F.nh_codes);
  uint8_t* nh_s = at<uint8_t>(workspace, F.nh_scales);
  uint8_t* nwgu_c = at<uint8_t>(workspace, F.nwgu_codes);
  uint8_t* nwgu_s = at<uint8_t>(workspace, F.nwgu_scales);
  uint8_t* nwd_c = at<uint8_t>(workspace, F.nwd_codes);
  uint8_t* nwd_s = at<uint8_t>(workspace, F.nwd_scales);
  if (D.nv) {
    MOK_CUDA(launch_nv_tensor_scale(w_gate_up, D.E * 2 * D.I * D.d, nvw + 0, st));
    // W_gate_up in both orientations: along d for this GEMM, along 2I (into
    // saved) for the backward's gate/up dgrad
    uint8_t* wt = at<uint8_t>(saved, L.w_gate_up_t);
    MOK_CUDA(launch_nv_quant_2d(w_gate_up, D.E, 2 * D.I, D.d, nvw + 0, nwgu_c, nwgu_s, wt,
                                wt + D.E * 2 * D.I * D.d / 2, st));
    MOK_CUDA(launch_nv_tensor_scale(w_down, D.E * D.d * D.I, nvw + 1, st));
    MOK_CUDA(launch_nv_quant_tiled(w_down, D.E * D.d, D.I, nvw + 1, nwd_c, nwd_s, nullptr, 0,
                                   st));
  }
  const size_t y_esz = D.act_bf16 ? 2 : 4;
  float* logits = at<float>(workspace, F.logits);
  void* h = D.mx ? nullptr : at<char>(workspace, F.h);
  void* O = at<char>(workspace, F.o);
  for (int i = 0; i < D.nmb; ++i) {
    // micro-batch i: tokens [i*T, (i+1)*T), dispatched into ring slot i % ring
    const char* xi = static_cast<const char*>(x) + static_cast<size_t>(i) * D.T * D.d * 2;
    char* yi = static_cast<char*>(y) + static_cast<size_t>(i) * D.T * D.d * y_esz;
    const size_t blk = static_cast<size_t>(i) * L.mb_stride;
    int32_t* topk_idx = at<int32_t>(saved, L.topk_idx + blk);
    float* topk_w = at<float>(saved, L.topk_w + blk);
    MOK_CUDA(launch_router_logits(D, xi, w_router, logits, status, st));
    PlanOut o;
    o.counts = at<int32_t>(saved, L.counts + blk);
    o.offsets = at<int32_t>(saved, L.offsets + blk);
    o.pos = at<int32_t>(saved, L.pos + blk);
    o.token_of_row = at<int32_t>(saved, L.token_of_row + blk);
    o.padded_offsets = at<int32_t>(saved, L.padded_offsets + blk);
    o.mtile_prefix = at<int32_t>(saved, mt_off + blk);
    o.ppos = at<int32_t>(saved, L.padded_pos + blk);
    o.ptok = at<int32_t>(saved, L.padded_token + blk);
    o.row_w = at<float>(saved, L.row_weight + blk);
    D.coff = o.offsets;  // this micro-batch's grouped GEMMs skip its unread rows
    // top-k selection, histogram, scans and stable placement: one persistent
    // kernel walking the front-end schedule table
    MOK_CUDA(launch_route_plan(D, logits, router_bias, topk_idx, topk_w,
                               at<int32_t>(workspace, F.block_counts),
                               at<int32_t>(workspace, F.block_base),
                               at<unsigned>(workspace, F.front_sync), o, status, st));
    void* x_perm = D.mx                   ? nullptr
                   : D.recompute_dispatch ? at<char>(workspace, F.x_perm)
                                          : at<char>(saved, L.x_perm + (i % D.ring) *
                                                                L.ring_slot_bytes);
    void* gu = D.recompute_gu ? nullptr : at<char>(saved, L.gate_up + blk);
    if (!D.mx && !D.nv)
      MOK_CUDA(launch_dispatch_rows(D, xi, o.ppos, o.ptok, o.padded_offsets, x_perm, status, st));
    if (D.nv) {
      // expert GEMMs on the block-scaled FP4 tensor cores: the x rows go to
      // NVFP4 straight from the token rows; h is written in bf16, then gets
      // its tensor scale (over the plan's rows) and its codes
      MOK_CUDA(launch_nv_tensor_scale(xi, D.T * D.d, nvg + 0, st));
      MOK_CUDA(launch_nv_quant_tiled(xi, D.rows_max, D.d, nvg + 0, nxq_c, nxq_s, o.ptok,
                                     static_cast<int>(D.T), st, o.padded_offsets + D.E));
      MOK_CUDA(gemm_fwd_gate_up_nv(D, nxq_c, nxq_s, nvg + 0, nwgu_c, nwgu_s, nvw + 0,
                                   o.mtile_prefix, o.padded_offsets, gu, h, status, st));
      // (over the routed rows: the padding rows nothing reads hold no h)
      MOK_CUDA(launch_nv_tensor_scale(h, D.rows_max * D.I, nvg + 1, st,
                                      o.padded_offsets + D.E, D.I, o.ptok));
      MOK_CUDA(launch_nv_quant_tiled(h, D.rows_max, D.I, nvg + 1, nh_c, nh_s, nullptr, 0, st,
                                     o.padded_offsets + D.E));
      MOK_CUDA(gemm_fwd_down_nv(D, nh_c, nh_s, nvg + 1, nwd_c, nwd_s, nvw + 1, o.mtile_prefix,
                                o.padded_offsets, O, status, st));
    } else if (D.mx) {
      // expert GEMMs on the block-scaled tensor cores: the dispatched x rows
      // go to MXFP8 straight from the token rows (no bf16 copy), the gate/up
      // GEMM writes h as MXFP8 for the down projection
      MOK_CUDA(launch_mx_rows(xi, nullptr, D.rows_max, D.d, xq_c, xq_s, st, true, o.ptok,
                              static_cast<int>(D.T), o.padded_offsets + D.E));
      MOK_CUDA(gemm_fwd_gate_up_mx(D, xq_c, xq_s, wgu_c, wgu_s, o.mtile_prefix, o.padded_offsets,
                                   gu, h_c, h_s, status, st));
      MOK_CUDA(gemm_fwd_down_mx(D, h_c, h_s, wd_c, wd_s, o.mtile_prefix, o.padded_offsets, O,
                                status, st));
    } else {
      MOK_CUDA(gemm_fwd_gate_up(D, x_perm, w_gate_up, o.mtile_prefix, o.padded_offsets, gu, h,
                                status, st));
      MOK_CUDA(gemm_fwd_down(D, h, w_down, o.mtile_prefix, o.padded_offsets, O, status, st));
    }
    MOK_CUDA(launch_combine(D, static_cast<const float*>(O), o.ppos, topk_w, yi, st));
  }
  return MOK_OK;
}

mok_status mok_moe_backward(const mok_moe_desc* desc, const void* dy, const void* x,
                            const void* w_router, const float* router_bias,
                            const void* w_gate_up, const void* w_down, const void* saved,
                            size_t saved_bytes, void* dx, void* dw_router, void* dw_gate_up,
                            void* dw_down, void* workspace, size_t ws_bytes, void* stream) {
  NvtxRange nvtx("mok_moe_backward");
  (void)router_bias;
  Dims D;
  mok_status s = make_dims(desc, &D);
  if (s != MOK_OK) return s;
  const bool empty = D.T == 0;  // no token rows: dy, x and dx may be NULL
  // x is read by every backward with tokens (the router-weight gradient, and
  // the row dispatch or MXFP8 quantisers of the weight gradients)
  if ((!dy && !empty) || (!x && !empty) || !w_router || !w_gate_up ||
      !w_down || !saved || (!dx && !empty) || !dw_router || !dw_gate_up || !dw_down ||
      !workspace)
    return MOK_ERR_INVALID_ARG;
  if (!aligned16(dy) || !aligned16(x) || !aligned16(w_router) || !aligned16(w_gate_up) ||
      !aligned16(w_down) || !aligned16(saved) || !aligned16(dx) || !aligned16(dw_router) ||
      !aligned16(dw_gate_up) || !aligned16(dw_down) || !aligned16(workspace))
    return MOK_ERR_INVALID_ARG;
  mok_saved_layout L;
  size_t mt_off;
  saved_layout(D, &L, &mt_off);
  BwdWs B;
  bwd_layout(D, &B);
  if (saved_bytes < L.total || ws_bytes < B.total) return MOK_ERR_WORKSPACE;
  s = mok_check_device();
  if (s != MOK_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  // the status word lives in `saved`; the backward reports into it as well
  int* status = const_cast<int*>(at<int>(saved, L.status));
  void* dy_perm = at<char>(workspace, B.dy_perm);
  void* dgu_hi = at<char>(workspace, B.dgu_hi);
  void* dgu_lo = at<char>(workspace, B.dgu_lo);
  void* p_hi = at<char>(workspace, B.p_hi);
  void* p_lo = at<char>(workspace, B.p_lo);
  float* dp_part = at<float>(workspace, B.dp_part);
  float* dx_perm = at<float>(workspace, B.dx_perm);
  void* dl_hi = at<char>(workspace, B.dl_hi);
  void* dl_lo = at<char>(workspace, B.dl_lo);
  int32_t* rw_off = at<int32_t>(workspace, B.rw_off);
  float* rw_part = at<float>(workspace, B.rw_part);
  const bool bs = D.mx || D.nv;  // block-scaled gate/up dgrad
  uint8_t* dgu_c = bs ? at<uint8_t>(workspace, B.dgu_codes) : nullptr;
  uint8_t* dgu_s = bs ? at<uint8_t>(workspace, B.dgu_scales) : nullptr;
  // (NVFP4: the forward left W_gate_up along 2I in saved)
  // (the forward left W_gate_up along 2I in saved: codes, then scales)
  const uint8_t* wgu_t_c = bs ? at<uint8_t>(saved, L.w_gate_up_t) : nullptr;
  const uint8_t* wgu_t_s = D.mx   ? wgu_t_c + D.E * 2 * D.I * D.d
                           : D.nv ? wgu_t_c + D.E * 2 * D.I * D.d / 2
                                  : nullptr;
  // NVFP4: dG/dU's tensor scale (per micro-batch) and W_gate_up's (the forward's)
  float* nv_dgu_g = D.nv ? at<float>(workspace, B.nv_g) : nullptr;
  const float* nv_wgu_g = D.nv ? at<float>(saved, L.nv_weight_scales) : nullptr;
  const void* wd_op = w_down;
  // MXFP8 operands of the recomputed gate/up GEMM (the forward's kernel)
  uint8_t* rwgu_c = at<uint8_t>(workspace, B.wgu_codes);
  uint8_t* rwgu_s = at<uint8_t>(workspace, B.wgu_scales);
  uint8_t* rxq_c = at<uint8_t>(workspace, B.xq_codes);
  uint8_t* rxq_s = at<uint8_t>(workspace, B.xq_scales);
  if (D.mx && D.recompute_gu)
    MOK_CUDA(launch_mx_rows(w_gate_up, nullptr, D.E * 2 * D.I, D.d, rwgu_c, rwgu_s, st, true));
  // MXFP8: W_down along d (bf16 values, blocks of 32 rows), from the forward
  if (D.mx) wd_op = at<char>(saved, L.w_down_col);
  const size_t dx_esz = D.act_bf16 ? 2 : 4;
  // micro-batches in reverse, so the last ring slots are still resident.
  // With several micro-batches the expert weight gradients are deferred: each
  // micro-batch leaves its operands in its own slot and one launch per weight
  // runs K through every micro-batch's rows after the loop (dW written once);
  // the router gradient still accumulates micro-batch by micro-batch.
  const bool defer = D.nmb > 1;
  const size_t rows = static_cast<size_t>(D.rows_max);
  auto slot = [&](void* base, int i, size_t bytes) {
    return static_cast<void*>(static_cast<char*>(base) + (defer ? static_cast<size_t>(i) : 0) *
                                                             bytes);
  };
  for (int i = D.nmb - 1; i >= 0; --i) {
    const bool first = (i == D.nmb - 1) && !D.accumulate;
    const size_t blk = static_cast<size_t>(i) * L.mb_stride;
    void* dgu_hi_i = slot(dgu_hi, i, rows * 2 * D.I * 2);
    void* dgu_lo_i = slot(dgu_lo, i, rows * 2 * D.I * 2);
    void* p_hi_i = slot(p_hi, i, rows * D.I * 2);
    void* p_lo_i = slot(p_lo, i, rows * D.I * 2);
    void* dy_perm_i = D.mx ? dy_perm : slot(dy_perm, i, rows * D.d * 2);
    const char* dyi = static_cast<const char*>(dy) + static_cast<size_t>(i) * D.T * D.d * 2;
    const char* xi = static_cast<const char*>(x) + static_cast<size_t>(i) * D.T * D.d * 2;
    char* dxi = static_cast<char*>(dx) + static_cast<size_t>(i) * D.T * D.d * dx_esz;
    const int32_t* topk_idx = at<int32_t>(saved, L.topk_idx + blk);
    const float* topk_w = at<float>(saved, L.topk_w + blk);
    const int32_t* poff = at<int32_t>(saved, L.padded_offsets + blk);
    const int32_t* mtp = at<int32_t>(saved, mt_off + blk);
    const int32_t* ppos = at<int32_t>(saved, L.padded_pos + blk);
    const int32_t* ptok = at<int32_t>(saved, L.padded_token + blk);
    const float* row_w = at<float>(saved, L.row_weight + blk);
    D.coff = at<int32_t>(saved, L.offsets + blk);  // grouped GEMMs: unread rows skipped
    const void* gu = D.recompute_gu ? at<char>(workspace, B.gu) : at<char>(saved, L.gate_up + blk);
    void* x_perm = (D.mx || D.recompute_dispatch)
                       ? nullptr
                       : const_cast<char*>(at<char>(saved, L.x_perm + (i % D.ring) *
                                                                 L.ring_slot_bytes));
    if (defer && !D.mx) {
      // this micro-batch's rows go to its own slot (the deferred wgrad reads them)
      x_perm = at<char>(workspace, B.x_def) + static_cast<size_t>(i) * rows * D.d * 2;
      MOK_CUDA(launch_dispatch_rows(D, xi, ppos, ptok, poff, x_perm, status, st));
    } else if (D.recompute_dispatch) {
      // saved keeps no dispatched rows: gather x into expert order again
      x_perm = at<char>(workspace, B.x_rd);
      MOK_CUDA(launch_dispatch_rows(D, xi, ppos, ptok, poff, x_perm, status, st));
    } else if (i < D.nmb - D.ring && !D.mx) {
      // the slot now holds a later micro-batch: dispatch this one again
      // (MXFP8 reads the token rows through the row -> token map instead)
      MOK_CUDA(launch_dispatch_rows(D, xi, ppos, ptok, poff, x_perm, status, st));
    }
    if (D.recompute_gu) {
      // the forward's gate/up GEMM again, g and u only (no h)
      if (D.mx) {
        MOK_CUDA(launch_mx_rows(xi, nullptr, D.rows_max, D.d, rxq_c, rxq_s, st, true, ptok,
                                static_cast<int>(D.T), poff + D.E));
        MOK_CUDA(gemm_fwd_gate_up_mx(D, rxq_c, rxq_s, rwgu_c, rwgu_s, mtp, poff,
                                     const_cast<void*>(gu), nullptr, nullptr, status, st));
      } else {
        MOK_CUDA(gemm_fwd_gate_up(D, x_perm, w_gate_up, mtp, poff, const_cast<void*>(gu),
                                  nullptr, status, st));
      }
    }
    // reverse-combine: dy rows into expert order (MXFP8: the quantisers below
    // read them through the row -> token map instead)
    if (!D.mx) MOK_CUDA(launch_dispatch_rows(D, dyi, ppos, ptok, poff, dy_perm_i, status, st));
    const void* dy_row_op = dy_perm_i;
    const void* dy_col_op = dy_perm_i;
    const void* x_col_op = x_perm;
    if (D.mx) {
      void* q1 = at<char>(workspace, B.dyq_row);
      void* q2 = slot(at<char>(workspace, B.dyq_col), i, rows * D.d * 2);
      void* q3 = slot(at<char>(workspace, B.xq_col), i, rows * D.d * 2);
      // dy in both block directions from one read of its token rows; rows
      // past the plan's padded total are read by no GEMM and left unwritten
      MOK_CUDA(launch_mx_cols(dyi, q2, D.rows_max, D.d, nullptr, nullptr, st, q1, ptok,
                              static_cast<int>(D.T), poff + D.E));
      MOK_CUDA(launch_mx_cols(xi, q3, D.rows_max, D.d, nullptr, nullptr, st, nullptr, ptok,
                              static_cast<int>(D.T), poff + D.E));
      dy_row_op = q1;
      dy_col_op = q2;
      x_col_op = q3;
    }
    // down-projection dgrad + SwiGLU backward + router-weight partials;
    // dG, dU and P = p h leave as bf16 hi/lo pairs (and dG, dU as MXFP8)
    MOK_CUDA(gemm_bwd_down_dgrad(D, dy_row_op, wd_op, mtp, poff, static_cast<const float*>(gu),
                                 row_w, dgu_hi_i, dgu_lo_i, p_hi_i, p_lo_i,
                                 D.mx ? dgu_c : nullptr, D.mx ? dgu_s : nullptr, dp_part, status,
                                 st));
    // the weight gradients' K loops stop at each expert's real rows
    WgradSegs one;
    one.coff = at<int32_t>(saved, L.offsets + blk);
    // down-projection wgrad: dW_down_e (+)= dY_e^T (P_hi + P_lo)_e
    if (!defer)
      MOK_CUDA(gemm_wgrad_down(D, dy_col_op, p_hi_i, p_lo_i, poff, dw_down, !first, status, st,
                               one));
    // gate/up dgrad: dX_perm = dGU W_gu (fp32 rows)
    if (D.mx) {
      MOK_CUDA(gemm_bwd_gate_up_dgrad_mx(D, dgu_c, dgu_s, wgu_t_c, wgu_t_s, mtp, poff, dx_perm,
                                         status, st));
    } else if (D.nv) {
      // dG/dU (bf16, the hi half) to NVFP4 along 2I: the tensor scale over
      // the routed rows (padding rows, whose values nothing reads, skipped)
      MOK_CUDA(launch_nv_tensor_scale(dgu_hi_i, D.rows_max * 2 * D.I, nv_dgu_g, st, poff + D.E,
                                      2 * D.I, ptok));
      MOK_CUDA(launch_nv_quant_tiled(dgu_hi_i, D.rows_max, 2 * D.I, nv_dgu_g, dgu_c, dgu_s,
                                     nullptr, 0, st, poff + D.E));
      MOK_CUDA(gemm_bwd_gate_up_dgrad_nv(D, dgu_c, dgu_s, nv_dgu_g, wgu_t_c, wgu_t_s, nv_wgu_g,
                                         mtp, poff, dx_perm, status, st));
    } else
      MOK_CUDA(gemm_bwd_gate_up_dgrad(D, dgu_hi_i, w_gate_up, mtp, poff, dx_perm, status, st));
    // gate/up wgrad: dW_gu_e (+)= (dGU_hi + dGU_lo)_e^T X_e
    if (!defer)
      MOK_CUDA(gemm_wgrad_gate_up(D, dgu_hi_i, dgu_lo_i, x_col_op, poff, dw_gate_up, !first,
                                  status, st, one));
    // reverse-dispatch + router backward
    MOK_CUDA(launch_reverse_dispatch(D, dx_perm, ppos, topk_idx, topk_w, dp_part, w_router, dxi,
                                     dl_hi, dl_lo, rw_off, st));
    MOK_CUDA(gemm_router_wgrad(D, xi, dl_hi, dl_lo, rw_off, rw_part, status, st));
    MOK_CUDA(launch_router_wgrad_reduce(D, rw_part, dw_router, !first, st));
  }
  if (defer) {
    // the expert weight gradients over all micro-batches: K runs through
    // micro-batch 0, 1, ... rows of each expert (offsets one block apart)
    WgradSegs sg;
    sg.nseg = D.nmb;
    sg.poff_stride = static_cast<int>(L.mb_stride / 4);
    sg.coff = at<int32_t>(saved, L.offsets);
    const int32_t* poff0 = at<int32_t>(saved, L.padded_offsets);
    const void* dy_col = D.mx ? at<char>(workspace, B.dyq_col) : dy_perm;
    const void* x_col = D.mx ? at<char>(workspace, B.xq_col) : at<char>(workspace, B.x_def);
    MOK_CUDA(gemm_wgrad_down(D, dy_col, p_hi, p_lo, poff0, dw_down, D.accumulate, status, st,
                             sg));
    MOK_CUDA(gemm_wgrad_gate_up(D, dgu_hi, dgu_lo, x_col, poff0, dw_gate_up, D.accumulate, status,
                                st, sg));
  }
  return MOK_OK;
}

mok_status mok_moe_stage_workspace_size(const mok_moe_desc* desc, size_t* bytes) {
  if (!bytes) return MOK_ERR_INVALID_ARG;
  Dims D;
  mok_status s = make_dims(desc, &D);
  if (s != MOK_OK) return s;
  StageWs W;
  stage_layout(D, &W);
  *bytes = W.total;
  return MOK_OK;
}

mok_status mok_moe_route(const mok_moe_desc* desc, const void* x, const void* w_router,
                         const float* router_bias, int32_t* topk_idx, float* topk_w,
                         void* workspace, size_t ws_bytes, void* stream) {
  Dims D;
  mok_status s = make_dims(desc, &D);
  if (s != MOK_OK) return s;
  if (D.nmb != 1) return MOK_ERR_UNSUPPORTED;
  if (((!x || !topk_idx || !topk_w) && D.T > 0) || !w_router || !workspace)
    return MOK_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(workspace)) return MOK_ERR_INVALID_ARG;
  StageWs W;
  stage_layout(D, &W);
  if (ws_bytes < W.total) return MOK_ERR_WORKSPACE;
  s = mok_check_device();
  if (s != MOK_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* status = at<int>(workspace, W.status);
  MOK_CUDA(cudaMemsetAsync(status, 0, sizeof(int), st));
  float* logits = at<float>(workspace, W.logits);
  MOK_CUDA(launch_router_logits(D, x, w_router, logits, status, st));
  MOK_CUDA(launch_router_topk(D, logits, router_bias, topk_idx, topk_w, status, st));
  return MOK_OK;
}

mok_status mok_moe_dispatch_plan(const mok_moe_desc* desc, const int32_t* topk_idx,
                                 int32_t* counts, int32_t* offsets, int32_t* pos,
                                 int32_t* token_of_row, void* workspace, size_t ws_bytes,
                                 void* stream) {
  Dims D;
  mok_status s = make_dims(desc, &D);
  if (s != MOK_OK) return s;
  if (D.nmb != 1) return MOK_ERR_UNSUPPORTED;
  if ((!topk_idx && D.T > 0) || !counts || !offsets || (!pos && D.T > 0) ||
      (!token_of_row && D.T > 0) || !workspace)
    return MOK_ERR_INVALID_ARG;
  if (!aligned16(workspace)) return MOK_ERR_INVALID_ARG;
  StageWs W;
  stage_layout(D, &W);
  if (ws_bytes < W.total) return MOK_ERR_WORKSPACE;
  s = mok_check_device();
  if (s != MOK_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* status = at<int>(workspace, W.status);
  MOK_CUDA(cudaMemsetAsync(status, 0, sizeof(int), st));
  // slots skipped as invalid keep pos = -1; rows they would have taken stay
  // unwritten, so pre-set the inverse map to -1
  if (D.R > 0) MOK_CUDA(cudaMemsetAsync(token_of_row, 0xFF, static_cast<size_t>(D.R) * 4, st));
  PlanOut o;
  o.counts = counts;
  o.offsets = offsets;
  o.pos = pos;
  o.token_of_row = token_of_row;
  o.padded_offsets = at<int32_t>(workspace, W.padded_offsets);
  o.mtile_prefix = at<int32_t>(workspace, W.mtile_prefix);
  o.ppos = at<int32_t>(workspace, W.ppos);
  o.ptok = at<int32_t>(workspace, W.ptok);
  o.row_w = nullptr;
  MOK_CUDA(launch_plan(D, topk_idx, nullptr, at<int32_t>(workspace, W.block_counts),
                       at<int32_t>(workspace, W.block_base), o, status, st));
  return MOK_OK;
}

mok_status mok_gemm_bf16(int64_t M, int64_t N, int64_t K, const void* A, int a_mn_major,
                         const void* B, int b_mn_major, void* C, void* workspace,
                         size_t ws_bytes, void* stream) {
  if (M <= 0 || N <= 0 || K <= 0 || !A || !B || !C || !workspace) return MOK_ERR_INVALID_ARG;
  if (M % 128 || N % 128 || K % 128) return MOK_ERR_UNSUPPORTED;
  if (M > (1 << 24) || N > (1 << 24) || K > (1 << 24)) return MOK_ERR_UNSUPPORTED;
  if (a_mn_major && !b_mn_major) return MOK_ERR_UNSUPPORTED;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C) || !aligned16(workspace))
    return MOK_ERR_INVALID_ARG;
  if (ws_bytes < 256) return MOK_ERR_WORKSPACE;
  mok_status s = mok_check_device();
  if (s != MOK_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* status = static_cast<int*>(workspace);
  MOK_CUDA(cudaMemsetAsync(status, 0, sizeof(int), st));
  MOK_CUDA(gemm_dense_bf16(M, N, K, A, a_mn_major != 0, B, b_mn_major != 0, C, status, st));
  return MOK_OK;
}

mok_status mok_gemm_mxfp8(int64_t M, int64_t N, int64_t K, const uint8_t* A, const uint8_t* sa,
                          const uint8_t* B, const uint8_t* sb, float* C, int cta_pair,
                          void* workspace, size_t ws_bytes, void* stream) {
  if (M <= 0 || N <= 0 || K <= 0 || !A || !sa || !B || !sb || !C || !workspace)
    return MOK_ERR_INVALID_ARG;
  if (M % 128 || N % 128 || K % 128) return MOK_ERR_UNSUPPORTED;
  if (cta_pair && (M % 256 || N % 256)) return MOK_ERR_UNSUPPORTED;
  if (M > (1 << 24) || N > (1 << 24) || K > (1 << 24)) return MOK_ERR_UNSUPPORTED;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(sa) & 3u) || (reinterpret_cast<uintptr_t>(sb) & 3u))
    return MOK_ERR_INVALID_ARG;
  if (ws_bytes < 256) return MOK_ERR_WORKSPACE;
  mok_status s = mok_check_device();
  if (s != MOK_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* status = static_cast<int*>(workspace);
  MOK_CUDA(cudaMemsetAsync(status, 0, sizeof(int), st));
  MOK_CUDA(gemm_dense_mxfp8(M, N, K, A, sa, B, sb, C, cta_pair != 0, status, st));
  return MOK_OK;
}

mok_status mok_selftest_bounded_wait(void* workspace, size_t ws_bytes, void* stream) {
  if (!workspace || !aligned16(workspace)) return MOK_ERR_INVALID_ARG;
  if (ws_bytes < 256) return MOK_ERR_WORKSPACE;
  mok_status s = mok_check_device();
  if (s != MOK_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* status = static_cast<int*>(workspace);
  MOK_CUDA(cudaMemsetAsync(status, 0, sizeof(int), st));
  MOK_CUDA(launch_bounded_wait_selftest(status, st));
  return MOK_OK;
}

mok_status mok_fill_zero(void* dst, size_t bytes, void* stream) {
  if (bytes == 0) return MOK_OK;
  if (!dst || !aligned16(dst) || bytes % 16) return MOK_ERR_INVALID_ARG;
  mok_status s = mok_check_device();
  if (s != MOK_OK) return s;
  MOK_CUDA(launch_fill_zero(dst, bytes, static_cast<cudaStream_t>(stream)));
  return MOK_OK;
}

mok_status mok_get_device_status(const void* buf, void* stream, int32_t* code) {
  if (!buf || !code) return MOK_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOK_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, buf, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return MOK_ERR_CUDA;
  *code = v;
  return MOK_OK;
}

const char* mok_status_string(mok_status status) {
  switch (status) {
    case MOK_OK: return "ok";
    case MOK_ERR_INVALID_ARG: return "invalid argument";
    case MOK_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case MOK_ERR_WORKSPACE: return "buffer smaller than the size query";
    case MOK_ERR_CUDA: return "CUDA runtime error";
    case MOK_ERR_NO_DEVICE: return "current device is not sm_103";
    case MOK_ERR_SCRATCH_LIMIT: return "problem needs more than the fixed device scratch of the no-allocation entry point";
    case MOK_ERR_DEVICE_NONFINITE: return "device: NaN router logit (treated as -inf)";
    case MOK_ERR_DEVICE_INDEX: return "device: expert index out of range or repeated (skipped)";
    case MOK_ERR_DEVICE_TIMEOUT: return "device: bounded wait timed out (results invalid)";
  }
  return "unknown status";
}

int32_t mok_last_launch_count(void) { return launch_count(); }

mok_status mok_profile_enable(int on) {
  g_prof = on != 0;
  return MOK_OK;
}

mok_status mok_profile_reset(void) {
  g_recs.clear();
  g_pool_used = 0;
  return MOK_OK;
}

mok_status mok_profile_collect(mok_kernel_time* out, int32_t max, int32_t* n) {
  if (!n || (max > 0 && !out)) return MOK_ERR_INVALID_ARG;
  std::map<std::string, std::pair<int32_t, double>> agg;
  std::vector<std::string> order;
  for (const ProfRec& r : g_recs) {
    if (cudaEventSynchronize(r.b) != cudaSuccess) return MOK_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) return MOK_ERR_CUDA;
    auto it = agg.find(r.name);
    if (it == agg.end()) {
      order.push_back(r.name);
      agg[r.name] = {1, ms};
    } else {
      it->second.first += 1;
      it->second.second += ms;
    }
  }
  int32_t i = 0;
  for (const std::string& name : order) {
    if (i >= max) break;
    memset(out[i].name, 0, sizeof(out[i].name));
    strncpy(out[i].name, name.c_str(), sizeof(out[i].name) - 1);
    out[i].launches = agg[name].first;
    out[i].total_ms = agg[name].second;
    ++i;
  }
  *n = i;
  return MOK_OK;
}

}  // extern "C"
