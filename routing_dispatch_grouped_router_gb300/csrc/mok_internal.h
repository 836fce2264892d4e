// Host-side internals shared by the translation units of libmok: buffer
// layouts, launch helpers of every kernel, and error plumbing.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/mok.h"

namespace mok {

constexpr int kRowPad = 128;     // expert segments are padded to this many rows
constexpr int kMaxExperts = 512;
constexpr int kMaxTopK = 8;
constexpr int kPlanBlock = 256;  // tokens per block of the dispatch plan

// Sizes derived from a descriptor.  T is the tokens of one micro-batch (the
// whole batch when the descriptor asks for no micro-batching); every kernel
// sees one micro-batch at a time.
struct Dims {
  int64_t T_total;   // tokens of the whole call
  int nmb;           // micro-batches (T_total / T)
  int ring;          // ring slots holding dispatched token rows
  int64_t T, d, E, I;
  int k;
  int64_t R;         // T*k routed rows
  int64_t rows_max;  // bound on padded rows: R + 127*min(E,R), rounded up to 128
  int64_t nb;        // dispatch-plan blocks: ceil(T / kPlanBlock)
  int bn_dgrad;      // N tile of the down-projection dgrad (over I)
  int np;            // dp partials per row = (I / bn_dgrad) * 2
  bool act_bf16;     // y and dx written as bf16 (else fp32)
  bool wgrad_bf16;   // dW_* written as bf16 (else fp32)
  bool mx;           // MXFP8 expert GEMM operands
  bool accumulate;   // backward adds into the weight gradients
  bool recompute_gu; // g, u not kept: the backward recomputes them
  bool nv;           // NVFP4 forward expert GEMMs (backward on the BF16 path)
  bool recompute_dispatch;  // BF16: dispatched x rows not kept in saved;
                            // the backward dispatches them again
  bool pair;         // grouped GEMMs with 256-row tiles on CTA pairs (2-SM MMA)
  // Set by the layer before the M-grouped GEMMs of a micro-batch (NULL
  // otherwise): its plan's [E+1] real row offsets.  Rows of expert e from its
  // real rows rounded up to 64 to its 128-padded end are read by nothing, so
  // those GEMMs skip their epilogue there (whole 32-row quarters).
  const int32_t* coff = nullptr;
};

// Split-K factor of the router logit GEMM: the largest power of two (up to
// 8, dividing d/64) that keeps its tiles within 128 CTAs.  A function of the
// shape only, so the logits are the same on every call.
inline int router_k_splits(const Dims& D) {
  const int64_t bn = D.E > 128 ? 256 : 128;
  const int64_t tiles = ((D.T + 127) / 128) * ((D.E + bn - 1) / bn);
  const int64_t nkb = (D.d + 63) / 64;
  int s = 1;
  while (s < 8 && tiles * s * 2 <= 128 && nkb % (s * 2) == 0) s *= 2;
  return s;
}

// Offsets inside one micro-batch's block of `saved` (relative to the block).
struct BlockL {
  size_t topk_idx, topk_w, counts, offsets, pos, token_of_row, padded_offsets, mtile_prefix,
      padded_pos, padded_token, row_weight, gate_up, total;
};
struct FwdWs {
  size_t front_sync, block_counts, block_base, h, o, logits;
  size_t x_perm;  // dispatched x rows when saved keeps none (recompute_dispatch)
  // NVFP4: codes and tiled scales of the x rows, h, W_gate_up, W_down, and
  // the four fp32 tensor scales (x, h, W_gate_up, W_down)
  size_t nxq_codes, nxq_scales, nh_codes, nh_scales, nwgu_codes, nwgu_scales, nwd_codes,
      nwd_scales, nv_g;
  // MXFP8: E4M3 codes and E8M0 scale bytes of x rows, h, W_gate_up, W_down
  size_t xq_codes, xq_scales, h_codes, h_scales, wgu_codes, wgu_scales, wd_codes, wd_scales;
  size_t total;
};
struct BwdWs {
  size_t dy_perm, dgu_hi, dgu_lo, p_hi, p_lo, dp_part, dx_perm, dl_hi, dl_lo, rw_off, rw_part,
      dyq_row, dyq_col,
      xq_col, dgu_codes, dgu_scales, gu, xq_codes, xq_scales,
      wgu_codes, wgu_scales, x_def, x_rd, nv_g, total;
};
struct StageWs {
  size_t status, block_counts, block_base, padded_offsets, mtile_prefix, ppos, ptok, row_w,
      logits, total;
};

mok_status make_dims(const mok_moe_desc* desc, Dims* out);
void block_layout(const Dims& D, BlockL* B);
void saved_layout(const Dims& D, mok_saved_layout* L, size_t* mtile_prefix_off);
void fwd_layout(const Dims& D, FwdWs* W);
void bwd_layout(const Dims& D, BwdWs* W);
void stage_layout(const Dims& D, StageWs* W);

int num_sms_current_device();
mok_status mok_check_device();  // MOK_OK when the current device is sm_103

// ------------------------------------------------------------------ kernels --

// Router: logits through the GEMM engine, then top-k + softmax per token.
cudaError_t launch_router_logits(const Dims& D, const void* x, const void* w_router, float* logits,
                                 int* status, cudaStream_t st);
cudaError_t launch_router_topk(const Dims& D, const float* logits, const float* bias,
                               int32_t* topk_idx, float* topk_w, int* status, cudaStream_t st);

// Dispatch plan: histogram, scan, stable placement.
struct PlanOut {
  int32_t* counts;          // [E]
  int32_t* offsets;         // [E+1]
  int32_t* pos;             // [T,k] (may be null)
  int32_t* token_of_row;    // [R] (may be null)
  int32_t* padded_offsets;  // [E+1]
  int32_t* mtile_prefix;    // [2(E+1)]: prefix of 128-row tiles, then of tile pairs
  int32_t* ppos;            // [T,k]
  int32_t* ptok;            // [rows_max]
  float* row_w;             // [rows_max] (may be null)
};
cudaError_t launch_plan(const Dims& D, const int32_t* topk_idx, const float* topk_w,
                        int32_t* block_counts, int32_t* block_base, const PlanOut& o, int* status,
                        cudaStream_t st);
// The router's top-k and the dispatch plan in one persistent cooperative
// kernel driven by a schedule table (front.cu); bitwise the same results as
// launch_router_topk followed by launch_plan.  sync: 256 bytes of scratch;
// it and block_counts are zeroed by this call (one memset when block_counts
// starts 256 bytes after sync).
cudaError_t launch_route_plan(const Dims& D, const float* logits, const float* bias,
                              int32_t* topk_idx, float* topk_w, int32_t* block_counts,
                              int32_t* block_base, unsigned* sync, const PlanOut& o, int* status,
                              cudaStream_t st);

// Rows [0, padded_offsets[E]) of dst: dst[ppos[t, s]] = src[t] for every
// token t and slot s, zeros where ptok[r] < 0 (padding).  Each src row is
// read once.
cudaError_t launch_dispatch_rows(const Dims& D, const void* src, const int32_t* ppos,
                                 const int32_t* ptok, const int32_t* padded_offsets, void* dst,
                                 int* status, cudaStream_t st);

// y_t = sum_s p[t,s] O[ppos[t,s]] (O fp32; y fp32 or bf16).
cudaError_t launch_combine(const Dims& D, const float* O, const int32_t* ppos, const float* topk_w,
                           void* y, cudaStream_t st);

// dl (router logit grad) from dp partials; dx_t = sum_s dX[ppos] + dl W_r[e]
// (dX fp32; dx fp32 or bf16).  Also writes dl as the dense operand of the
// router-weight gradient, dl[t, e] for e < router_e_pad(D) (zero where e is
// not among t's experts) as a bf16 hi/lo pair, and that GEMM's K-chunk
// offsets (router_wgrad_split(D).ks + 1 of them, one chunk apart).
cudaError_t launch_reverse_dispatch(const Dims& D, const float* dX_perm, const int32_t* ppos,
                                    const int32_t* topk_idx, const float* topk_w,
                                    const float* dp_part, const void* w_router, void* dx,
                                    void* dl_hi, void* dl_lo, int32_t* rw_off, cudaStream_t st);

// The router-weight gradient dW_r = dl^T x runs as a tensor-core GEMM over
// token chunks: M = the experts padded to 128 (rows of dl^T), N = d, K = the
// tokens, split into ks chunks of kb 64-row blocks; chunk s writes its fp32
// partial product to part + s * router_e_pad(D) * d, and a second kernel adds
// the ks partials in order.  ks targets 152 CTAs (the SM count of a GB300)
// whatever the device, so that the sums do not depend on it.
inline int64_t router_e_pad(const Dims& D) { return (D.E + 127) / 128 * 128; }
inline int router_wgrad_bn(const Dims& D) { return D.d % 256 == 0 ? 256 : 128; }
struct RwSplit {
  int ks;  // K chunks (>= 1)
  int kb;  // 64-token blocks per chunk
};
inline RwSplit router_wgrad_split(const Dims& D) {
  const int64_t bn = router_wgrad_bn(D);
  const int64_t tiles = router_e_pad(D) / 128 * ((D.d + bn - 1) / bn);
  const int64_t nkb = (D.T + 63) / 64 > 0 ? (D.T + 63) / 64 : 1;
  int64_t ks = 152 / tiles;
  if (ks < 1) ks = 1;
  if (ks > nkb) ks = nkb;
  const int64_t kb = (nkb + ks - 1) / ks;
  ks = (nkb + kb - 1) / kb;
  return {static_cast<int>(ks), static_cast<int>(kb)};
}
cudaError_t gemm_router_wgrad(const Dims& D, const void* x, const void* dl_hi, const void* dl_lo,
                              const int32_t* rw_off, float* part, int* status, cudaStream_t st);
// dW_r (+)= sum over s < ks of the partials, in order (fp32 or bf16 out;
// accumulation fp32 only)
cudaError_t launch_router_wgrad_reduce(const Dims& D, const float* part, void* dw_router,
                                       bool accumulate, cudaStream_t st);

// Grouped GEMMs on tcgen05 (see gemm.cu).
cudaError_t gemm_fwd_gate_up(const Dims& D, const void* X_perm, const void* w_gate_up,
                             const int32_t* mtile_prefix, const int32_t* poff, void* GU, void* H,
                             int* status, cudaStream_t st);
cudaError_t gemm_fwd_gate_up_mx(const Dims& D, const uint8_t* x_codes, const uint8_t* x_scales,
                                const uint8_t* wgu_codes, const uint8_t* wgu_scales,
                                const int32_t* mtile_prefix, const int32_t* poff, void* GU,
                                uint8_t* h_codes, uint8_t* h_scales, int* status,
                                cudaStream_t st);
// NVFP4 forward GEMMs on CTA pairs (gemm.cu): packed E2M1 codes [rows, K/2],
// tiled E4M3 scales (launch_nv_quant_tiled), device tensor scales.
cudaError_t gemm_fwd_gate_up_nv(const Dims& D, const uint8_t* x_codes, const uint8_t* x_scales,
                                const float* x_g, const uint8_t* wgu_codes,
                                const uint8_t* wgu_scales, const float* wgu_g,
                                const int32_t* mtile_prefix, const int32_t* poff, void* GU,
                                void* H, int* status, cudaStream_t st);
cudaError_t gemm_fwd_down_nv(const Dims& D, const uint8_t* h_codes, const uint8_t* h_scales,
                             const float* h_g, const uint8_t* wd_codes, const uint8_t* wd_scales,
                             const float* wd_g, const int32_t* mtile_prefix, const int32_t* poff,
                             void* O, int* status, cudaStream_t st);
// the gate/up dgrad dX_perm = [dG dU] W_gate_up on NVFP4 operands: dG/dU
// codes [rows_max, I] (2I values) and W_gate_up transposed [E*d, I] codes
cudaError_t gemm_bwd_gate_up_dgrad_nv(const Dims& D, const uint8_t* dgu_codes,
                                      const uint8_t* dgu_scales, const float* dgu_g,
                                      const uint8_t* wgu_t_codes, const uint8_t* wgu_t_scales,
                                      const float* wgu_g, const int32_t* mtile_prefix,
                                      const int32_t* poff, void* dX_perm, int* status,
                                      cudaStream_t st);
cudaError_t gemm_fwd_down_mx(const Dims& D, const uint8_t* h_codes, const uint8_t* h_scales,
                             const uint8_t* wd_codes, const uint8_t* wd_scales,
                             const int32_t* mtile_prefix, const int32_t* poff, void* O,
                             int* status, cudaStream_t st);
cudaError_t gemm_fwd_down(const Dims& D, const void* H, const void* w_down,
                          const int32_t* mtile_prefix, const int32_t* poff, void* O, int* status,
                          cudaStream_t st);
cudaError_t gemm_bwd_down_dgrad(const Dims& D, const void* dY_perm, const void* w_down,
                                const int32_t* mtile_prefix, const int32_t* poff, const float* GU,
                                const float* row_w, void* dGU_hi, void* dGU_lo, void* P_hi,
                                void* P_lo, uint8_t* dgu_codes, uint8_t* dgu_scales,
                                float* dp_part, int* status, cudaStream_t st);
// MXFP8: dX_perm = dGU W_gate_up per expert on the block-scaled tensor cores,
// dGU as the codes B2 writes, W_gate_up as launch_mx_quant_2d writes it (along 2I).
cudaError_t gemm_bwd_gate_up_dgrad_mx(const Dims& D, const uint8_t* dgu_codes,
                                      const uint8_t* dgu_scales, const uint8_t* wgu_t_codes,
                                      const uint8_t* wgu_t_scales, const int32_t* mtile_prefix,
                                      const int32_t* poff, void* dX_perm, int* status,
                                      cudaStream_t st);
cudaError_t gemm_bwd_gate_up_dgrad(const Dims& D, const void* dGU, const void* w_gate_up,
                                   const int32_t* mtile_prefix, const int32_t* poff,
                                   void* dX_perm, int* status, cudaStream_t st);
// Weight-gradient GEMMs over nseg row spaces (the micro-batches of a call):
// operands are [nseg * rows_max, cols] with row space s at rows s*rows_max;
// row space s has its padded offsets at poff + s*poff_stride.  K runs through
// the row spaces in order.  coff: the real (unpadded) row offsets in the same
// layout, or NULL; given, each expert's K loop stops after its real rows
// (rounded up to 64) instead of running through its zero padding rows.
struct WgradSegs {
  int nseg = 1;
  int poff_stride = 0;  // int32 elements between successive offset arrays
  const int32_t* coff = nullptr;
};
cudaError_t gemm_wgrad_down(const Dims& D, const void* dY_perm, const void* P_hi,
                            const void* P_lo, const int32_t* poff, void* dw_down,
                            bool accumulate, int* status, cudaStream_t st,
                            const WgradSegs& sg = WgradSegs());
cudaError_t gemm_wgrad_gate_up(const Dims& D, const void* dGU_hi, const void* dGU_lo,
                               const void* X_perm, const int32_t* poff, void* dw_gate_up,
                               bool accumulate, int* status, cudaStream_t st,
                               const WgradSegs& sg = WgradSegs());
// 2-D TMA map over a row-major [outer, inner] array (row stride row_elems),
// box {box_inner, box_rows}, zero fill out of bounds.
bool make_tensor_map_2d(CUtensorMap* m, CUtensorMapDataType dt, int esz, const void* base,
                        uint64_t inner, uint64_t outer, uint64_t row_elems, uint32_t box_inner,
                        uint32_t box_rows, CUtensorMapSwizzle swz);
// C[M,N] fp32 = dequant(A)[M,K] dequant(B)[N,K]^T, MXFP8 operands (E4M3 codes,
// one E8M0 scale byte per 32 consecutive K values) on block-scaled tcgen05.
cudaError_t gemm_dense_mxfp8(int64_t M, int64_t N, int64_t K, const uint8_t* A,
                             const uint8_t* A_scales, const uint8_t* B, const uint8_t* B_scales,
                             float* C, bool cta_pair, int* status, cudaStream_t st);
cudaError_t gemm_dense_bf16(int64_t M, int64_t N, int64_t K, const void* A, bool a_mn,
                            const void* B, bool b_mn, void* C, int* status, cudaStream_t st);

// MXFP8 fake quantisation (mx.cu): rows = blocks along each row, cols =
// blocks of 32 rows; codes/scales may be null.
// tiled: scales in the tiled layout of mx_tiled_off (rows, cols multiples of
// 128), the layout of the expert GEMMs' MXFP8 operands; else row-major.
// rowmap != NULL: output row r quantises input row rowmap[r] (zeros where that is
// not in [0, T)), so the dispatched rows need not be materialised.
// rows_dev (or NULL; row-map form only): the device count of leading rows
// that anything reads; later rows are left unwritten.
cudaError_t launch_mx_rows(const void* in, void* out, long long rows, long long cols,
                           uint8_t* codes, uint8_t* scales, cudaStream_t st, bool tiled = false,
                           const int32_t* rowmap = nullptr, int T = 0,
                           const int32_t* rows_dev = nullptr);

// A weight [ng*K, C] in both block directions from one read: rows (blocks of
// 32 along C) as codes [ng*K, C] with tiled scales, and columns (blocks of 32
// along K) as codes [ng*C, K] with tiled scales (ccodes) or as bf16 values in
// the input's layout (cvals; exactly one of the two).  K, C multiples of 128.
cudaError_t launch_mx_quant_2d(const void* in, long long ng, long long K, long long C,
                               uint8_t* rcodes, uint8_t* rscales, uint8_t* ccodes,
                               uint8_t* cscales, void* cvals, cudaStream_t st);
// Column blocks (rows % 32 == 0, cols % 8 == 0); rows_out != NULL also writes
// the row-block dequantised values of the same input (cols % 32 == 0).
// rows_dev (or NULL): as launch_mx_rows' (whole 32-row blocks).
cudaError_t launch_mx_cols(const void* in, void* out, long long rows, long long cols,
                           uint8_t* codes, uint8_t* scales, cudaStream_t st,
                           void* rows_out = nullptr, const int32_t* rowmap = nullptr, int T = 0,
                           const int32_t* rows_dev = nullptr);

// NVFP4 (nvfp4.cu): the tensor scale of n bf16 values into the device *g
// (which the call also uses as scratch), and codes [rows, cols/2] with E4M3
// block scales in the tiled layout (one 512-byte block per 128 rows x 64
// values, consecutive along K) of bf16 [rows, cols] or, with `map`, of the
// rows map[r] of a [T, cols] input (zeros where map[r] is not in [0, T)).
// rows_dev (or NULL): only the first *rows_dev rows of row_elems values count;
// rowmap (or NULL): rows r with rowmap[r] < 0 do not count.
cudaError_t launch_nv_tensor_scale(const void* in, long long n, float* g, cudaStream_t st,
                                   const int32_t* rows_dev = nullptr, long long row_elems = 0,
                                   const int32_t* rowmap = nullptr);
// NVFP4 of ng stacked bf16 [K, C] matrices in both orientations from one
// read: rows (blocks along C: codes [ng*K, C/2], tiled scales) and columns
// (blocks along K: codes [ng*C, K/2], scales tiled or row-major); NULL codes
// skip an orientation.  K and C multiples of 128.
cudaError_t launch_nv_quant_2d(const void* in, long long ng, long long K, long long C,
                               const float* g, uint8_t* rcodes, uint8_t* rscales,
                               uint8_t* ccodes, uint8_t* cscales, cudaStream_t st,
                               bool ctiled = true);
// rows_dev (or NULL): the device count of leading rows that anything reads;
// later rows are left unwritten.
cudaError_t launch_nv_quant_tiled(const void* in, long long rows, long long cols, const float* g,
                                  uint8_t* codes, uint8_t* scales, const int32_t* map, int T,
                                  cudaStream_t st, const int32_t* rows_dev = nullptr);

// One CTA whose mbarrier wait can never complete: exercises the bounded wait.
cudaError_t launch_bounded_wait_selftest(int* status, cudaStream_t st);
// zeroes `bytes` (a multiple of 16) at 16-byte aligned dst with bulk stores
cudaError_t launch_fill_zero(void* dst, size_t bytes, cudaStream_t st);

// launches counter (host side)
void count_launch(int n = 1);
void reset_launch_count();
int32_t launch_count();

// Per-kernel CUDA-event timing (enabled through mok_profile_enable): the
// scope records an event before and after the kernel it encloses.
void prof_begin(const char* name, cudaStream_t st);
void prof_end(cudaStream_t st);
struct ProfScope {
  cudaStream_t st;
  ProfScope(const char* name, cudaStream_t s) : st(s) { prof_begin(name, s); }
  ~ProfScope() { prof_end(st); }
};

}  // namespace mok
