/*
 * mok.h - C ABI of a deterministic Mixture-of-Experts training layer for one
 * GB300 GPU (sm_103a): top-k router, dispatch into expert-contiguous order,
 * grouped SwiGLU expert GEMMs, weighted combine, and the backward mirror
 * (reverse-combine, grouped dgrad/wgrad GEMMs, reverse-dispatch, router grad).
 *
 * Sources (page title, section):
 *   [gtnt]     "MoK揭秘：NVL72上大规模MoE训练工程方案深度解读" (gtnt.cn)
 *   [aikraft]  "Cursor MoK: revolution in MoE model training on NVL72"
 *              (aikraft.ru), sections 01-04
 *   [dothoosh] "Cursor Mixture-of-Kittens cuts MoE training latency by 5.8x"
 *              (dothoosh.com), section "MoK technical details" with bullets
 *              "Hybrid communication", "Overlap granularity",
 *              "Ring buffer logic", "Precision and scheduling"
 *
 * Conventions for every entry point
 *   - Pointers named as device buffers are device pointers on the current CUDA
 *     device; the caller allocates and owns every buffer.  The library never
 *     allocates, frees or copies device->host, and never synchronises the
 *     stream (mok_get_device_status is the one exception).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *     All work is enqueued on it in order.
 *   - bf16 tensors are row-major, contiguous, 16-byte aligned.  Every weight
 *     is stored [out, in] (nn.Linear style), so the reduction dimension is
 *     the contiguous one.
 *   - Arguments are validated before anything is enqueued; on an error
 *     return nothing was enqueued.
 *   - Results are bitwise identical from call to call for the same inputs,
 *     descriptor and device (no floating-point atomics anywhere).
 *
 * Shape requirements (MOK_ERR_UNSUPPORTED otherwise)
 *   1 <= k <= min(E, 8);  1 <= E <= 512;  0 <= T;  T*k < 2^31;
 *   d and I multiples of 32, 128 <= d, I <= 16384 (widths that are not
 *   multiples of the GEMM tiles give ragged tiles: zero-filled loads, unstored
 *   columns); MOK_MXFP8: d and I multiples of 128; MOK_NVFP4: of 256;
 *   micro-batching: T a multiple of mb_tokens, 0 <= ring_slots <= T/mb_tokens,
 *   fp32 weight-gradient outputs (they accumulate over micro-batches).
 */
#ifndef MOK_H_
#define MOK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mok_status {
  MOK_OK = 0,
  MOK_ERR_INVALID_ARG = 1,      /* null pointer, misaligned pointer, bad size */
  MOK_ERR_UNSUPPORTED = 2,      /* shape/dtype outside the requirements above */
  MOK_ERR_WORKSPACE = 3,        /* a buffer is smaller than the size query says */
  MOK_ERR_CUDA = 4,             /* a CUDA runtime call failed */
  MOK_ERR_NO_DEVICE = 5,        /* the current device is not sm_103 */
  MOK_ERR_SCRATCH_LIMIT = 6,    /* larger than the fixed scratch of mok_moe_dispatch_plan_noalloc */
  /* codes written on the device, read back with mok_get_device_status */
  MOK_ERR_DEVICE_NONFINITE = 16, /* a router logit was NaN; it was treated as -inf */
  MOK_ERR_DEVICE_INDEX = 17,     /* an expert index outside [0, E) was met and skipped */
  MOK_ERR_DEVICE_TIMEOUT = 18    /* a bounded wait inside a GEMM gave up; results invalid */
} mok_status;

typedef enum mok_dtype {
  MOK_BF16 = 0,  /* bf16 operands, fp32 accumulation, bf16 I/O */
  MOK_MXFP8 = 1, /* expert GEMMs on MXFP8 operands: E4M3 with one E8M0 scale per 32
                    values along K, fp32 accumulation (see mok_moe_forward) */
  MOK_NVFP4 = 2  /* expert GEMMs on NVFP4 operands (see mok_nvfp4_quantize),
                    each with its tensor scale over the whole tensor.  Forward:
                    x, W_gate_up along d and h, W_down along I; h rounded to
                    bf16 before its quantisation.  Backward: the gate/up dgrad
                    on dG/dU (bf16, along 2I, tensor scale over the
                    micro-batch's routed rows) and W_gate_up along 2I; the
                    down-projection dgrad and the weight gradients as in
                    MOK_BF16, with dp = <dy W_down, h>.  d and I multiples of
                    256; CTA-pair GEMMs only (MOK_FLAG_SINGLE_CTA_GEMM and
                    MOK_FLAG_RECOMPUTE_GATE_UP unsupported); no dispatched rows
                    are kept in saved */
} mok_dtype;

/* Output dtypes.  By default y, dx and the three weight gradients are fp32
 * (the value of the fp32 accumulation, unrounded, as an fp32 master-gradient
 * would receive it).  These flags select bf16 outputs (round to nearest even
 * of the same fp32 value). */
#define MOK_FLAG_BF16_ACT_OUT 0x1u   /* y and dx written as bf16 */
#define MOK_FLAG_BF16_WGRAD_OUT 0x2u /* dw_router, dw_gate_up, dw_down written as bf16 */
#define MOK_FLAG_ACCUMULATE_WGRAD 0x4u /* backward adds into the fp32 dw_* instead of
                                          overwriting them (gradient accumulation) */
/* Activation recompute: the forward keeps no pre-activations g, u; the
 * backward recomputes them from the dispatched rows with the same kernel and
 * schedule (results bitwise identical to the default).  Saves rows_max*2I*4
 * bytes of `saved` per micro-batch for one more gate/up GEMM in the backward.
 * (h is never kept: the backward always derives it from g, u.) */
#define MOK_FLAG_RECOMPUTE_GATE_UP 0x8u
/* Engine choice.  By default the grouped GEMMs with 256-wide tiles run on
 * clusters of two CTAs (256-row tiles, tcgen05.mma.cta_group::2, each SM
 * staging half of the weight tile).  This flag runs every GEMM on single-CTA
 * 128-row tiles instead.  Both engines accumulate every output element over
 * the same K sequence, so the results are bitwise the same. */
#define MOK_FLAG_SINGLE_CTA_GEMM 0x10u
/* Dispatch recompute ([dothoosh] "Ring buffer logic": the reverse ring walk
 * keeps forward activation replay small): `saved` keeps no dispatched token
 * rows (x_perm is MOK_NOT_KEPT, ring_slot_bytes 0); the forward dispatches
 * into its workspace and the backward gathers x into expert order again with
 * the same kernel, so every result is bitwise the same.  Saves
 * rows_max*d*2 bytes of `saved` per ring slot for one more row dispatch in
 * the backward.  MXFP8 keeps no dispatched rows anyway (the flag is accepted
 * and changes nothing there). */
#define MOK_FLAG_RECOMPUTE_DISPATCH 0x20u

/* Offset value of a mok_saved_layout field the flags leave out of `saved`. */
#define MOK_NOT_KEPT ((size_t)-1)

/* Layer shape.  T tokens of width d, E experts with FFN width I, top-k. */
typedef struct mok_moe_desc {
  int64_t T, d, E, I;
  int32_t k;
  int32_t dtype;       /* mok_dtype */
  int32_t mb_tokens;   /* 0: one pass over all T tokens; else tokens per
                          micro-batch (T a multiple of it) */
  int32_t ring_slots;  /* micro-batching: slots of the dispatched-row ring
                          (0 = one per micro-batch) */
  uint32_t flags;      /* MOK_FLAG_* */
  uint32_t reserved;
} mok_moe_desc;

/* Byte offsets, inside the `saved` buffer, of the forward results that the
 * backward consumes.  Row-indexed arrays use the padded row space: expert e
 * owns rows [padded_offsets[e], padded_offsets[e+1]), each segment a multiple
 * of 128 rows, its first counts[e] rows real, the padding rows after them zero
 * up to the next multiple of 64 rows (the weight gradients' K blocks read
 * them), and the rest of the segment unspecified (read by nothing).
 * With micro-batching the per-token fields describe micro-batch 0 (T =
 * mb_tokens) and micro-batch i's are at + i * mb_stride; x_perm is ring slot
 * 0 and slot j is at + j * ring_slot_bytes (micro-batch i was dispatched to
 * slot i % ring_slots). */
typedef struct mok_saved_layout {
  size_t status;          /* int32 device status word */
  size_t topk_idx;        /* int32 [T,k] expert of each slot, descending logit */
  size_t topk_w;          /* fp32 [T,k] routing weight of each slot */
  size_t counts;          /* int32 [E] rows routed to each expert */
  size_t offsets;         /* int32 [E+1] exclusive prefix sum of counts */
  size_t pos;             /* int32 [T,k] row of (t,s) in expert order */
  size_t token_of_row;    /* int32 [T*k] inverse of pos */
  size_t padded_offsets;  /* int32 [E+1] */
  size_t padded_pos;      /* int32 [T,k] row of (t,s) in the padded row space */
  size_t padded_token;    /* int32 [rows_max] token of each padded row; padding rows -1
                             up to the segment's next multiple of 64 rows, -2 after */
  size_t row_weight;      /* fp32 [rows_max] routing weight of each padded row, 0 for padding */
  size_t x_perm;          /* bf16 [rows_max, d] dispatched token rows; MOK_NOT_KEPT with
                             MOK_MXFP8 (its quantisers read the token rows through
                             padded_token instead) and with MOK_FLAG_RECOMPUTE_DISPATCH */
  size_t gate_up;         /* fp32 [rows_max, 2I] pre-activation gate (cols 0..I-1) and up (I..2I-1);
                             MOK_NOT_KEPT with MOK_FLAG_RECOMPUTE_GATE_UP */
  size_t nv_weight_scales; /* MOK_NVFP4: fp32 [2] tensor scales of W_gate_up and W_down (the
                             backward reuses W_gate_up's, so the weights must not change
                             between the two calls); MOK_NOT_KEPT otherwise */
  size_t w_gate_up_t;     /* W_gate_up along 2I, the gate/up dgrad's operand, written by the
                             forward (column c of expert e's [2I, d] matrix as row e*d + c):
                             MOK_NVFP4: E2M1 codes [E*d, I], then E*2I*d/16 E4M3 scale bytes;
                             MOK_MXFP8: E4M3 codes [E*d, 2I], then E*2I*d/32 E8M0 bytes; the
                             scales in the GEMM's tiled layout.  MOK_NOT_KEPT for MOK_BF16 */
  size_t w_down_col;      /* MOK_MXFP8: W_down fake-quantised along d (blocks of 32 rows of
                             each expert's [d, I] matrix), bf16 [E*d, I], the down dgrad's
                             operand, written by the forward; MOK_NOT_KEPT otherwise */
  size_t rows_max;        /* number of padded rows the buffers hold: T*k + 127*min(E, T*k), rounded to 128 */
  size_t mb_count;        /* micro-batches (1 without micro-batching) */
  size_t mb_stride;       /* bytes between consecutive micro-batches' fields */
  size_t ring_slots;      /* slots of dispatched rows (1 without micro-batching) */
  size_t ring_slot_bytes; /* bytes between ring slots (0 when x_perm is not kept) */
  size_t total;           /* size of `saved` in bytes */
} mok_saved_layout;

/* Sizes of the three caller-provided buffers for a layer of shape `desc`.
 *   fwd_ws_bytes : scratch of mok_moe_forward (free after it returns on the stream)
 *   saved_bytes  : forward results kept for mok_moe_backward
 *   bwd_ws_bytes : scratch of mok_moe_backward
 * Any output pointer may be NULL.  No device work. */
mok_status mok_moe_workspace_size(const mok_moe_desc* desc, size_t* fwd_ws_bytes,
                                  size_t* saved_bytes, size_t* bwd_ws_bytes);

/* Offsets of the forward results inside `saved` (see mok_saved_layout). */
mok_status mok_moe_saved_layout(const mok_moe_desc* desc, mok_saved_layout* out);

/* Forward of the layer ([dothoosh] "Hybrid communication": dispatch, expert
 * compute, combine; [gtnt] §1.1 router; [dothoosh] "Precision and scheduling":
 * SwiGLU experts):
 *   l = x W_r^T (+ b)                      fp32 logits
 *   S_t = top-k of l_t, larger first, exact ties to the lower expert index
 *   p_{t,s} = softmax over the k chosen logits (sums to 1)
 *   rows of expert e = tokens routed to e in ascending token order (dropless)
 *   [g | u] = X_e W_gu_e^T,  h = silu(g) * u,  O = h W_down_e^T
 *   y_t = sum_{s=0..k-1} p_{t,s} O[pos[t,s]]   (fp32 sum in slot order)
 * Precision: bf16 inputs and weights; fp32 accumulation; g and u kept in
 * fp32; h rounded to bf16 (the down GEMM's operand); O stays fp32.
 * x [T,d] bf16; w_router [E,d] bf16; router_bias [E] fp32 or NULL;
 * w_gate_up [E,2I,d] bf16 (gate rows 0..I-1, up rows I..2I-1);
 * w_down [E,d,I] bf16; y [T,d] output, fp32 (bf16 with MOK_FLAG_BF16_ACT_OUT).
 * saved: >= saved_bytes, filled for the backward; its status word is reset.
 * workspace: >= fwd_ws_bytes.  Buffers must not overlap. */
mok_status mok_moe_forward(const mok_moe_desc* desc, const void* x, const void* w_router,
                           const float* router_bias, const void* w_gate_up, const void* w_down,
                           void* y, void* saved, size_t saved_bytes, void* workspace,
                           size_t ws_bytes, void* stream);

/* Backward of L = sum(y * dy) given the `saved` of the matching forward
 * ([dothoosh] "Hybrid communication": reverse-combine, then reverse-dispatch;
 * "Precision and scheduling": router-weight gradient inside the SwiGLU
 * backward, dp = <dy W_down, h>):
 *   dA = dy_r W_down per routed row, dH = p dA (fp32), dp = <dA, h>;
 *   dG, dU from dH and the stored fp32 g, u; the gate/up dgrad takes them
 *   rounded to bf16 (dX rows fp32); the two weight-gradient GEMMs take dG, dU
 *   and p h as bf16 hi + lo pairs (about 16 significant bits).
 *   dx [T,d], dw_router [E,d], dw_gate_up [E,2I,d], dw_down [E,d,I]:
 *   outputs, overwritten, fp32 (bf16 with the MOK_FLAG_BF16_* flags); fp32
 *   accumulation inside, one writer per element, fixed summation order.
 *   The routing set is piecewise constant, so the router receives gradient
 *   only through p.  The bias gets no gradient.
 * x, w_router, router_bias, w_gate_up, w_down: the forward's inputs.
 * workspace: >= bwd_ws_bytes. */
mok_status mok_moe_backward(const mok_moe_desc* desc, const void* dy, const void* x,
                            const void* w_router, const float* router_bias,
                            const void* w_gate_up, const void* w_down, const void* saved,
                            size_t saved_bytes, void* dx, void* dw_router, void* dw_gate_up,
                            void* dw_down, void* workspace, size_t ws_bytes, void* stream);

/* Bytes of scratch that mok_moe_route / mok_moe_dispatch_plan need. */
mok_status mok_moe_stage_workspace_size(const mok_moe_desc* desc, size_t* bytes);

/* Router alone ([gtnt] §1.1): topk_idx [T,k] int32 and topk_w [T,k] fp32, as
 * in the forward.  workspace >= the stage size (its first word is the status). */
mok_status mok_moe_route(const mok_moe_desc* desc, const void* x, const void* w_router,
                         const float* router_bias, int32_t* topk_idx, float* topk_w,
                         void* workspace, size_t ws_bytes, void* stream);

/* Dispatch plan alone ([dothoosh] "Hybrid communication", "Ring buffer logic":
 * dropless): from topk_idx [T,k] int32 (values in [0,E)) computes
 *   counts [E], offsets [E+1] (exclusive prefix sum), pos [T,k] with
 *   pos[t,s] = offsets[e] + #{t' < t routed to e}, token_of_row [T*k] = pos^-1.
 * An index outside [0,E) sets MOK_ERR_DEVICE_INDEX and that slot is skipped
 * (its pos is -1).  workspace >= the stage size. */
mok_status mok_moe_dispatch_plan(const mok_moe_desc* desc, const int32_t* topk_idx,
                                 int32_t* counts, int32_t* offsets, int32_t* pos,
                                 int32_t* token_of_row, void* workspace, size_t ws_bytes,
                                 void* stream);

/* Dispatch plan without scratch memory from the caller.  No counterpart on
 * the pages: an addition of this library.
 *
 * Same inputs, outputs and results as mok_moe_dispatch_plan, for callers
 * that cannot allocate device memory at the point of the call and so have no
 * workspace to hand over: for instance code running inside another
 * library's allocator or memory-pool callback, or a process whose device
 * memory is entirely reserved up front by its framework.  It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *
 * The scratch is one 4 MiB array in device memory defined inside libmok
 * (held by every device that loads the library until the process exits).
 * Problems whose plan needs more than that -- roughly T*k*4 + 4*(T*k +
 * 127*E) + 8*E*ceil(T/256) bytes -- are rejected with
 * MOK_ERR_SCRATCH_LIMIT before anything is enqueued.
 *   status: device int32 that receives the device-side error code (reset to
 *           MOK_OK by this call), e.g. MOK_ERR_DEVICE_INDEX for an expert
 *           index outside [0, E); or NULL, and then the code stays inside the
 *           scratch where the caller cannot read it.
 * Every call resolves the array's device address in the current context
 * (cudaGetSymbolAddress, which allocates nothing).  The first call in a
 * process also loads the library's device code, so make one call before any
 * stream capture.  All calls share the one array, whose contents
 * are whatever the last call left: each call rewrites what it reads, and two
 * calls whose work overlaps on the GPU (different streams, or different host
 * threads on one device) race on it. */
mok_status mok_moe_dispatch_plan_noalloc(const mok_moe_desc* desc, const int32_t* topk_idx,
                                         int32_t* counts, int32_t* offsets, int32_t* pos,
                                         int32_t* token_of_row, int32_t* status, void* stream);

/* MXFP8 quantisation ([dothoosh] "Precision and scheduling": MXFP8; the
 * scaling rule is the OCP Microscaling v1.0 one): E4M3 elements with one E8M0
 * power-of-two scale per block of 32 values,
 *   shared = floor(log2 max|v|) - 8 (clamped to [-127,127], -127 for an
 *            all-zero block),  q = RNE_E4M3(v / 2^shared) saturating at 448.
 * in: bf16 [rows, cols] row-major.  along_rows = 0: blocks of 32 consecutive
 * values of a row (cols % 32 == 0); along_rows = 1: blocks of 32 consecutive
 * rows of a column (rows % 32 == 0, cols % 8 == 0).
 * out: bf16 [rows, cols], the dequantised values q * 2^shared (exact in
 * bf16); may equal `in`.  codes: NULL or uint8 [rows, cols] E4M3 codes.
 * in, out and codes 16-byte aligned (else MOK_ERR_INVALID_ARG).
 * scales: NULL or uint8 E8M0 bytes (shared + 127), [rows, cols/32]
 * (along_rows = 0) or [rows/32, cols] (along_rows = 1). */
mok_status mok_mx_quantize(const void* in, int64_t rows, int64_t cols, int along_rows, void* out,
                           uint8_t* codes, uint8_t* scales, void* stream);

/* NVFP4 ([dothoosh] "Background: solving the MoE bottleneck": Cursor's earlier
 * expert GEMMs ran in MXFP8 and NVFP4; the format is NVIDIA's, the order of
 * its fp32 operations this library's): E2M1 elements, one E4M3 scale per 16
 * consecutive values along K, one fp32 scale per tensor.
 *   g   = amax / 2688 (= 6 * 448), 1 for an all-zero tensor
 *   s_b = RNE_E4M3(amax_b * RN(1 / RN(6 g)))          (<= 448)
 *   q   = RNE_E2M1(v * RN(1 / RN(s_b g)))             (+-6 saturated; the
 *         reciprocal capped at the largest finite float; 0 where s_b = 0)
 * (RN: one fp32 rounding to nearest even.)
 * Finite inputs only (a NaN is ignored by the tensor amax).
 *
 * mok_nvfp4_tensor_scale: g of the n bf16 values at `in` (n % 8 == 0, `in`
 * 16-byte aligned), written to the device fp32 *g (used as scratch first). */
mok_status mok_nvfp4_tensor_scale(const void* in, int64_t n, float* g, void* stream);

/* NVFP4 codes and block scales of bf16 [rows, cols] row-major (blocks of 16
 * along a row, cols % 16 == 0) with the tensor scale at device *g:
 * codes uint8 [rows, cols/2] (value 2i in the low nibble of byte i, 2i+1 in
 * the high one; 8-byte aligned), scales uint8 [rows, cols/16] E4M3 bytes. */
mok_status mok_nvfp4_quantize(const void* in, int64_t rows, int64_t cols, const float* g,
                              uint8_t* codes, uint8_t* scales, void* stream);

/* NVFP4 of the columns of ng stacked bf16 matrices [K, C] (row-major, K
 * along the rows; blocks of 16 along K) with the tensor scale at device *g:
 * out row i*C + c holds column c of matrix i.  codes uint8 [ng*C, K/2] (low
 * nibble first), scales uint8 [ng*C, K/16] E4M3 bytes.  K % 64 == 0,
 * C % 128 == 0; in and codes 16-byte aligned.  The layer uses it for
 * W_gate_up along 2I, the gate/up dgrad's reduction dimension. */
mok_status mok_nvfp4_quantize_cols(const void* in, int64_t ng, int64_t K, int64_t C,
                                   const float* g, uint8_t* codes, uint8_t* scales,
                                   void* stream);

/* Dense NVFP4 GEMM on the block-scaled FP4 tensor cores
 * (tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X), a diagnostic of
 * the scale placement:  C[M,N] fp32 = gA gB sum_k qA[m,k] sA[m,k/16] qB[n,k]
 * sB[n,k/16], with A [M, K/2] and B [N, K/2] codes, A_scales [M, K/16] and
 * B_scales [N, K/16] bytes (as mok_nvfp4_quantize writes them) and the tensor
 * scales at device A_g, B_g.  M, N multiples of 128, K of 256.  workspace: at
 * least 256 bytes (its first int32 is the device status word). */
mok_status mok_gemm_nvfp4(int64_t M, int64_t N, int64_t K, const uint8_t* A,
                          const uint8_t* A_scales, const float* A_g, const uint8_t* B,
                          const uint8_t* B_scales, const float* B_g, float* C, void* workspace,
                          size_t ws_bytes, void* stream);

/* Dense GEMM through the layer's tcgen05 engine, C[M,N] = A B in bf16 with
 * fp32 accumulation and bf16 output (a diagnostic of the grouped engine):
 *   a_mn_major = 0: A stored [M,K];  1: A stored [K,M]
 *   b_mn_major = 0: B stored [N,K];  1: B stored [K,N]
 * (a_mn_major, b_mn_major) = (1, 0) is not served.  M, N, K multiples of 128.
 * workspace >= 256 bytes (status word). */
mok_status mok_gemm_bf16(int64_t M, int64_t N, int64_t K, const void* A, int a_mn_major,
                         const void* B, int b_mn_major, void* C, void* workspace,
                         size_t ws_bytes, void* stream);

/* Dense MXFP8 GEMM on the block-scaled tensor cores ([dothoosh] "MoK
 * technical details", "Precision and scheduling": MXFP8 expert GEMMs):
 *   C[m,n] = sum_k A[m,k] 2^(sa[m,k/32]-127) * B[n,k] 2^(sb[n,k/32]-127)
 * A: uint8 [M,K] E4M3 codes, sa: uint8 [M,K/32] E8M0 scale bytes; B, sb the
 * same for [N,K]; C: fp32 [M,N] (fp32 accumulation).  This is the layout
 * mok_mx_quantize writes with along_rows = 0.  M, N, K multiples of 128;
 * A, B, C 16-byte aligned, sa, sb 4-byte aligned.  cta_pair = 0: 128 x 128
 * tiles on single CTAs; 1: 256 x 256 tiles on clusters of two CTAs
 * (tcgen05.mma.cta_group::2; M, N multiples of 256).  Both accumulate every
 * element over the same K sequence.  workspace >= 256 bytes (status word). */
mok_status mok_gemm_mxfp8(int64_t M, int64_t N, int64_t K, const uint8_t* A, const uint8_t* sa,
                          const uint8_t* B, const uint8_t* sb, float* C, int cta_pair,
                          void* workspace, size_t ws_bytes, void* stream);

/* Failure-path self-test: enqueues one CTA that waits on an mbarrier phase
 * nothing completes.  The wait is the bounded one every GEMM uses: it gives
 * up after its limit (0.2 s) and the kernel writes MOK_ERR_DEVICE_TIMEOUT to
 * the status word at the start of `workspace` (>= 256 bytes, reset first)
 * and returns, leaving the context usable.  Read it with
 * mok_get_device_status. */
mok_status mok_selftest_bounded_wait(void* workspace, size_t ws_bytes, void* stream);

/* Diagnostic: sets `bytes` bytes at device address `dst` to zero with bulk
 * asynchronous stores (cp.async.bulk) from a zeroed shared-memory chunk, the
 * store path the row-dispatch kernel writes with; timed alone it measures the
 * HBM write bandwidth that path reaches.  dst 16-byte aligned and bytes a
 * multiple of 16, else MOK_ERR_INVALID_ARG; bytes = 0 enqueues nothing.
 * Asynchronous on `stream`; the caller owns `dst`. */
mok_status mok_fill_zero(void* dst, size_t bytes, void* stream);

/* Waits for `stream`, then reads the device status word at the start of
 * `buf` (the `saved` buffer of forward/backward, or the workspace of the
 * other entry points) into *code (a mok_status; MOK_OK = no device error). */
mok_status mok_get_device_status(const void* buf, void* stream, int32_t* code);

/* Static description of a status code. */
const char* mok_status_string(mok_status status);

/* Number of kernels enqueued since the start of the last mok_moe_forward
 * call (host-side count; after a forward + backward pair it is the number
 * of kernels of one training step of the layer). */
int32_t mok_last_launch_count(void);

/* Per-kernel timing.  While enabled, the library brackets each kernel it
 * enqueues with a pair of CUDA events on the same stream.  The kernels are
 * unchanged, but the events are stream operations between them: they keep a
 * GEMM's programmatic dependent launch from overlapping the kernel before it,
 * so a profiled step runs slightly slower than an unprofiled one.
 * mok_profile_collect waits
 * for the recorded events, then writes up to `max` entries, one per kernel
 * name, with launch counts and summed durations since the last reset, and
 * stores the number of entries in *n.  Not thread-safe: enable it around a
 * single-threaded timing loop. */
typedef struct mok_kernel_time {
  char name[48];
  int32_t launches;
  double total_ms;
} mok_kernel_time;
mok_status mok_profile_enable(int on);
mok_status mok_profile_reset(void);
mok_status mok_profile_collect(mok_kernel_time* out, int32_t max, int32_t* n);

#ifdef __cplusplus
}
#endif

#endif /* MOK_H_ */
