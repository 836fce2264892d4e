// NVFP4: E2M1 elements, one E4M3 scale per 16 consecutive values along K, and
// one fp32 scale per tensor -- the quantiser and a dense GEMM on the
// block-scaled FP4 tensor cores (tcgen05.mma.kind::mxf4nvf4.block_scale,
// scale_vec::4X).
//
// Source: [dothoosh] "Cursor Mixture-of-Kittens cuts MoE training latency by
// 5.8x", section "Background: solving the MoE bottleneck": Cursor's earlier
// training kernels ran the expert GEMMs in MXFP8 and NVFP4.  The pages do not
// define the format; NVIDIA's published NVFP4 is taken, with one fixed order
// of fp32 operations:
//   tensor scale   g   = amax / 2688 (6 * 448), or 1 for an all-zero tensor
//   block scale    s_b = RNE_E4M3(amax_b * RN(1 / RN(6 g)))
//   element        q   = RNE_E2M1(v * RN(1 / RN(s_b g)))   (the reciprocal
//                        capped at the largest finite float; 0 where s_b = 0),
//                        saturating at +-6
//   value          q * s_b * g.
// (Products with rounded reciprocals rather than quotients: one multiply per
// element, which keeps the quantisers off the ALU limit.)
//
// The GEMM computes C[M,N] = alpha * sum_k qA[m,k] sA[m,k/16] qB[n,k] sB[n,k/16]
// with alpha = gA * gB: the tensor cores apply the block scales, the epilogue
// the tensor scales.  One CTA per 128 x 128 tile of C:
//   warp 0      producer: TMA loads of the A and B code tiles (128 rows x 128
//               bytes = 256 values, 128-byte swizzle) and the gather of their
//               scale bytes: per 64-value MMA step j one 512-byte block, row r
//               at byte 16*(r%32) + 4*(r/32) + i for its 16-value block i;
//   warp 1      MMA: per stage, tcgen05.cp of the eight scale blocks to TMEM
//               (32x128b, replicated to the four lane quarters) and four
//               tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X (K = 64
//               each, four scales per row);
//   warps 2..5  epilogue: TMEM -> registers -> alpha * acc -> fp32 C.
#include <cuda.h>
#include <cuda_runtime.h>

#include "mok_internal.h"
#include "mx.cuh"
#include "ptx.cuh"
#include "quant_tile.cuh"

namespace mok {
namespace {

// ------------------------------------------------------------- quantiser --

}  // namespace

// Byte of the scale of row r, 16-value block c16, in the tiled layout of a
// matrix with 64 * nkb columns: one 512-byte block per 128 rows x 64 values,
// the blocks of a 128-row tile consecutive along K, and inside a block row r
// at byte 16 * (r % 32) + 4 * ((r / 32) % 4) + c16 % 4 -- the arrangement
// the 32x128b scale copy to TMEM takes, so a CTA loads a stage's blocks with
// one TMA copy.
static __host__ __device__ inline long long nv_tiled_off(long long r, long long c16,
                                                        long long nkb) {
  return ((r >> 7) * nkb + (c16 >> 2)) * 512 + 16 * (r & 31) + 4 * ((r >> 5) & 3) + (c16 & 3);
}

namespace {

// Largest |value| of eight bf16 values (one 16-byte chunk).
__device__ __forceinline__ float amax8(const uint4& w) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
  float m = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    m = fmaxf(m, fabsf(bf16lo(u[j])));
    m = fmaxf(m, fabsf(bf16hi(u[j])));
  }
  return m;
}

// The warp's amax into *amax_bits as the bits of a non-negative float (the
// integer order of such bits is their value order, so atomicMax takes the
// maximum whatever the order of the updates).
__device__ __forceinline__ void amax_publish(float m, unsigned* amax_bits) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if ((threadIdx.x & 31) == 0) atomicMax(amax_bits, __float_as_uint(m));
}

// Plain tensor of nchunks 16-byte chunks (8 bf16 values each), grid-strided
// with four independent loads in flight per thread.
__global__ void nv_amax_kernel(const uint4* __restrict__ in, long long nchunks,
                               unsigned* __restrict__ amax_bits) {
  float m = 0.f;
  const long long G = static_cast<long long>(gridDim.x) * blockDim.x;
  long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 3 * G < nchunks; i += 4 * G) {
    uint4 w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) w[j] = __ldg(in + i + j * G);
#pragma unroll
    for (int j = 0; j < 4; ++j) m = fmaxf(m, amax8(w[j]));
  }
  for (; i < nchunks; i += G) m = fmaxf(m, amax8(__ldg(in + i)));
  amax_publish(m, amax_bits);
}

// A [nrows, row_chunks] tensor, one warp per row (the lanes split the row's
// chunks, four loads in flight each): rows_dev (or NULL) limits it to the
// first *rows_dev rows, and rows r with rowmap[r] < 0 (padding) do not count.
__global__ void nv_amax_rows_kernel(const uint4* __restrict__ in, long long nrows,
                                    int row_chunks, unsigned* __restrict__ amax_bits,
                                    const int32_t* __restrict__ rows_dev,
                                    const int32_t* __restrict__ rowmap) {
  if (rows_dev) {
    const long long lim = *rows_dev;
    nrows = lim < nrows ? lim : nrows;
  }
  const int lane = threadIdx.x & 31;
  const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  float m = 0.f;
  for (long long r = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
       r < nrows; r += nw) {
    if (rowmap && rowmap[r] < 0) continue;  // the same row for the whole warp
    const uint4* p = in + r * row_chunks;
    int c = lane;
    for (; c + 96 < row_chunks; c += 128) {
      uint4 w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = __ldg(p + c + 32 * j);
#pragma unroll
      for (int j = 0; j < 4; ++j) m = fmaxf(m, amax8(w[j]));
    }
    for (; c < row_chunks; c += 32) m = fmaxf(m, amax8(__ldg(p + c)));
  }
  amax_publish(m, amax_bits);
}

// *g (holding the amax bits) <- the tensor scale
__global__ void nv_scale_kernel(float* g) {
  const float amax = __uint_as_float(*reinterpret_cast<unsigned*>(g));
  *g = amax > 0.f ? amax / 2688.0f : 1.0f;
}

__device__ __forceinline__ uint8_t cvt_e2m1x2(float hi, float lo) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return static_cast<uint8_t>(r);
}

// One NVFP4 block of 16 values: its E4M3 scale byte (returned) and its eight
// code bytes (value 2i in the low nibble of byte i) in c.  r6 = RN(1 / RN(6 g)):
//   s_b = RNE_E4M3(amax_b * r6),  q = RNE_E2M1(v * r_b),  r_b = RN(1 / RN(s_b g))
// (r_b capped at the largest finite float, so that v = 0 gives 0).
__device__ __forceinline__ uint8_t nv_block(const float (&v)[16], float g, float r6,
                                            uint32_t (&c)[2]) {
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
  const uint8_t sb = static_cast<uint8_t>(cvt_e4m3x2(0.f, amax * r6) & 0xFFu);
  float sb_hi, sb_f;
  e4m3x2_to_f32(sb, &sb_hi, &sb_f);
  c[0] = c[1] = 0u;
  if (sb != 0) {
    const float rb = fminf(__frcp_rn(sb_f * g), 3.402823466e38f);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      c[j >> 2] |= static_cast<uint32_t>(cvt_e2m1x2(v[2 * j + 1] * rb, v[2 * j] * rb))
                   << (8 * (j & 3));
  }
  return sb;
}

// One thread per block of 16 values along a row: 8 code bytes (value 2i in
// the low nibble of byte i, 2i+1 in the high one) and one E4M3 scale byte.
// tiled_nkb > 0: the scale bytes go to the tiled layout of a matrix with
// 64 * tiled_nkb columns (nv_tiled_off); 0: row-major [rows, cols/16].
// map (or NULL): output row r takes input row map[r] when that is a row of
// the input (0 <= map[r] < T), zeros otherwise (codes 0, scale 0).
// rows_dev (or NULL): only the first *rows_dev rows (the rows anything reads).
__global__ void nv_quant_kernel(const uint4* __restrict__ in, long long nblk, int blk_per_row,
                                const float* __restrict__ g_ptr, uint8_t* __restrict__ codes,
                                uint8_t* __restrict__ scales, long long tiled_nkb,
                                const int32_t* __restrict__ map, int T,
                                const int32_t* __restrict__ rows_dev) {
  if (rows_dev) {
    const long long lim = static_cast<long long>(*rows_dev) * blk_per_row;
    nblk = lim < nblk ? lim : nblk;
  }
  const float g = *g_ptr;
  const float r6 = __frcp_rn(6.0f * g);
  const long long G = static_cast<long long>(gridDim.x) * blockDim.x;
  long long b = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  // row and block-in-row of b, stepped by G (one division per thread)
  long long r = b / blk_per_row;
  int c16 = static_cast<int>(b - r * blk_per_row);
  const long long dr = G / blk_per_row;
  const int dc = static_cast<int>(G - dr * blk_per_row);
  for (; b < nblk; b += G) {
    long long src = b;
    bool zero = false;
    if (map) {
      const int t = map[r];
      zero = !(t >= 0 && t < T);
      src = static_cast<long long>(zero ? 0 : t) * blk_per_row + c16;
    }
    uint4 w0 = make_uint4(0u, 0u, 0u, 0u), w1 = w0;
    if (!zero) {
      w0 = in[2 * src];
      w1 = in[2 * src + 1];
    }
    const uint32_t u[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    float v[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[2 * j] = bf16lo(u[j]);
      v[2 * j + 1] = bf16hi(u[j]);
    }
    uint32_t c[2];
    const uint8_t sb = nv_block(v, g, r6, c);
    *reinterpret_cast<uint2*>(codes + 8 * b) = make_uint2(c[0], c[1]);
    scales[tiled_nkb > 0 ? nv_tiled_off(r, c16, tiled_nkb) : b] = sb;
    r += dr;
    c16 += dc;
    if (c16 >= blk_per_row) {
      c16 -= blk_per_row;
      ++r;
    }
  }
}

// NVFP4 of `ng` stacked bf16 matrices [K, C] (row-major) in both
// orientations from one read: the rows (blocks of 16 along C; codes
// [ng*K, C/2], scales tiled with C/64 blocks per 128 rows) and the columns
// (blocks of 16 along K; out row g*C + c holds column c of matrix g: codes
// [ng*C, K/2], scales tiled with K/64 blocks per 128 rows, or row-major
// [ng*C, K/16]).  Either output may be skipped (NULL codes).  Persistent CTAs
// walk the 128 x 128 tiles (quant_tile.cuh).  Warps 0-3 take the rows, one
// row per thread (64 contiguous code bytes); warps 4-7 the columns, a pair of
// adjacent columns and half of the tile's K per thread, read as 4-byte pairs
// (one 128-byte run per warp and row), so each column gets a 32-byte code run.
__global__ void __launch_bounds__(256, 3)
    nv_quant_2d_kernel(const uint16_t* __restrict__ in, int K, int C, int ng,
                       const float* __restrict__ g_ptr, uint8_t* __restrict__ rcodes,
                       uint8_t* __restrict__ rscales, uint8_t* __restrict__ ccodes,
                       uint8_t* __restrict__ cscales, bool ctiled) {
  extern __shared__ __align__(16) uint16_t qt_smem[];
  const float g = *g_ptr;
  const float r6 = __frcp_rn(6.0f * g);
  const int t = threadIdx.x;
  qt_walk(in, K, C, ng, qt_smem, [&](uint16_t* tile, const QtTile& q) {
    if (t < 128) {
      if (!rcodes) return;
      // row t of the tile: eight blocks along C
      const long long row = static_cast<long long>(q.grp) * K + q.kt * 128 + t;
      uint4* cp = reinterpret_cast<uint4*>(rcodes + row * (C / 2) + q.ct * 64);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t sw = 0u, cw[8];
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
          const uint16_t* src = tile + t * kQtPitch + 64 * half + 16 * blk;
          const uint4 a = *reinterpret_cast<const uint4*>(src);
          const uint4 b = *reinterpret_cast<const uint4*>(src + 8);
          const uint32_t u[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
          float v[16];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            v[2 * j] = bf16lo(u[j]);
            v[2 * j + 1] = bf16hi(u[j]);
          }
          uint32_t c[2];
          sw |= static_cast<uint32_t>(nv_block(v, g, r6, c)) << (8 * blk);
          cw[2 * blk] = c[0];
          cw[2 * blk + 1] = c[1];
        }
        cp[2 * half] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
        cp[2 * half + 1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
        *reinterpret_cast<uint32_t*>(
            rscales + nv_tiled_off(row, q.ct * 8 + 4 * half, C / 64)) = sw;
      }
    } else {
      if (!ccodes) return;
      // columns 2p, 2p+1 of the tile, K rows 64 h .. 64 h + 63: four blocks each
      const int p = t & 63, h = (t - 128) >> 6;
      uint32_t sw0 = 0u, sw1 = 0u, cw0[8], cw1[8];
#pragma unroll
      for (int blk = 0; blk < 4; ++blk) {
        const uint16_t* src = tile + (64 * h + 16 * blk) * kQtPitch + 2 * p;
        float v0[16], v1[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const uint32_t w = *reinterpret_cast<const uint32_t*>(src + j * kQtPitch);
          v0[j] = bf16lo(w);
          v1[j] = bf16hi(w);
        }
        uint32_t c[2];
        sw0 |= static_cast<uint32_t>(nv_block(v0, g, r6, c)) << (8 * blk);
        cw0[2 * blk] = c[0];
        cw0[2 * blk + 1] = c[1];
        sw1 |= static_cast<uint32_t>(nv_block(v1, g, r6, c)) << (8 * blk);
        cw1[2 * blk] = c[0];
        cw1[2 * blk + 1] = c[1];
      }
      const long long row = static_cast<long long>(q.grp) * C + q.ct * 128 + 2 * p;
      const long long k16 = q.kt * 8 + 4 * h;
      uint4* c0 = reinterpret_cast<uint4*>(ccodes + row * (K / 2) + k16 * 8);
      uint4* c1 = reinterpret_cast<uint4*>(ccodes + (row + 1) * (K / 2) + k16 * 8);
      c0[0] = make_uint4(cw0[0], cw0[1], cw0[2], cw0[3]);
      c0[1] = make_uint4(cw0[4], cw0[5], cw0[6], cw0[7]);
      c1[0] = make_uint4(cw1[0], cw1[1], cw1[2], cw1[3]);
      c1[1] = make_uint4(cw1[4], cw1[5], cw1[6], cw1[7]);
      *reinterpret_cast<uint32_t*>(cscales + (ctiled ? nv_tiled_off(row, k16, K / 64)
                                                     : row * (K / 16) + k16)) = sw0;
      *reinterpret_cast<uint32_t*>(cscales + (ctiled ? nv_tiled_off(row + 1, k16, K / 64)
                                                     : (row + 1) * (K / 16) + k16)) = sw1;
    }
  });
}

// ---------------------------------------------------------------- GEMM ----

constexpr int kNvStages = 4;
constexpr int kNvTile = 128;                  // M = N = 128
constexpr int kNvBK = 128;                    // code bytes per row per stage (256 values)
constexpr int kNvCodeBytes = kNvTile * kNvBK;  // 16 KB per operand tile
constexpr int kNvSfBlock = 512;               // 128 rows x 4 scale bytes (one MMA step)
constexpr int kNvSfBytes = 4 * kNvSfBlock;    // four MMA steps per stage
constexpr int kNvStageBytes = 2 * kNvCodeBytes + 2 * kNvSfBytes;  // 36 KB
constexpr int kNvThreads = 192;
// TMEM: accumulator columns [0,128); stage s keeps A scales at 128 + 32s
// (four columns per MMA step) and B scales at 144 + 32s
constexpr uint32_t kNvTmemCols = 256;
constexpr int kNvSmem = 1024 + kNvStages * kNvStageBytes + 256;

__global__ void __launch_bounds__(kNvThreads, 1)
    nv_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const uint8_t* __restrict__ sa, const uint8_t* __restrict__ sb,
                   const float* __restrict__ ga, const float* __restrict__ gb, float* C, int N,
                   int K, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kNvStages * kNvStageBytes);
  uint64_t* empty = full + kNvStages;
  uint64_t* tfull = empty + kNvStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tfull + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tile = blockIdx.x, m_tile = blockIdx.y;
  const int nkb = K / (2 * kNvBK);  // 256 values per stage
  const long long ks = K / 16;      // scale bytes per row

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNvStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kNvTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  volatile int* vabort = abort_flag;

  if (warp == 0) {
    // ---------------------------------------------------------- producer --
    bool ok = true;
    for (int kb = 0; kb < nkb && ok; ++kb) {
      const int s = kb % kNvStages;
      const uint32_t par = static_cast<uint32_t>((kb / kNvStages) & 1);
      if (!mbar_wait(&empty[s], par ^ 1u, vabort)) {
        ok = false;
        break;
      }
      uint8_t* st = smem + s * kNvStageBytes;
      // scale bytes of this stage: 16 per row, 4 per MMA step
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        gather_sf(st + 2 * kNvCodeBytes + j * kNvSfBlock, sa, ks, (long long)m_tile * kNvTile,
                  (long long)kb * 16 + 4 * j, lane);
        gather_sf(st + 2 * kNvCodeBytes + kNvSfBytes + j * kNvSfBlock, sb, ks,
                  (long long)n_tile * kNvTile, (long long)kb * 16 + 4 * j, lane);
      }
      fence_proxy_async_smem();  // the scale copies read these bytes through the async proxy
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(&full[s], 2 * kNvCodeBytes);
        tma_load_2d(st, &tmA, &full[s], kb * kNvBK, m_tile * kNvTile);
        tma_load_2d(st + kNvCodeBytes, &tmB, &full[s], kb * kNvBK, n_tile * kNvTile);
      }
    }
    if (!ok && lane == 0) {
      *vabort = 1;
      set_status(status, MOK_ERR_DEVICE_TIMEOUT);
      spin_ns(1000000ull);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // --------------------------------------------------------------- MMA --
      bool ok = true;
      for (int kb = 0; kb < nkb && ok; ++kb) {
        const int s = kb % kNvStages;
        const uint32_t par = static_cast<uint32_t>((kb / kNvStages) & 1);
        if (!mbar_wait(&full[s], par, vabort)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t a_base = smem_addr(smem + s * kNvStageBytes);
        const uint32_t b_base = a_base + kNvCodeBytes;
        const uint32_t sfa_col = tmem_base + 128u + 32u * s;
        const uint32_t sfb_col = sfa_col + 16u;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          tmem_cp_sf(sfa_col + 4u * j, smem_desc_sf(a_base + 2 * kNvCodeBytes + j * kNvSfBlock));
          tmem_cp_sf(sfb_col + 4u * j,
                     smem_desc_sf(a_base + 2 * kNvCodeBytes + kNvSfBytes + j * kNvSfBlock));
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          // 64 values = 32 bytes per step inside the 128-byte swizzled rows
          const uint64_t ad = smem_desc_sw128(a_base + j * 32, 16, 1024);
          const uint64_t bd = smem_desc_sw128(b_base + j * 32, 16, 1024);
          mma_nvf4(tmem_base, ad, bd, idesc_nvf4(kNvTile, kNvTile), sfa_col + 4u * j,
                   sfb_col + 4u * j, (kb | j) != 0 ? 1u : 0u);
        }
        mma_commit(&empty[s]);
      }
      if (ok) {
        mma_commit(tfull);
      } else {
        *vabort = 1;
        set_status(status, MOK_ERR_DEVICE_TIMEOUT);
        mma_commit(tfull);  // lets the epilogue leave; its results are void
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue --
    const int q = warp & 3;  // TMEM lane quarter of this warp
    const int zero = 0;
    if (!mbar_wait(tfull, 0, &zero)) set_status(status, MOK_ERR_DEVICE_TIMEOUT);
    tc_fence_after_sync();
    const float alpha = *ga * *gb;
    const long long row = (long long)m_tile * kNvTile + q * 32 + lane;
    float* out = C + row * N + (long long)n_tile * kNvTile;
#pragma unroll 1
    for (int c = 0; c < kNvTile; c += 16) {
      uint32_t r[16];
      tmem_ld16(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + c, r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; j += 4)
        *reinterpret_cast<float4*>(out + c + j) =
            make_float4(alpha * __uint_as_float(r[j]), alpha * __uint_as_float(r[j + 1]),
                        alpha * __uint_as_float(r[j + 2]), alpha * __uint_as_float(r[j + 3]));
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kNvTmemCols);
  }
}

}  // namespace

cudaError_t launch_nv_tensor_scale(const void* in, long long n, float* g, cudaStream_t st,
                                   const int32_t* rows_dev, long long row_elems,
                                   const int32_t* rowmap) {
  if ((rows_dev || rowmap) && row_elems < 8) return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(g, 0, sizeof(float), st);
  if (e != cudaSuccess) return e;
  const long long nchunks = n / 8;
  if (nchunks > 0) {
    const long long cap = static_cast<long long>(num_sms_current_device()) * 8;
    ProfScope prof("nvfp4_amax", st);
    if (rows_dev || rowmap) {
      // whole rows of row_elems values (a multiple of 8)
      const long long row_chunks = row_elems / 8, nrows = nchunks / row_chunks;
      if (row_elems % 8 || row_chunks > (1 << 30)) return cudaErrorInvalidValue;
      long long grid = (nrows + 7) / 8;  // eight warps per CTA, one row each
      if (grid > cap) grid = cap;
      if (grid < 1) grid = 1;
      nv_amax_rows_kernel<<<static_cast<unsigned>(grid), 256, 0, st>>>(
          static_cast<const uint4*>(in), nrows, static_cast<int>(row_chunks),
          reinterpret_cast<unsigned*>(g), rows_dev, rowmap);
    } else {
      long long grid = (nchunks + 255) / 256;
      if (grid > cap) grid = cap;
      nv_amax_kernel<<<static_cast<unsigned>(grid), 256, 0, st>>>(
          static_cast<const uint4*>(in), nchunks, reinterpret_cast<unsigned*>(g));
    }
    count_launch();
  }
  nv_scale_kernel<<<1, 1, 0, st>>>(g);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_nv_quant_2d(const void* in, long long ng, long long K, long long C,
                               const float* g, uint8_t* rcodes, uint8_t* rscales,
                               uint8_t* ccodes, uint8_t* cscales, cudaStream_t st, bool ctiled) {
  // whole 128 x 128 tiles (whole 128-row blocks of both tiled layouts)
  if (K % 128 || C % 128 || ng <= 0 || K / 128 > 65535 || C / 128 > 65535 || ng > 65535)
    return cudaErrorInvalidValue;
  if ((rcodes && !rscales) || (ccodes && !cscales) || (!rcodes && !ccodes))
    return cudaErrorInvalidValue;
  if (reinterpret_cast<uintptr_t>(in) % 16 || reinterpret_cast<uintptr_t>(rcodes) % 16 ||
      reinterpret_cast<uintptr_t>(ccodes) % 16 || reinterpret_cast<uintptr_t>(rscales) % 4 ||
      reinterpret_cast<uintptr_t>(cscales) % 4)
    return cudaErrorInvalidValue;
  ProfScope prof(rcodes && ccodes ? "nvfp4_quantize_2d" : "nvfp4_quantize_cols", st);
  const cudaError_t e = cudaFuncSetAttribute(  // the two staging buffers
      nv_quant_2d_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kQtSmemBytes);
  if (e != cudaSuccess) return e;
  const long long ntiles = ng * (K / 128) * (C / 128);
  if (ntiles >= (1LL << 31)) return cudaErrorInvalidValue;
  const long long cap = static_cast<long long>(num_sms_current_device()) * 3;
  nv_quant_2d_kernel<<<static_cast<unsigned>(ntiles < cap ? ntiles : cap), 256, kQtSmemBytes,
                       st>>>(static_cast<const uint16_t*>(in), static_cast<int>(K),
                             static_cast<int>(C), static_cast<int>(ng), g, rcodes, rscales,
                             ccodes, cscales, ctiled);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_nv_quant_tiled(const void* in, long long rows, long long cols, const float* g,
                                  uint8_t* codes, uint8_t* scales, const int32_t* map, int T,
                                  cudaStream_t st, const int32_t* rows_dev) {
  const long long nblk = rows * cols / 16;
  if (nblk == 0) return cudaSuccess;
  long long grid = (nblk + 255) / 256;
  const long long cap = static_cast<long long>(num_sms_current_device()) * 16;
  if (grid > cap) grid = cap;
  ProfScope prof("nvfp4_quantize", st);
  nv_quant_kernel<<<static_cast<unsigned>(grid), 256, 0, st>>>(
      static_cast<const uint4*>(in), nblk, static_cast<int>(cols / 16), g, codes, scales,
      cols / 64, map, T, rows_dev);
  count_launch();
  return cudaGetLastError();
}

}  // namespace mok

using namespace mok;

extern "C" mok_status mok_nvfp4_tensor_scale(const void* in, int64_t n, float* g, void* stream) {
  if (n < 0) return MOK_ERR_INVALID_ARG;
  if (!g || (n > 0 && !in)) return MOK_ERR_INVALID_ARG;
  if (n % 8 != 0 || (reinterpret_cast<uintptr_t>(in) & 15u) ||
      (reinterpret_cast<uintptr_t>(g) & 3u))
    return MOK_ERR_INVALID_ARG;
  mok_status s = mok_check_device();
  if (s != MOK_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(g, 0, sizeof(float), st) != cudaSuccess) return MOK_ERR_CUDA;
  const long long nchunks = n / 8;
  if (nchunks > 0) {
    long long grid = (nchunks + 255) / 256;
    const long long cap = static_cast<long long>(num_sms_current_device()) * 8;
    if (grid > cap) grid = cap;
    ProfScope prof("nvfp4_amax", st);
    nv_amax_kernel<<<static_cast<unsigned>(grid), 256, 0, st>>>(
        static_cast<const uint4*>(in), nchunks, reinterpret_cast<unsigned*>(g));
    count_launch();
  }
  nv_scale_kernel<<<1, 1, 0, st>>>(g);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? MOK_OK : MOK_ERR_CUDA;
}

extern "C" mok_status mok_nvfp4_quantize(const void* in, int64_t rows, int64_t cols,
                                         const float* g, uint8_t* codes, uint8_t* scales,
                                         void* stream) {
  if (rows < 0 || cols <= 0 || cols % 16 != 0) return MOK_ERR_INVALID_ARG;
  if (rows > 0 && (!in || !g || !codes || !scales)) return MOK_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(in) & 15u) || (reinterpret_cast<uintptr_t>(codes) & 7u) ||
      (reinterpret_cast<uintptr_t>(g) & 3u))
    return MOK_ERR_INVALID_ARG;
  mok_status s = mok_check_device();
  if (s != MOK_OK) return s;
  const long long nblk = rows * cols / 16;
  if (nblk == 0) return MOK_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  long long grid = (nblk + 255) / 256;
  const long long cap = static_cast<long long>(num_sms_current_device()) * 16;
  if (grid > cap) grid = cap;
  ProfScope prof("nvfp4_quantize", st);
  nv_quant_kernel<<<static_cast<unsigned>(grid), 256, 0, st>>>(
      static_cast<const uint4*>(in), nblk, static_cast<int>(cols / 16), g, codes, scales, 0,
      nullptr, 0, nullptr);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? MOK_OK : MOK_ERR_CUDA;
}

extern "C" mok_status mok_nvfp4_quantize_cols(const void* in, int64_t ng, int64_t K, int64_t C,
                                              const float* g, uint8_t* codes, uint8_t* scales,
                                              void* stream) {
  if (ng < 0 || K <= 0 || C <= 0 || K % 128 || C % 128) return MOK_ERR_INVALID_ARG;
  if (ng > 0 && (!in || !g || !codes || !scales)) return MOK_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(in) & 15u) || (reinterpret_cast<uintptr_t>(codes) & 15u) ||
      (reinterpret_cast<uintptr_t>(scales) & 3u) || (reinterpret_cast<uintptr_t>(g) & 3u) ||
      K / 128 > 65535 || C / 128 > 65535 || ng > 65535)
    return MOK_ERR_INVALID_ARG;
  mok_status s = mok_check_device();
  if (s != MOK_OK) return s;
  if (ng == 0) return MOK_OK;
  return launch_nv_quant_2d(in, ng, K, C, g, nullptr, nullptr, codes, scales,
                            static_cast<cudaStream_t>(stream), false) == cudaSuccess
             ? MOK_OK
             : MOK_ERR_CUDA;
}

extern "C" mok_status mok_gemm_nvfp4(int64_t M, int64_t N, int64_t K, const uint8_t* A,
                                     const uint8_t* A_scales, const float* A_g, const uint8_t* B,
                                     const uint8_t* B_scales, const float* B_g, float* C,
                                     void* workspace, size_t ws_bytes, void* stream) {
  if (!A || !A_scales || !A_g || !B || !B_scales || !B_g || !C || !workspace)
    return MOK_ERR_INVALID_ARG;
  if (ws_bytes < 256) return MOK_ERR_WORKSPACE;
  if (M <= 0 || N <= 0 || K <= 0 || M % kNvTile || N % kNvTile || K % 256)
    return MOK_ERR_UNSUPPORTED;
  if (M > (1 << 24) || N > (1 << 24) || K > (1 << 20)) return MOK_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(A) & 15u) || (reinterpret_cast<uintptr_t>(B) & 15u) ||
      (reinterpret_cast<uintptr_t>(A_scales) & 3u) || (reinterpret_cast<uintptr_t>(B_scales) & 3u) ||
      (reinterpret_cast<uintptr_t>(C) & 15u))
    return MOK_ERR_INVALID_ARG;
  mok_status s = mok_check_device();
  if (s != MOK_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* status = static_cast<int*>(workspace);
  if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return MOK_ERR_CUDA;
  CUtensorMap ta, tb;
  const auto u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  // codes: [rows, K/2] bytes, 128-byte boxes of 128 rows
  if (!make_tensor_map_2d(&ta, u8, 1, A, K / 2, M, K / 2, kNvBK, kNvTile, sw) ||
      !make_tensor_map_2d(&tb, u8, 1, B, K / 2, N, K / 2, kNvBK, kNvTile, sw))
    return MOK_ERR_INVALID_ARG;
  if (cudaFuncSetAttribute(nv_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kNvSmem) != cudaSuccess)
    return MOK_ERR_CUDA;
  dim3 grid(static_cast<unsigned>(N / kNvTile), static_cast<unsigned>(M / kNvTile));
  ProfScope prof("gemm_nvfp4", st);
  nv_gemm_kernel<<<grid, kNvThreads, kNvSmem, st>>>(ta, tb, A_scales, B_scales, A_g, B_g, C,
                                                    static_cast<int>(N), static_cast<int>(K),
                                                    status);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? MOK_OK : MOK_ERR_CUDA;
}
