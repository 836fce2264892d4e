// MXFP8 quantisation kernels (E4M3 elements, one E8M0 scale per 32 values),
// row-wise (blocks of 32 consecutive values of a row) and column-wise (blocks
// of 32 consecutive rows of a column).  They write the dequantised bf16 values
// (exact: 4 significant bits times a power of two), and optionally the E4M3
// codes and E8M0 scale bytes.
// Source: [dothoosh] "Cursor Mixture-of-Kittens cuts MoE training latency by
// 5.8x", "MoK technical details", bullet "Precision and scheduling"; the
// rule itself is the OCP Microscaling v1.0 one (see mx.cuh).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mok_internal.h"
#include "mx.cuh"
#include "ptx.cuh"
#include "quant_tile.cuh"

namespace mok {

// Shared exponent of a block from its largest magnitude (the rule above).
__device__ __forceinline__ int mx_shared_of(float amax) {
  if (!(amax > 0.f)) return -127;
  int e;
  frexpf(amax, &e);  // amax = m * 2^e with 0.5 <= m < 1
  const int s = e - 1 - 8;
  return s < -127 ? -127 : (s > 127 ? 127 : s);
}

__device__ __forceinline__ void unpack8(const uint4& w, float (&v)[8]) {
  v[0] = bf16lo(w.x); v[1] = bf16hi(w.x); v[2] = bf16lo(w.y); v[3] = bf16hi(w.y);
  v[4] = bf16lo(w.z); v[5] = bf16hi(w.z); v[6] = bf16lo(w.w); v[7] = bf16hi(w.w);
}

__device__ __forceinline__ float amax8(const float (&v)[8]) {
  float m = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(v[j]));
  return m;
}

// Quantises 8 values, value j with the factors down[j] = 2^-shared_j and
// up[j] = 2^shared_j: CODES gives the E4M3 codes (value j in byte j), DEQ the
// dequantised values q * 2^shared rounded to bf16 (exact), packed as 8 bf16.
template <bool CODES, bool DEQ>
__device__ __forceinline__ void mx_quant8(const float (&v)[8], const float (&down)[8],
                                          const float (&up)[8], uint2* codes, uint4* deq) {
  uint32_t c[4], d[4];
#pragma unroll
  for (int j = 0; j < 8; j += 2) {
    // cvt packs its first operand into the upper byte
    const uint16_t q = cvt_e4m3x2(v[j + 1] * down[j + 1], v[j] * down[j]);
    c[j / 2] = q;
    if (DEQ) {
      float hi, lo;
      e4m3x2_to_f32(q, &hi, &lo);
      d[j / 2] = pack_bf16x2(lo * up[j], hi * up[j + 1]);
    }
  }
  if (CODES) *codes = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
  if (DEQ) *deq = make_uint4(d[0], d[1], d[2], d[3]);
}

// The factors of one shared exponent for all 8 values.
__device__ __forceinline__ void uniform_factors(int s, float (&down)[8], float (&up)[8]) {
  const float dn = exp2i(-s), u = exp2i(s);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    down[j] = dn;
    up[j] = u;
  }
}

// Row blocks.  Four consecutive lanes hold one block of 32 values (8 each, one
// 16-byte load), so a warp reads 512 contiguous bytes; the block maximum is
// two shuffles.  Each lane keeps kRowUnroll independent chunks in flight.
// The loop runs per warp (every lane takes the same trips) and nchunks is a
// multiple of 4, so a block's four lanes are all in range or all out.
// tiled_nkg > 0: scales in the tiled layout of a matrix with tiled_nkg*128
// columns (mx_tiled_off); 0: row-major [rows, cols/32].
// Optional source-row map of the quantisers: output row r takes input row
// map[r] when that is a row of the input (0 <= map[r] < T), zeros otherwise
// (the layer's dispatched rows: output row = padded row, input = token rows).
struct RowMap {
  const int32_t* map;  // NULL: output row r is input row r
  int T;
  // NULL, or the number of leading output rows anything reads (the plan's
  // padded row total, on the device): rows past it are left unwritten
  const int32_t* nrows;
};

constexpr int kRowUnroll = 4;
template <bool CODES, bool OUT>
__global__ void __launch_bounds__(256) mx_rows_kernel(const uint4* __restrict__ in,
                                                      uint4* __restrict__ out,
                                                      uint8_t* __restrict__ codes,
                                                      uint8_t* __restrict__ scales,
                                                      long long nchunks, long long tiled_nkg) {
  grid_dep_launch();  // a GEMM after this kernel may start its prologue
  const int lane = threadIdx.x & 31;
  const long long G = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i0 = static_cast<long long>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31);
       i0 < nchunks; i0 += kRowUnroll * G) {
    uint4 w[kRowUnroll];
#pragma unroll
    for (int u = 0; u < kRowUnroll; ++u) {
      const long long c = i0 + lane + u * G;
      w[u] = c < nchunks ? ld_global_nc_v4(in + c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kRowUnroll; ++u) {
      const long long c = i0 + lane + u * G;
      float v[8];
      unpack8(w[u], v);
      float m = amax8(v);
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
      if (c >= nchunks) continue;
      const int s = mx_shared_of(m);
      float down[8], up[8];
      uniform_factors(s, down, up);
      uint2 q;
      uint4 deq;
      mx_quant8<CODES, OUT>(v, down, up, &q, &deq);
      if (CODES) reinterpret_cast<uint2*>(codes)[c] = q;
      if (OUT) out[c] = deq;
      if (scales && (lane & 3) == 0) {
        // block index below 2^32 (checked by the launcher): 32-bit division
        const uint32_t b = static_cast<uint32_t>(c >> 2);
        const uint32_t bpr = static_cast<uint32_t>(tiled_nkg) * 4;  // blocks per row
        const long long off = tiled_nkg > 0 ? mx_tiled_off(b / bpr, b % bpr, tiled_nkg) : b;
        scales[off] = static_cast<uint8_t>(s + 127);
      }
    }
  }
}

// Row blocks of rows taken through a row map (output row r quantises input row
// map[r], zeros when that is not a row of the input): one warp per output
// row, the map read once per row (the warp's next row's entry is read while
// this row is processed); the lanes walk the row in 16-byte chunks, kMapUnroll
// in flight per lane, four lanes per 32-value block as in mx_rows_kernel.
// c8 % 4 == 0.
constexpr int kMapUnroll = 8;
template <bool CODES, bool OUT>
__global__ void __launch_bounds__(256) mx_rows_map_kernel(const uint4* __restrict__ in,
                                                          uint4* __restrict__ out,
                                                          uint8_t* __restrict__ codes,
                                                          uint8_t* __restrict__ scales,
                                                          long long rows, uint32_t c8,
                                                          long long tiled_nkg, RowMap rm) {
  grid_dep_launch();  // a GEMM after this kernel may start its prologue
  if (rm.nrows) {
    const long long lim = *rm.nrows;
    rows = lim < rows ? lim : rows;
  }
  const int lane = threadIdx.x & 31;
  const long long nw = static_cast<long long>(gridDim.x) * (blockDim.x / 32);
  long long r = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
  int t_next = r < rows ? rm.map[r] : -1;
  for (; r < rows; r += nw) {
    const int t = t_next;
    if (r + nw < rows) t_next = rm.map[r + nw];
    const bool src_ok = t >= 0 && t < rm.T;
    const uint4* src = in + static_cast<long long>(src_ok ? t : 0) * c8;
    for (uint32_t j0 = 0; j0 < c8; j0 += 32 * kMapUnroll) {  // the same trips for every lane
      uint4 w[kMapUnroll];
#pragma unroll
      for (int u = 0; u < kMapUnroll; ++u) {
        const uint32_t j = j0 + u * 32 + lane;
        w[u] = (src_ok && j < c8) ? ld_global_nc_v4(src + j) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kMapUnroll; ++u) {
        const uint32_t j = j0 + u * 32 + lane;
        float v[8];
        unpack8(w[u], v);
        float m = amax8(v);
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        if (j >= c8) continue;
        const int s = mx_shared_of(m);
        float down[8], up[8];
        uniform_factors(s, down, up);
        uint2 q;
        uint4 deq;
        mx_quant8<CODES, OUT>(v, down, up, &q, &deq);
        const long long c = r * c8 + j;  // output chunk
        if (CODES) reinterpret_cast<uint2*>(codes)[c] = q;
        if (OUT) out[c] = deq;
        if (scales && (lane & 3) == 0) {
          const long long off = tiled_nkg > 0 ? mx_tiled_off(r, j >> 2, tiled_nkg) : (c >> 2);
          scales[off] = static_cast<uint8_t>(s + 127);
        }
      }
    }
  }
}

// Column blocks, one 32-row x 256-column tile per CTA trip (256 threads).
// Warp w loads rows w, w+8, w+16, w+24 of the tile and lane l columns
// 8l..8l+7 (16-byte loads, 512 contiguous bytes per warp and row).  The 32-row
// column maxima meet in shared memory; each thread then quantises its own 32
// values with its 8 columns' exponents.  ROWS_OUT (cols % 32 == 0): the same
// tile is also quantised in row blocks (four lanes per block, as in
// mx_rows_kernel) into rows_out, so both layouts cost one read.
template <bool CODES, bool OUT, bool ROWS_OUT>
__global__ void __launch_bounds__(256, ROWS_OUT ? 3 : 4) mx_cols_kernel(const uint4* __restrict__ in,
                                                         uint4* __restrict__ out,
                                                         uint8_t* __restrict__ codes,
                                                         uint8_t* __restrict__ scales,
                                                         uint4* __restrict__ rows_out,
                                                         long long row_blocks, long long cols,
                                                         RowMap rm) {
  grid_dep_launch();  // a GEMM after this kernel may start its prologue
  __shared__ __align__(16) float s_part[8][256];
  __shared__ __align__(16) int s_exp[256];
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const long long c8 = cols / 8;  // 16-byte chunks per row
  if (rm.nrows) {
    const long long lim = (static_cast<long long>(*rm.nrows) + 31) / 32;
    row_blocks = lim < row_blocks ? lim : row_blocks;
  }
  // tile counts below 2^31 (checked by the launcher): 32-bit division
  const uint32_t tiles_c = static_cast<uint32_t>((cols + 255) / 256);
  const uint32_t ntiles = static_cast<uint32_t>(row_blocks) * tiles_c;
  // this thread's four chunks of tile t (zeros outside the input)
  auto load_tile = [&](uint32_t t, uint4 (&x)[4]) {
    const long long rb = t / tiles_c, tc = t - static_cast<uint32_t>(rb) * tiles_c;
    const long long ch = tc * 32 + l;
    const bool ok = ch < c8;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      long long src = rb * 32 + w + 8 * r;
      if (rm.map) {
        const int t = rm.map[src];
        src = (t >= 0 && t < rm.T) ? t : -1;
      }
      x[r] = (ok && src >= 0) ? ld_global_nc_v4(in + src * c8 + ch) : make_uint4(0, 0, 0, 0);
    }
  };
  // the next trip's loads (and their row-map reads) are in flight while this
  // trip is reduced and quantised
  uint4 xn[4];
  if (blockIdx.x < ntiles) load_tile(blockIdx.x, xn);
  for (uint32_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const long long rb = t / tiles_c, tc = t - static_cast<uint32_t>(rb) * tiles_c;
    const long long ch = tc * 32 + l;  // this lane's chunk of each row
    const bool ok = ch < c8;
    uint4 x[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) x[r] = xn[r];
    if (t + gridDim.x < ntiles) load_tile(t + gridDim.x, xn);
    float part[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      float v[8];
      unpack8(x[r], v);
#pragma unroll
      for (int j = 0; j < 8; ++j) part[j] = fmaxf(part[j], fabsf(v[j]));
    }
    reinterpret_cast<float4*>(&s_part[w][8 * l])[0] = make_float4(part[0], part[1], part[2], part[3]);
    reinterpret_cast<float4*>(&s_part[w][8 * l])[1] = make_float4(part[4], part[5], part[6], part[7]);
    __syncthreads();
    {
      float m = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) m = fmaxf(m, s_part[k][threadIdx.x]);
      const int s = mx_shared_of(m);
      s_exp[threadIdx.x] = s;
      const long long col = tc * 256 + threadIdx.x;
      if (scales && col < cols) scales[rb * cols + col] = static_cast<uint8_t>(s + 127);
    }
    __syncthreads();
    if (ok && (CODES || OUT)) {
      const int4 e0 = reinterpret_cast<const int4*>(&s_exp[8 * l])[0];
      const int4 e1 = reinterpret_cast<const int4*>(&s_exp[8 * l])[1];
      const int sh[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
      float down[8], up[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        down[j] = exp2i(-sh[j]);
        up[j] = exp2i(sh[j]);
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const long long idx = (rb * 32 + w + 8 * r) * c8 + ch;
        float v[8];
        unpack8(x[r], v);
        uint2 q;
        uint4 deq;
        mx_quant8<CODES, OUT>(v, down, up, &q, &deq);
        if (CODES) reinterpret_cast<uint2*>(codes)[idx] = q;
        if (OUT) out[idx] = deq;
      }
    }
    if (ROWS_OUT) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        float v[8];
        unpack8(x[r], v);
        float m = amax8(v);
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        if (!ok) continue;
        float down[8], up[8];
        uniform_factors(mx_shared_of(m), down, up);
        uint2 q;
        uint4 deq;
        mx_quant8<false, true>(v, down, up, &q, &deq);
        rows_out[(rb * 32 + w + 8 * r) * c8 + ch] = deq;
      }
    }
  }
}

// A weight [ng*K, C] (ng stacked [K, C] matrices) in both block directions
// from one read: the rows (blocks of 32 along C) as E4M3 codes [ng*K, C] with
// tiled scales (C/128 K groups), and the columns (blocks of 32 along K)
// either as codes written transposed, [ng*C, K] (row g*C + c holds column c
// of matrix g) with tiled scales (K/128 K groups), or as dequantised bf16
// values in the input's layout.  Persistent CTAs walk the 128 x 128 tiles
// (quant_tile.cuh).  Warps 0-3 take the rows, one row per thread (128
// contiguous code bytes); warps 4-7 the columns, a pair of adjacent columns
// and half of the tile's K per thread, read as 4-byte pairs (one 128-byte run
// per warp and row).  Column codes leave as 64-byte runs per column, column
// values as 4-byte pairs (again one 128-byte run per warp and row).

// MX encoding (mx_encode32's rule) of the 32 values held in the low (HI =
// false) or high halves of 32 packed bf16 pairs.
template <bool HI>
__device__ __forceinline__ uint32_t mx_encode_half32(const uint32_t (&x)[32], uint32_t (&w)[8]) {
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(HI ? bf16hi(x[j]) : bf16lo(x[j])));
  const int sh = mx_shared_of(amax);
  const float down = exp2i(-sh);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    // cvt packs its first operand into the upper byte
    const uint32_t p01 = cvt_e4m3x2((HI ? bf16hi(x[4 * i + 1]) : bf16lo(x[4 * i + 1])) * down,
                                    (HI ? bf16hi(x[4 * i]) : bf16lo(x[4 * i])) * down);
    const uint32_t p23 = cvt_e4m3x2((HI ? bf16hi(x[4 * i + 3]) : bf16lo(x[4 * i + 3])) * down,
                                    (HI ? bf16hi(x[4 * i + 2]) : bf16lo(x[4 * i + 2])) * down);
    w[i] = p01 | (p23 << 16);
  }
  return static_cast<uint32_t>(sh + 127);
}

// MX fake quantisation (mx_fake32's rule, rounded to bf16 as mx_quant8 does)
// of the 32 values in one half of 32 packed bf16 pairs, in place.
template <bool HI>
__device__ __forceinline__ void mx_fake_half32(uint32_t (&x)[32]) {
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(HI ? bf16hi(x[j]) : bf16lo(x[j])));
  const int sh = mx_shared_of(amax);
  const float down = exp2i(-sh), up = exp2i(sh);
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    const uint16_t qv = cvt_e4m3x2((HI ? bf16hi(x[j + 1]) : bf16lo(x[j + 1])) * down,
                                   (HI ? bf16hi(x[j]) : bf16lo(x[j])) * down);
    float fh, fl;
    e4m3x2_to_f32(qv, &fh, &fl);
    const uint32_t b0 = __bfloat16_as_ushort(__float2bfloat16_rn(fl * up));
    const uint32_t b1 = __bfloat16_as_ushort(__float2bfloat16_rn(fh * up));
    x[j] = HI ? ((x[j] & 0xFFFFu) | (b0 << 16)) : ((x[j] & 0xFFFF0000u) | b0);
    x[j + 1] = HI ? ((x[j + 1] & 0xFFFFu) | (b1 << 16)) : ((x[j + 1] & 0xFFFF0000u) | b1);
  }
}

__global__ void __launch_bounds__(256, 3)
    mx_quant_2d_kernel(const uint16_t* __restrict__ in, int K, int C, int ng,
                       uint8_t* __restrict__ rcodes, uint8_t* __restrict__ rscales,
                       uint8_t* __restrict__ ccodes, uint8_t* __restrict__ cscales,
                       uint16_t* __restrict__ cvals) {
  extern __shared__ __align__(16) uint16_t qt_smem[];
  const int t = threadIdx.x;
  qt_walk(in, K, C, ng, qt_smem, [&](uint16_t* tile, const QtTile& q) {
    const long long row0 = static_cast<long long>(q.grp) * K + q.kt * 128;
    if (t < 128) {
      // row t: four blocks along C
      const long long row = row0 + t;
      uint4* cp = reinterpret_cast<uint4*>(rcodes + row * C + q.ct * 128);
      uint32_t sc = 0u;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        float v[32];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float u[8];
          unpack8(*reinterpret_cast<const uint4*>(tile + t * kQtPitch + 32 * b + 8 * c), u);
#pragma unroll
          for (int j = 0; j < 8; ++j) v[8 * c + j] = u[j];
        }
        uint32_t cw[8];
        sc |= mx_encode32(v, cw) << (8 * b);
        cp[2 * b] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
        cp[2 * b + 1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
      }
      *reinterpret_cast<uint32_t*>(rscales + mx_tiled_off(row, q.ct * 4, C / 128)) = sc;
    } else {
      // columns 2p, 2p+1, K rows 64 h .. 64 h + 63: two blocks each
      const int p = t & 63, h = (t - 128) >> 6;
      const long long orow = static_cast<long long>(q.grp) * C + q.ct * 128 + 2 * p;
      uint32_t s0 = 0u, s1 = 0u;
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const int k0 = 64 * h + 32 * b;
        uint32_t x[32];
#pragma unroll
        for (int j = 0; j < 32; ++j)
          x[j] = *reinterpret_cast<const uint32_t*>(tile + (k0 + j) * kQtPitch + 2 * p);
        if (ccodes) {
          uint32_t cw[8];
          s0 |= mx_encode_half32<false>(x, cw) << (8 * b);
          uint4* c0 = reinterpret_cast<uint4*>(ccodes + orow * K + q.kt * 128 + k0);
          c0[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
          c0[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
          s1 |= mx_encode_half32<true>(x, cw) << (8 * b);
          uint4* c1 = reinterpret_cast<uint4*>(ccodes + (orow + 1) * K + q.kt * 128 + k0);
          c1[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
          c1[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
        } else {
          mx_fake_half32<false>(x);
          mx_fake_half32<true>(x);
          uint16_t* dst = cvals + (row0 + k0) * C + q.ct * 128 + 2 * p;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            *reinterpret_cast<uint32_t*>(dst + static_cast<long long>(j) * C) = x[j];
        }
      }
      if (ccodes) {
        *reinterpret_cast<uint16_t*>(cscales + mx_tiled_off(orow, q.kt * 4 + 2 * h, K / 128)) =
            static_cast<uint16_t>(s0);
        *reinterpret_cast<uint16_t*>(cscales +
                                     mx_tiled_off(orow + 1, q.kt * 4 + 2 * h, K / 128)) =
            static_cast<uint16_t>(s1);
      }
    }
  });
}

static unsigned grid_for(long long n, int threads) {
  long long g = (n + threads - 1) / threads;
  const long long cap = static_cast<long long>(num_sms_current_device()) * 8;
  if (g > cap) g = cap;
  return static_cast<unsigned>(g < 1 ? 1 : g);
}

cudaError_t launch_mx_rows(const void* in, void* out, long long rows, long long cols,
                           uint8_t* codes, uint8_t* scales, cudaStream_t st, bool tiled,
                           const int32_t* rowmap, int T, const int32_t* rows_dev) {
  if (cols % 32) return cudaErrorInvalidValue;
  if (tiled && (rows % 128 || cols % 128)) return cudaErrorInvalidValue;
  const long long nchunks = rows * (cols / 8);
  if (nchunks == 0) return cudaSuccess;
  if (nchunks / 4 >= (1LL << 32)) return cudaErrorInvalidValue;  // 32-bit block index
  if (rows_dev && !rowmap) return cudaErrorInvalidValue;  // (the row-map kernel honours it)
  const RowMap rm{rowmap, T, rows_dev};
  const uint32_t c8 = static_cast<uint32_t>(cols / 8);
  ProfScope prof("mx_quant_rows", st);
  const uint4* i4 = static_cast<const uint4*>(in);
  uint4* o4 = static_cast<uint4*>(out);
  const long long nkg = tiled ? cols / 128 : 0;
  if (rowmap) {  // one warp per output row
    const long long cap = static_cast<long long>(num_sms_current_device()) * 8;
    const long long need = (rows + 7) / 8;
    const unsigned g = static_cast<unsigned>(need < cap ? need : cap);
    if (codes && out)
      mx_rows_map_kernel<true, true><<<g, 256, 0, st>>>(i4, o4, codes, scales, rows, c8, nkg, rm);
    else if (codes)
      mx_rows_map_kernel<true, false><<<g, 256, 0, st>>>(i4, o4, codes, scales, rows, c8, nkg, rm);
    else if (out)
      mx_rows_map_kernel<false, true><<<g, 256, 0, st>>>(i4, o4, codes, scales, rows, c8, nkg, rm);
    else
      mx_rows_map_kernel<false, false><<<g, 256, 0, st>>>(i4, o4, codes, scales, rows, c8, nkg,
                                                          rm);
    count_launch();
    return cudaGetLastError();
  }
  const unsigned grid = grid_for((nchunks + kRowUnroll - 1) / kRowUnroll, 256);
  if (codes && out)
    mx_rows_kernel<true, true><<<grid, 256, 0, st>>>(i4, o4, codes, scales, nchunks, nkg);
  else if (codes)
    mx_rows_kernel<true, false><<<grid, 256, 0, st>>>(i4, o4, codes, scales, nchunks, nkg);
  else if (out)
    mx_rows_kernel<false, true><<<grid, 256, 0, st>>>(i4, o4, codes, scales, nchunks, nkg);
  else
    mx_rows_kernel<false, false><<<grid, 256, 0, st>>>(i4, o4, codes, scales, nchunks, nkg);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_mx_cols(const void* in, void* out, long long rows, long long cols,
                           uint8_t* codes, uint8_t* scales, cudaStream_t st, void* rows_out,
                           const int32_t* rowmap, int T, const int32_t* rows_dev) {
  const RowMap rm{rowmap, T, rows_dev};
  if (rows % 32 || cols % 8 || (rows_out && (cols % 32 || !out || codes)))
    return cudaErrorInvalidValue;
  const long long ntiles = (rows / 32) * ((cols + 255) / 256);
  if (ntiles == 0) return cudaSuccess;
  if (ntiles >= (1LL << 31)) return cudaErrorInvalidValue;
  ProfScope prof("mx_quant_cols", st);
  const long long cap = static_cast<long long>(num_sms_current_device()) * 8;
  const unsigned grid = static_cast<unsigned>(ntiles < cap ? ntiles : cap);
  const uint4* i4 = static_cast<const uint4*>(in);
  uint4* o4 = static_cast<uint4*>(out);
  uint4* r4 = static_cast<uint4*>(rows_out);
  const long long rb = rows / 32;
  if (rows_out)  // the layer's dy: bf16 values in both directions
    mx_cols_kernel<false, true, true><<<grid, 256, 0, st>>>(i4, o4, codes, scales, r4, rb, cols, rm);
  else if (codes && out)
    mx_cols_kernel<true, true, false><<<grid, 256, 0, st>>>(i4, o4, codes, scales, r4, rb, cols, rm);
  else if (codes)
    mx_cols_kernel<true, false, false><<<grid, 256, 0, st>>>(i4, o4, codes, scales, r4, rb, cols, rm);
  else if (out)
    mx_cols_kernel<false, true, false><<<grid, 256, 0, st>>>(i4, o4, codes, scales, r4, rb, cols, rm);
  else
    mx_cols_kernel<false, false, false><<<grid, 256, 0, st>>>(i4, o4, codes, scales, r4, rb, cols, rm);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_mx_quant_2d(const void* in, long long ng, long long K, long long C,
                               uint8_t* rcodes, uint8_t* rscales, uint8_t* ccodes,
                               uint8_t* cscales, void* cvals, cudaStream_t st) {
  if (K % 128 || C % 128 || ng <= 0 || K / 128 > 65535 || C / 128 > 65535 || ng > 65535)
    return cudaErrorInvalidValue;
  if (!rcodes || !rscales || (!ccodes == !cvals) || (ccodes && !cscales))
    return cudaErrorInvalidValue;
  if ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(rcodes) |
       reinterpret_cast<uintptr_t>(ccodes) | reinterpret_cast<uintptr_t>(cvals)) & 15u ||
      (reinterpret_cast<uintptr_t>(rscales) | reinterpret_cast<uintptr_t>(cscales)) & 1u)
    return cudaErrorInvalidValue;
  ProfScope prof("mx_quant_2d", st);
  const cudaError_t e = cudaFuncSetAttribute(  // the two staging buffers
      mx_quant_2d_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kQtSmemBytes);
  if (e != cudaSuccess) return e;
  const long long ntiles = ng * (K / 128) * (C / 128);
  if (ntiles >= (1LL << 31)) return cudaErrorInvalidValue;
  const long long cap = static_cast<long long>(num_sms_current_device()) * 3;
  mx_quant_2d_kernel<<<static_cast<unsigned>(ntiles < cap ? ntiles : cap), 256, kQtSmemBytes,
                       st>>>(static_cast<const uint16_t*>(in), static_cast<int>(K),
                             static_cast<int>(C), static_cast<int>(ng), rcodes, rscales, ccodes,
                             cscales, static_cast<uint16_t*>(cvals));
  count_launch();
  return cudaGetLastError();
}

}  // namespace mok

using namespace mok;

extern "C" mok_status mok_mx_quantize(const void* in, int64_t rows, int64_t cols, int along_rows,
                                      void* out, uint8_t* codes, uint8_t* scales, void* stream) {
  if (rows < 0 || cols < 0 || (rows * cols > 0 && (!in || !out))) return MOK_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out) |
       reinterpret_cast<uintptr_t>(codes)) & 15u)
    return MOK_ERR_INVALID_ARG;
  if (along_rows ? (rows % 32 || cols % 8) : (cols % 32)) return MOK_ERR_UNSUPPORTED;
  const mok_status s = mok_check_device();
  if (s != MOK_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const cudaError_t e = along_rows ? launch_mx_cols(in, out, rows, cols, codes, scales, st)
                                   : launch_mx_rows(in, out, rows, cols, codes, scales, st);
  return e == cudaSuccess ? MOK_OK : MOK_ERR_CUDA;
}
