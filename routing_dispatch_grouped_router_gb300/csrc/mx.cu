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

namespace mok {

// E4M3 code and E8M0 scale byte of one dequantised value v' = q * 2^shared.
__device__ __forceinline__ uint8_t e4m3_code_of(float vq, int shared) {
  const uint16_t q = cvt_e4m3x2(vq * exp2i(-shared), 0.f);
  return static_cast<uint8_t>(q >> 8);
}

__device__ __forceinline__ int mx_shared_exp(const float (&v)[32]) {
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
  if (!(amax > 0.f)) return -127;
  int e;
  frexpf(amax, &e);
  const int s = e - 1 - 8;
  return s < -127 ? -127 : (s > 127 ? 127 : s);
}

// One thread per block of 32 consecutive values of a row.
// tiled_nkg > 0: scales in the tiled layout of a matrix with tiled_nkg*128
// columns (mx_tiled_off); 0: row-major [rows, cols/32].
__global__ void mx_rows_kernel(const uint4* __restrict__ in, uint4* __restrict__ out,
                               uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                               long long nblocks, long long tiled_nkg) {
  for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < nblocks;
       b += (long long)gridDim.x * blockDim.x) {
    float v[32];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 w = ld_global_nc_v4(in + b * 4 + j);
      v[8 * j + 0] = bf16lo(w.x); v[8 * j + 1] = bf16hi(w.x);
      v[8 * j + 2] = bf16lo(w.y); v[8 * j + 3] = bf16hi(w.y);
      v[8 * j + 4] = bf16lo(w.z); v[8 * j + 5] = bf16hi(w.z);
      v[8 * j + 6] = bf16lo(w.w); v[8 * j + 7] = bf16hi(w.w);
    }
    if (codes || scales) {
      uint32_t w[8];
      const uint32_t sbyte = mx_encode32(v, w);
      if (codes) {
        uint4* c = reinterpret_cast<uint4*>(codes + b * 32);
        c[0] = make_uint4(w[0], w[1], w[2], w[3]);
        c[1] = make_uint4(w[4], w[5], w[6], w[7]);
      }
      if (scales) {
        const long long off =
            tiled_nkg > 0 ? mx_tiled_off(b / (tiled_nkg * 4), b % (tiled_nkg * 4), tiled_nkg) : b;
        scales[off] = static_cast<uint8_t>(sbyte);
      }
    }
    if (out) {  // NULL: codes and scales only
      mx_fake32(v);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        out[b * 4 + j] = make_uint4(pack_bf16x2(v[8 * j], v[8 * j + 1]),
                                    pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                                    pack_bf16x2(v[8 * j + 4], v[8 * j + 5]),
                                    pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
    }
  }
}

// One thread per (32-row block, pair of adjacent columns): the two columns'
// blocks are quantised independently; loads and stores move bf16 pairs.
__global__ void mx_cols_kernel(const __nv_bfloat162* __restrict__ in,
                               __nv_bfloat162* __restrict__ out, uint8_t* __restrict__ codes,
                               uint8_t* __restrict__ scales, long long row_blocks, long long cols) {
  const long long cp = cols / 2;  // column pairs
  const long long n = row_blocks * cp;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const long long rb = i / cp, c2 = i - rb * cp;
    const long long base = rb * 32 * cp + c2;
    float v0[32], v1[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float2 f = __bfloat1622float2(in[base + j * cp]);
      v0[j] = f.x;
      v1[j] = f.y;
    }
    const int s0 = mx_shared_exp(v0), s1 = mx_shared_exp(v1);
    mx_fake32(v0);
    mx_fake32(v1);
#pragma unroll
    for (int j = 0; j < 32; ++j) out[base + j * cp] = __floats2bfloat162_rn(v0[j], v1[j]);
    const long long c = 2 * c2;
    if (codes) {
      const long long cb = rb * 32 * cols + c;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const uint16_t pair = static_cast<uint16_t>(e4m3_code_of(v0[j], s0)) |
                              (static_cast<uint16_t>(e4m3_code_of(v1[j], s1)) << 8);
        *reinterpret_cast<uint16_t*>(codes + cb + j * cols) = pair;
      }
    }
    if (scales) {
      scales[rb * cols + c] = static_cast<uint8_t>(s0 + 127);
      scales[rb * cols + c + 1] = static_cast<uint8_t>(s1 + 127);
    }
  }
}

static unsigned grid_for(long long n, int threads) {
  long long g = (n + threads - 1) / threads;
  const long long cap = static_cast<long long>(num_sms_current_device()) * 16;
  if (g > cap) g = cap;
  return static_cast<unsigned>(g < 1 ? 1 : g);
}

cudaError_t launch_mx_rows(const void* in, void* out, long long rows, long long cols,
                           uint8_t* codes, uint8_t* scales, cudaStream_t st, bool tiled) {
  if (tiled && (rows % 128 || cols % 128)) return cudaErrorInvalidValue;
  const long long nb = rows * (cols / 32);
  if (nb == 0) return cudaSuccess;
  ProfScope prof("mx_quant_rows", st);
  mx_rows_kernel<<<grid_for(nb, 256), 256, 0, st>>>(static_cast<const uint4*>(in),
                                                    static_cast<uint4*>(out), codes, scales, nb,
                                                    tiled ? cols / 128 : 0);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_mx_cols(const void* in, void* out, long long rows, long long cols,
                           uint8_t* codes, uint8_t* scales, cudaStream_t st) {
  const long long n = (rows / 32) * (cols / 2);
  if (n == 0) return cudaSuccess;
  ProfScope prof("mx_quant_cols", st);
  mx_cols_kernel<<<grid_for(n, 256), 256, 0, st>>>(static_cast<const __nv_bfloat162*>(in),
                                                   static_cast<__nv_bfloat162*>(out), codes,
                                                   scales, rows / 32, cols);
  count_launch();
  return cudaGetLastError();
}

}  // namespace mok

using namespace mok;

extern "C" mok_status mok_mx_quantize(const void* in, int64_t rows, int64_t cols, int along_rows,
                                      void* out, uint8_t* codes, uint8_t* scales, void* stream) {
  if (rows < 0 || cols < 0 || (rows * cols > 0 && (!in || !out))) return MOK_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out)) & 15u)
    return MOK_ERR_INVALID_ARG;
  if (along_rows ? (rows % 32 || cols % 2) : (cols % 32)) return MOK_ERR_UNSUPPORTED;
  const mok_status s = mok_check_device();
  if (s != MOK_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const cudaError_t e = along_rows ? launch_mx_cols(in, out, rows, cols, codes, scales, st)
                                   : launch_mx_rows(in, out, rows, cols, codes, scales, st);
  return e == cudaSuccess ? MOK_OK : MOK_ERR_CUDA;
}
