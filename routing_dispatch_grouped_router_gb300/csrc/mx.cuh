// MXFP8 fake-quantisation of 32 values held by one thread: E4M3 elements with
// one E8M0 (power-of-two) scale per block of 32, as in the OCP Microscaling
// v1.0 rule:
//   shared = floor(log2 max|v|) - 8   (clamped to [-127, 127]; -127 when all
//            values are zero), 8 being the exponent of the largest E4M3 normal
//   q      = v * 2^-shared rounded to nearest even on the E4M3 grid,
//            saturating at +-448
//   v'     = q * 2^shared            (exact in fp32 and in bf16)
// Source: [dothoosh] "Cursor Mixture-of-Kittens cuts MoE training latency by
// 5.8x", "MoK technical details", bullet "Precision and scheduling" (MXFP8).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace mok {

// Two fp32 -> packed E4M3x2 (round to nearest even, saturate to finite).
// The first operand lands in the upper byte.
__device__ __forceinline__ uint16_t cvt_e4m3x2(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Packed E4M3x2 -> two fp32 (exact; upper byte to `hi`).
__device__ __forceinline__ void e4m3x2_to_f32(uint16_t q, float* hi, float* lo) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(q));
  *lo = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
  *hi = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16)));
}

// 2^n as an fp32 value, for n in [-149, 127] (below -126: subnormal).  A
// product with it is exact when representable and otherwise rounds like any
// fp32 multiplication, so x * exp2i(n) equals x scaled by 2^n with one rounding.
__device__ __forceinline__ float exp2i(int n) {
  return n >= -126 ? __int_as_float((n + 127) << 23) : __int_as_float(1 << (n + 149));
}

// In-place MXFP8 fake quantisation of one 32-value block.  shared lies in
// [-127, 119] for finite input (floor(log2 of the largest finite fp32) - 8 =
// 119), so both scale factors are fp32 powers of two.
__device__ __forceinline__ void mx_fake32(float (&v)[32]) {
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
  int shared = -127;
  if (amax > 0.f) {
    int e;
    frexpf(amax, &e);  // amax = m * 2^e with 0.5 <= m < 1
    shared = e - 1 - 8;
    shared = shared < -127 ? -127 : (shared > 127 ? 127 : shared);
  }
  const float down = exp2i(-shared), up = exp2i(shared);
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    const uint16_t q = cvt_e4m3x2(v[j + 1] * down, v[j] * down);
    float hi, lo;
    e4m3x2_to_f32(q, &hi, &lo);
    v[j] = lo * up;
    v[j + 1] = hi * up;
  }
}

// Tiled layout of the E8M0 scales of a [rows, K] MXFP8 operand (rows and K
// multiples of 128), the layout the block-scaled MMA's scale copy takes: the
// scales of rows 128a..128a+127 and K blocks 4b..4b+3 (32 values each) form
// one contiguous 512-byte block (index a * (K/128) + b), in which the scale of
// row r, K block j sits at byte 16*(r%32) + 4*((r/32)%4) + j%4.
__host__ __device__ __forceinline__ long long mx_tiled_off(long long r, long long j,
                                                           long long n_kg) {
  return ((r >> 7) * n_kg + (j >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (j & 3);
}

// MXFP8 encoding of one 32-value block held by one thread: the E4M3 codes
// (same rule as mx_fake32: v' = code * 2^shared) into four 32-bit words,
// codes of v[4i..4i+3] in word i, lowest byte first; returns the E8M0 byte.
__device__ __forceinline__ uint32_t mx_encode32(const float (&v)[32], uint32_t (&w)[8]) {
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
  int shared = -127;
  if (amax > 0.f) {
    int e;
    frexpf(amax, &e);
    shared = e - 1 - 8;
    shared = shared < -127 ? -127 : (shared > 127 ? 127 : shared);
  }
  const float down = exp2i(-shared);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    // cvt packs its first operand into the upper byte
    const uint16_t p01 = cvt_e4m3x2(v[4 * i + 1] * down, v[4 * i] * down);
    const uint16_t p23 = cvt_e4m3x2(v[4 * i + 3] * down, v[4 * i + 2] * down);
    w[i] = static_cast<uint32_t>(p01) | (static_cast<uint32_t>(p23) << 16);
  }
  return static_cast<uint32_t>(shared + 127);
}

}  // namespace mok
