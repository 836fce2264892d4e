// Dense MXFP8 GEMM on the block-scaled tensor cores:
//   C[M,N] (fp32) = sum_k A[m,k] 2^sa[m,k/32] * B[n,k] 2^sb[n,k/32]
// with A, B E4M3 codes (K contiguous) and sa, sb E8M0 scale bytes (value
// 2^(byte-127)), one per 32 consecutive K values, as mok_mx_quantize writes
// them.  One CTA per 128 x 128 tile of C:
//   warp 0      producer: TMA loads of the A and B code tiles (128 rows x 128
//               K bytes, 128-byte swizzle) and the gather of their scale bytes
//               into the 512-byte block the scale copy takes (row r, K block j
//               of a 128-row tile at byte 16*(r%32) + 4*(r/32) + j);
//   warp 1      MMA: per 128-K stage, tcgen05.cp of both scale blocks to TMEM
//               (32x128b, replicated to the four lane quarters) and four
//               tcgen05.mma.kind::mxf8f6f4.block_scale (K = 32 each, the scale
//               byte of K block j selected by the descriptor's scale ids);
//   warps 2..5  epilogue: TMEM -> registers -> fp32 C.
// Source: [dothoosh] "Cursor Mixture-of-Kittens cuts MoE training latency by
// 5.8x", "MoK technical details", bullet "Precision and scheduling" (MXFP8
// expert GEMMs); the scale rule is the OCP Microscaling v1.0 one (mx.cuh).
#include <cuda.h>
#include <cuda_runtime.h>

#include "mok_internal.h"
#include "ptx.cuh"

namespace mok {
namespace {

constexpr int kMxStages = 4;
constexpr int kMxTile = 128;               // M = N = 128
constexpr int kMxBK = 128;                 // K values (bytes) per stage
constexpr int kCodeBytes = kMxTile * kMxBK;  // 16 KB per operand tile
constexpr int kSfBytes = 512;              // 128 rows x 4 scale bytes
constexpr int kMxStageBytes = 2 * kCodeBytes + 2 * kSfBytes;
constexpr int kMxThreads = 192;
// TMEM: accumulator columns [0,128); stage s keeps A scales at 128 + 8s and
// B scales at 132 + 8s (four columns each)
constexpr uint32_t kMxTmemCols = 256;
constexpr int kMxSmem = 1024 + kMxStages * kMxStageBytes + 256;

__global__ void __launch_bounds__(kMxThreads, 1)
    mx_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const uint8_t* __restrict__ sa, const uint8_t* __restrict__ sb, float* C,
                   int N, int K, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kMxStages * kMxStageBytes);
  uint64_t* empty = full + kMxStages;
  uint64_t* tfull = empty + kMxStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tfull + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tile = blockIdx.x, m_tile = blockIdx.y;
  const int nkb = K / kMxBK;
  const long long ks = K / 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMxStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kMxTmemCols);
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
      const int s = kb % kMxStages;
      const uint32_t par = static_cast<uint32_t>((kb / kMxStages) & 1);
      if (!mbar_wait(&empty[s], par ^ 1u, vabort)) {
        ok = false;
        break;
      }
      uint8_t* st = smem + s * kMxStageBytes;
      gather_sf(st + 2 * kCodeBytes, sa, ks, (long long)m_tile * kMxTile, (long long)kb * 4, lane);
      gather_sf(st + 2 * kCodeBytes + kSfBytes, sb, ks, (long long)n_tile * kMxTile,
                (long long)kb * 4, lane);
      fence_proxy_async_smem();  // the scale copy reads these bytes through the async proxy
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(&full[s], 2 * kCodeBytes);
        tma_load_2d(st, &tmA, &full[s], kb * kMxBK, m_tile * kMxTile);
        tma_load_2d(st + kCodeBytes, &tmB, &full[s], kb * kMxBK, n_tile * kMxTile);
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
        const int s = kb % kMxStages;
        const uint32_t par = static_cast<uint32_t>((kb / kMxStages) & 1);
        if (!mbar_wait(&full[s], par, vabort)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t a_base = smem_addr(smem + s * kMxStageBytes);
        const uint32_t b_base = a_base + kCodeBytes;
        const uint32_t sfa_col = tmem_base + 128u + 8u * s;
        const uint32_t sfb_col = sfa_col + 4u;
        tmem_cp_sf(sfa_col, smem_desc_sf(a_base + 2 * kCodeBytes));
        tmem_cp_sf(sfb_col, smem_desc_sf(a_base + 2 * kCodeBytes + kSfBytes));
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint64_t ad = smem_desc_sw128(a_base + j * 32, 16, 1024);
          const uint64_t bd = smem_desc_sw128(b_base + j * 32, 16, 1024);
          mma_mxf8(tmem_base, ad, bd, idesc_mxf8(kMxTile, kMxTile, static_cast<uint32_t>(j)),
                   sfa_col, sfb_col, (kb | j) != 0 ? 1u : 0u);
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
    const long long row = (long long)m_tile * kMxTile + q * 32 + lane;
    float* out = C + row * N + (long long)n_tile * kMxTile;
#pragma unroll 1
    for (int c = 0; c < kMxTile; c += 16) {
      uint32_t r[16];
      tmem_ld16(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + c, r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; j += 4)
        *reinterpret_cast<float4*>(out + c + j) =
            make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                        __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kMxTmemCols);
  }
}

}  // namespace

cudaError_t gemm_dense_mxfp8(int64_t M, int64_t N, int64_t K, const uint8_t* A,
                             const uint8_t* A_scales, const uint8_t* B, const uint8_t* B_scales,
                             float* C, int* status, cudaStream_t st) {
  CUtensorMap ta, tb;
  const auto u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  if (!make_tensor_map_2d(&ta, u8, 1, A, K, M, K, kMxBK, kMxTile, sw)) return cudaErrorInvalidValue;
  if (!make_tensor_map_2d(&tb, u8, 1, B, K, N, K, kMxBK, kMxTile, sw)) return cudaErrorInvalidValue;
  cudaError_t e =
      cudaFuncSetAttribute(mx_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMxSmem);
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(N / kMxTile), static_cast<unsigned>(M / kMxTile));
  ProfScope prof("gemm_mxfp8", st);
  mx_gemm_kernel<<<grid, kMxThreads, kMxSmem, st>>>(ta, tb, A_scales, B_scales, C,
                                                    static_cast<int>(N), static_cast<int>(K),
                                                    status);
  count_launch();
  return cudaGetLastError();
}

}  // namespace mok
