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

// ------------------------------------------------------------- CTA pairs --
// 256 x 256 tiles on a cluster of two CTAs (tcgen05.mma.cta_group::2, M=256):
// CTA r stages its A rows m0 + 128r.. and B rows n0 + 128r.. of the tile, the
// scales of its own 128 A rows and of all 256 B rows; the leader copies the
// scale blocks to TMEM (each CTA's from its own shared memory) and issues the
// MMAs; each CTA's TMEM holds its 128 rows of the 256 accumulator columns.
constexpr int kPStages = 4;
constexpr int kPSfaOff = 2 * kCodeBytes;              // own A rows
constexpr int kPSfbOff = kPSfaOff + kSfBytes;         // B rows 0..127, then 128..255
constexpr int kPStageBytes = 35 * 1024;               // 2*16 KB + 1.5 KB, 1 KB aligned
constexpr int kPSmem = 1024 + kPStages * kPStageBytes + 256;
constexpr uint32_t kPTmemCols = 512;                  // 256 accumulator + 12 per stage

__global__ void __launch_bounds__(kMxThreads, 1)
    mx_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const uint8_t* __restrict__ sa,
                        const uint8_t* __restrict__ sb, float* C, int N, int K, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kPStages * kPStageBytes);
  uint64_t* empty = full + kPStages;
  uint64_t* tfull = empty + kPStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tfull + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_ctarank());
  const bool leader = rank == 0;
  const int n_tile = blockIdx.x >> 1, m_tile = blockIdx.y;
  const long long a_row0 = (long long)m_tile * 256 + rank * 128;
  const long long b_row0 = (long long)n_tile * 256;
  const int nkb = K / kMxBK;
  const long long ks = K / 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(&full[s], 2);  // the leader's armed arrival and the peer's scales-ready one
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kPTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  cluster_sync();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  volatile int* vabort = abort_flag;

  if (warp == 0) {
    // ---------------------------------------------------------- producer --
    const uint32_t full0 = mapa_shared(smem_addr(full), 0);
    bool ok = true;
    for (int kb = 0; kb < nkb && ok; ++kb) {
      const int s = kb % kPStages;
      const uint32_t par = static_cast<uint32_t>((kb / kPStages) & 1);
      if (!mbar_wait_cluster(&empty[s], par ^ 1u, vabort)) {
        ok = false;
        break;
      }
      uint8_t* st = smem + s * kPStageBytes;
      gather_sf(st + kPSfaOff, sa, ks, a_row0, (long long)kb * 4, lane);
      gather_sf(st + kPSfbOff, sb, ks, b_row0, (long long)kb * 4, lane);
      gather_sf(st + kPSfbOff + kSfBytes, sb, ks, b_row0 + 128, (long long)kb * 4, lane);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const uint32_t bar = full0 + 8u * s;
        if (leader) mbar_arrive_expect_tx(&full[s], 4 * kCodeBytes);
        tma_load_2d_pair(st, &tmA, bar, kb * kMxBK, static_cast<int>(a_row0));
        tma_load_2d_pair(st + kCodeBytes, &tmB, bar, kb * kMxBK,
                         static_cast<int>(b_row0 + rank * 128));
        if (!leader) mbar_arrive_cluster(bar);  // this CTA's scale blocks are written
      }
    }
    if (!ok && lane == 0) {
      *vabort = 1;
      set_status(status, MOK_ERR_DEVICE_TIMEOUT);
      spin_ns(1000000ull);
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // --------------------------------------------------------------- MMA --
      bool ok = true;
      for (int kb = 0; kb < nkb && ok; ++kb) {
        const int s = kb % kPStages;
        const uint32_t par = static_cast<uint32_t>((kb / kPStages) & 1);
        if (!mbar_wait_cluster(&full[s], par, vabort)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t a_base = smem_addr(smem + s * kPStageBytes);
        const uint32_t b_base = a_base + kCodeBytes;
        const uint32_t sfa = tmem_base + 256u + 12u * s;
        const uint32_t sfb = sfa + 4u;
        tmem_cp_sf_pair(sfa, smem_desc_sf(a_base + kPSfaOff));
        tmem_cp_sf_pair(sfb, smem_desc_sf(a_base + kPSfbOff));
        tmem_cp_sf_pair(sfb + 4u, smem_desc_sf(a_base + kPSfbOff + kSfBytes));
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint64_t ad = smem_desc_sw128(a_base + j * 32, 16, 1024);
          const uint64_t bd = smem_desc_sw128(b_base + j * 32, 16, 1024);
          mma_mxf8_pair(tmem_base, ad, bd, idesc_mxf8(256, 256, static_cast<uint32_t>(j)), sfa,
                        sfb, (kb | j) != 0 ? 1u : 0u);
        }
        mma_commit_pair(&empty[s]);
      }
      if (!ok) {
        *vabort = 1;
        set_status(status, MOK_ERR_DEVICE_TIMEOUT);
      }
      mma_commit_pair(tfull);  // on failure too, so that the epilogues leave
    }
  } else {
    // ---------------------------------------------------------- epilogue --
    const int q = warp & 3;
    const int zero = 0;
    if (!mbar_wait_cluster(tfull, 0, &zero)) set_status(status, MOK_ERR_DEVICE_TIMEOUT);
    tc_fence_after_sync();
    const long long row = a_row0 + q * 32 + lane;
    float* out = C + row * N + b_row0;
#pragma unroll 1
    for (int c = 0; c < 256; c += 16) {
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
  // the leader's MMAs read the peer's shared memory: both stay until done
  tc_fence_before_sync();
  cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, kPTmemCols);
  }
}

}  // namespace

cudaError_t gemm_dense_mxfp8(int64_t M, int64_t N, int64_t K, const uint8_t* A,
                             const uint8_t* A_scales, const uint8_t* B, const uint8_t* B_scales,
                             float* C, bool cta_pair, int* status, cudaStream_t st) {
  CUtensorMap ta, tb;
  const auto u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  if (cta_pair) {
    if (!make_tensor_map_2d(&ta, u8, 1, A, K, M, K, kMxBK, 128, sw) ||
        !make_tensor_map_2d(&tb, u8, 1, B, K, N, K, kMxBK, 128, sw))
      return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(mx_gemm_pair_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * (N / 256)), static_cast<unsigned>(M / 256), 1);
    cfg.blockDim = dim3(kMxThreads, 1, 1);
    cfg.dynamicSmemBytes = kPSmem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    ProfScope prof("gemm_mxfp8_pair", st);
    e = cudaLaunchKernelEx(&cfg, mx_gemm_pair_kernel, ta, tb, A_scales, B_scales, C,
                           static_cast<int>(N), static_cast<int>(K), status);
    count_launch();
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
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
