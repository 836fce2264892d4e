// Persistent walk over the 128 x 128 tiles of a stacked bf16 weight
// [ng * K, C] (ng matrices [K, C], row-major), for the quantisers that read a
// weight once for both block directions.  Each CTA (256 threads) takes tiles
// blockIdx.x, + gridDim.x, ... and stages them in shared memory through two
// buffers: while it quantises one tile the next one is already on its way
// (cp.async, 16 bytes per thread and copy, 8 copies per thread per tile).
// Rows are staged with a pitch of kQtPitch values, so that the 16-byte reads
// of eight consecutive rows by one warp quarter fall in distinct banks.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace mok {

constexpr int kQtPitch = 136;                          // bf16 values per staged row
constexpr int kQtTileBytes = 128 * kQtPitch * 2;       // one staged tile
constexpr int kQtSmemBytes = 2 * kQtTileBytes;         // two buffers

struct QtTile {
  int grp, kt, ct;  // matrix, 128-row block (along K), 128-column block (along C)
};

__device__ __forceinline__ QtTile qt_tile(int t, int nkt, int nct) {
  QtTile q;
  q.ct = t % nct;
  const int r = t / nct;
  q.kt = r % nkt;
  q.grp = r / nkt;
  return q;
}

// Issue the copies of tile `q` into `dst` and commit them as one group.
__device__ __forceinline__ void qt_issue(uint16_t* dst, const uint16_t* in, int K, int C,
                                         const QtTile& q) {
  const uint16_t* src = in + (static_cast<long long>(q.grp) * K + q.kt * 128) * C + q.ct * 128;
  const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int i = threadIdx.x + 256 * j, r = i >> 4, c8 = i & 15;
    const uint16_t* g = src + static_cast<long long>(r) * C + 8 * c8;
    const uint32_t s = base + static_cast<uint32_t>((r * kQtPitch + 8 * c8) * 2);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(g) : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// Calls body(tile_smem, q) for every tile of this CTA, the tile staged and
// visible to all threads; body may rewrite the staged tile (every thread
// has finished with a buffer before it is refilled).
template <class Body>
__device__ __forceinline__ void qt_walk(const uint16_t* in, int K, int C, int ng, uint16_t* smem,
                                        Body&& body) {
  const int nkt = K / 128, nct = C / 128;
  const int ntiles = ng * nkt * nct;
  int t = blockIdx.x;
  int buf = 0;
  if (t < ntiles) qt_issue(smem, in, K, C, qt_tile(t, nkt, nct));
  for (; t < ntiles; t += gridDim.x) {
    const int tn = t + gridDim.x;
    if (tn < ntiles) {
      qt_issue(smem + (buf ^ 1) * (kQtTileBytes / 2), in, K, C, qt_tile(tn, nkt, nct));
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();  // this tile's copies (every thread's) have landed
    body(smem + buf * (kQtTileBytes / 2), qt_tile(t, nkt, nct));
    __syncthreads();  // done with this buffer before it is refilled
    buf ^= 1;
  }
}

}  // namespace mok
