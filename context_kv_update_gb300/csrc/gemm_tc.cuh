// gemm_tc.cuh -- the weight-streaming projection GEMM (tcgen05 + TMA) used by
// the context-KV update, and the device-side reader of its partial sums.
//
// Y[n, m] = sum_k X[n, k] * W[m, k]: X = activations [Npad, K] bf16 (a few to a
// few hundred rows), W = weights [M, K] bf16.  The weights sit on the MMA's M
// side (128 rows per tile, K-major, 128-byte swizzle) and the activation rows
// on its N side, so a decode-sized batch still fills the 128-row datapath.
// The (N tile, M tile, 64-deep K block) units are spread evenly over one CTA
// per SM (stream-K): each CTA streams exactly its share of the weights once
// and writes one fp32 partial tile per output tile it touched.  Consumers sum
// the partials of a tile in CTA order (deterministic), see gemm_out_value.
#pragma once

#include <cuda.h>

#include "dflash_internal.cuh"
#include "sm100_ptx.cuh"

namespace dflash {

using ptx::griddep_launch;
using ptx::griddep_wait;

// Where a GEMM left its result: partial tiles plus the stream-K schedule.
struct GemmOut {
  const float *part;
  int ntile;        // activation rows per N tile (16..256)
  int mtiles;       // ceil(M / 128)
  int kblocks;      // ceil(K / 64)
  int ctas;         // CTAs of the launch
  int maxt;         // partial-tile slots per CTA
  long long units;  // n_tiles * mtiles * kblocks
};

// Sum of the partials of output (n, m), in increasing CTA order (one-off
// reads; bulk readers use GemmTileTable).
__device__ __forceinline__ float gemm_out_value(const GemmOut &y, int n, int m) {
  const int nt = n / y.ntile, nn = n - nt * y.ntile;
  const long long t = static_cast<long long>(nt) * y.mtiles + (m >> 7);
  const int row = m & 127;
  const long long U = y.units, C = y.ctas, KB = y.kblocks;
  const long long a = t * KB, b = (t + 1) * KB;
  const long long c0 = ((a + 1) * C - 1) / U;
  const long long c1 = (b * C - 1) / U;
  float acc = 0.f;
  for (long long c = c0; c <= c1; ++c) {
    const long long local = t - (c * U / C) / KB;
    acc += y.part[((c * y.maxt + local) * y.ntile + nn) * 128 + row];
  }
  return acc;
}

// Shared-memory table of the partial tiles behind output tiles [t0, t0 + nt):
// for tile k, entries base[start[k] .. start[k] + cnt[k]) are the float offsets
// of its partial tiles in CTA order.  Built by the whole block.
constexpr int kTableMaxTiles = 64;
constexpr int kTableMaxEntries = kTableMaxTiles + 160 + 8;
struct GemmTileTable {
  long long base[kTableMaxEntries];
  int start[kTableMaxTiles];
  int cnt[kTableMaxTiles];
};

__device__ __forceinline__ void gemm_tile_table(const GemmOut &y, long long t0, int nt,
                                                GemmTileTable *tb) {
  const long long U = y.units, C = y.ctas, KB = y.kblocks;
  for (int k = threadIdx.x; k < nt; k += blockDim.x) {
    const long long t = t0 + k;
    const long long c0 = ((t * KB + 1) * C - 1) / U;
    const long long c1 = ((t + 1) * KB * C - 1) / U;
    tb->cnt[k] = static_cast<int>(c1 - c0 + 1);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int k = 0; k < nt; ++k) {
      tb->start[k] = acc;
      acc += tb->cnt[k];
    }
  }
  __syncthreads();
  for (int k = threadIdx.x; k < nt; k += blockDim.x) {
    const long long t = t0 + k;
    const long long c0 = ((t * KB + 1) * C - 1) / U;
    for (int j = 0; j < tb->cnt[k]; ++j) {
      const long long c = c0 + j;
      const long long local = t - (c * U / C) / KB;
      tb->base[tb->start[k] + j] = (c * y.maxt + local) * y.ntile * 128;
    }
  }
  __syncthreads();
}

// Value at (row nn of the N tile, column m) using a table built for tiles
// starting at t0 (m counted from the start of tile t0).
__device__ __forceinline__ float gemm_table_value(const GemmOut &y, const GemmTileTable &tb, int nn,
                                                  int m) {
  const int k = m >> 7, row = m & 127;
  const long long off = static_cast<long long>(nn) * 128 + row;
  float acc = 0.f;
  for (int j = 0; j < tb.cnt[k]; ++j) acc += y.part[tb.base[tb.start[k] + j] + off];
  return acc;
}

// Bytes of partial-tile storage a GEMM of this shape needs on this device.
size_t gemm_partial_bytes(int M, int K, int Npad);

// Enqueue Y = X W^T.  X: [Npad, K] bf16 (rows >= N may hold anything; they
// are computed but never read back), W: [M, K] bf16.  `pdl` launches with
// programmatic stream serialization: the kernel prefetches weight tiles before
// waiting on the previous kernel's output.
cudaError_t launch_gemm(const uint16_t *X, int N, int K, const uint16_t *W, int M, float *part,
                        GemmOut *out, bool pdl, cudaStream_t s);

}  // namespace dflash
