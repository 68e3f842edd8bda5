// gemm_tc.cuh -- the weight-streaming projection GEMM (tcgen05 + TMA) used by
// the context-KV update, and the device-side reader of its partial sums.
//
// Y[n, m] = sum_k X[n, k] * W[m, k]: X = activations [Npad, K] bf16 (a few to a
// few hundred rows), W = weights [M, K] bf16.  The weights sit on the MMA's M
// side (128 rows per tile, K-major, 128-byte swizzle) and the activation rows
// on its N side, so a decode-sized batch still fills the 128-row datapath.
// The (N tile, M tile, 64-deep K block) units are spread evenly over one CTA
// per SM (stream-K): each CTA streams exactly its share of the weights once.
//
// The GEMM does not finish split tiles itself.  Every CTA that works on output
// tile t writes its fp32 share as partial j = c - c0(t) (c0 = the tile's first
// CTA), and the next kernel reads Y through gemm_out_issue / gemm_out_finish,
// which add a tile's partials in CTA order: the same sum, bit for bit, whichever CTA ended first,
// with no ticket, fence or extra pass at the GEMM's tail.
#pragma once

#include <cuda.h>

#include "ctx_rows.cuh"
#include "dflash_internal.cuh"
#include "sm100_ptx.cuh"

namespace dflash {

using ptx::griddep_launch;
using ptx::griddep_wait;

// Where a GEMM's result lives: part[t][j][nr][mr] fp32, t = output tile
// (nt * mtiles + m / 128), j < parts(t) the contributing CTA in order,
// nr = n - nt * ntile, mr = m % 128.
struct GemmOut {
  const float *part;
  unsigned units;  // (N tile, M tile, K block) units; units * ctas < 2^32
  int ctas, kblocks, mtiles, maxc, ntile;
};

// Number of CTAs that wrote partials of output tile t.
__device__ __forceinline__ int gemm_tile_parts(const GemmOut &g, unsigned t) {
  const unsigned C = static_cast<unsigned>(g.ctas), U = g.units,
                 KB = static_cast<unsigned>(g.kblocks);
  const unsigned c0 = ((t * KB + 1u) * C - 1u) / U;
  const unsigned c1 = ((t + 1u) * KB * C - 1u) / U;
  const int n = static_cast<int>(c1 - c0) + 1;
  return n < g.maxc ? n : g.maxc;
}

// Y[n, m] read in two halves, so that other loads can go out in between:
// gemm_out_issue starts the loads of up to 8 partials of the element,
// gemm_out_finish adds them (and any further ones) in CTA order.
struct GemmOutLoad {
  float v[8];
  const float *src;
  int cnt;
};

__device__ __forceinline__ void gemm_out_issue(const GemmOut &g, unsigned t, int cnt, int nr, int mr,
                                               GemmOutLoad &ld) {
  const size_t stride = static_cast<size_t>(g.ntile) * 128;
  ld.src = g.part + static_cast<size_t>(t) * g.maxc * stride + static_cast<size_t>(nr) * 128 + mr;
  ld.cnt = cnt;
#pragma unroll
  for (int j = 0; j < 8; ++j) ld.v[j] = j < cnt ? __ldcg(ld.src + j * stride) : 0.f;
}

__device__ __forceinline__ float gemm_out_finish(const GemmOut &g, const GemmOutLoad &ld) {
  const size_t stride = static_cast<size_t>(g.ntile) * 128;
  float acc = ld.v[0];
#pragma unroll
  for (int j = 1; j < 8; ++j)
    if (j < ld.cnt) acc += ld.v[j];
  for (int j = 8; j < ld.cnt; ++j) acc += __ldcg(ld.src + j * stride);
  return acc;
}

// Bytes of partial-tile storage a GEMM of this shape needs on this device.
size_t gemm_partial_bytes(int M, int K, int Npad);

// Enqueue Y = X W^T into `part` (gemm_partial_bytes) and describe it in *out.
// X: [N, K] bf16, W: [M, K] bf16.  A pipeline wait that times out ORs
// DFLASH_DEV_WAIT_TIMEOUT into *status (when non-null).  `pdl` launches with
// programmatic stream serialization: the kernel prefetches weight tiles
// before waiting on the previous kernel's output.  cudaErrorInvalidValue for a shape whose unit
// count does not fit the reader's 32-bit arithmetic.
cudaError_t launch_gemm(const uint16_t *X, int N, int K, const uint16_t *W, int M, float *part,
                        int32_t *status, bool pdl, cudaStream_t s, GemmOut *out);


// Decode-sized fc projection as a cluster split-K GEMM: h = bf16(X W^T)
// [R rows][M] bf16 (R = fc_cluster_rows(N): 16, 32 or 64; rows past N are
// zero) and, per 32-feature slice and row, the sum of h^2: ssq[M / 32][R]
// (the slices of a row, added in order, give its sum of squares).
// fc_cluster_ok: the shape (N <= 64 rows, M % 128 == 0, K % 256 == 0) and
// the device (every cluster resident at once) allow it.
bool fc_cluster_ok(int N, int K, int M);
int fc_cluster_rows(int N);
// rd / rf (optional, nullptr = none): while its CTAs wait for their
// accumulators, warp 2 of CTA n < N runs the row set-up of row n
// (row_setup_warp) for the epilogue.
cudaError_t launch_fc_cluster(const uint16_t *X, int N, int K, const uint16_t *W, int M,
                              uint16_t *h, float *ssq, int32_t *status, cudaStream_t st,
                              const RowDest *rd = nullptr, const RopeFreqs *rf = nullptr);

}  // namespace dflash
