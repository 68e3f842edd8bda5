// gemm_tc.cuh -- the weight-streaming projection GEMM (tcgen05 + TMA) used by
// the context-KV update, and the device-side reader of its partial sums.
//
// Y[n, m] = sum_k X[n, k] * W[m, k]: X = activations [Npad, K] bf16 (a few to a
// few hundred rows), W = weights [M, K] bf16.  The weights sit on the MMA's M
// side (128 rows per tile, K-major, 128-byte swizzle) and the activation rows
// on its N side, so a decode-sized batch still fills the 128-row datapath.
// The (N tile, M tile, 64-deep K block) units are spread evenly over one CTA
// per SM (stream-K): each CTA streams exactly its share of the weights once.
// A tile split between CTAs is finished by the last of them, which sums the
// partials in CTA order (deterministic) into the dense fp32 result.
#pragma once

#include <cuda.h>

#include "dflash_internal.cuh"
#include "sm100_ptx.cuh"

namespace dflash {

using ptx::griddep_launch;
using ptx::griddep_wait;

// Bytes of partial-tile storage a GEMM of this shape needs on this device.
size_t gemm_partial_bytes(int M, int K, int Npad);
// Output tiles (one stream-K ticket each) of a GEMM with M columns, Npad rows.
int gemm_num_tiles(int M, int Npad);

// Enqueue y = X W^T (fp32 [N, M], dense).  X: [N, K] bf16, W: [M, K] bf16.
// `part` is partial-tile scratch (gemm_partial_bytes), `counters` one int per
// output tile (gemm_num_tiles), zero on entry and left zero.  `pdl` launches
// with programmatic stream serialization: the kernel prefetches weight tiles
// before waiting on the previous kernel's output.
cudaError_t launch_gemm(const uint16_t *X, int N, int K, const uint16_t *W, int M, float *part,
                        float *y, int *counters, bool pdl, cudaStream_t s);

}  // namespace dflash
