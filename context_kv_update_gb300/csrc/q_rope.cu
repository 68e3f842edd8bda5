// q_rope.cu -- the query side of the drafter layer: RMSNorm + RoPE of the
// query rows at their positions.
//
// Follows TensorRT-LLM PR #13995, commits "use fused qk-norm+rope on non-YaRN
// draft" (query norm and rotation in one kernel) and "match RoPE between
// context and query" (the query rows must be rotated with exactly the cos/sin
// of the context keys): the angle comes from rope_cos_sin and the frequency
// table from fill_rope_freqs, the same code the context-KV update rotates its
// keys with, and the norm is written as the key norm is.
#include "dflash_internal.cuh"
#include "sm100_ptx.cuh"

namespace dflash {
namespace {

// grid (rows, heads), block = dim threads.  In place is allowed: every thread
// reads its element before the first barrier and writes after the last.
__global__ void q_norm_rope_kernel(const uint16_t *q_in, const uint16_t *gamma,
                                   const int32_t *pos, const RopeFreqs rf, uint16_t *q_out,
                                   int heads, int dim, float eps) {
  __shared__ float red[32];
  __shared__ float qbuf[kMaxHeadDim];
  ptx::griddep_launch();
  ptx::griddep_wait();
  const int row = blockIdx.x, h = blockIdx.y, d = threadIdx.x;
  const size_t off = (static_cast<size_t>(row) * heads + h) * dim + d;
  const int p = pos[row];
  float v = bf16_to_f32(q_in[off]);
  if (gamma) {
    const float ss = block_sum(v * v, red);
    const float inv = rsqrtf(ss / static_cast<float>(dim) + eps);
    v = v * inv * bf16_to_f32(gamma[d]);
  }
  qbuf[d] = v;
  __syncthreads();
  const int half = dim >> 1;
  const int j = d < half ? d : d - half;
  float c, s;
  rope_cos_sin(p, rf.f[j], &c, &s);
  v = d < half ? v * c - qbuf[d + half] * s : v * c + qbuf[d - half] * s;
  q_out[off] = f32_to_bf16_rn(v);
}

}  // namespace

cudaError_t launch_q_norm_rope(const dflash_geom &g, int rows, const void *q_in,
                               const void *gamma, const int32_t *pos, void *q_out,
                               cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const bool gqa = g.kind == DFLASH_KIND_GQA;
  const int dim = gqa ? g.head_dim : g.rope_dim;
  RopeFreqs rf;
  fill_rope_freqs(&rf, dim, g.rope_theta);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(rows, g.hq);
  cfg.blockDim = dim3(dim);
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, q_norm_rope_kernel, static_cast<const uint16_t *>(q_in),
                            static_cast<const uint16_t *>(gamma), pos, rf,
                            static_cast<uint16_t *>(q_out), g.hq, dim,
                            static_cast<float>(g.eps_k));
}

}  // namespace dflash
