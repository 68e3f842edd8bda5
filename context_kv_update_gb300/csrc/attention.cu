// attention.cu -- decode-shaped split-KV block attention over the paged cache.
//
// Follows vLLM PR #54092 (Purpose item 2, Changes item 2): the drafter's
// small uniform query block (1 bonus + N drafts) runs the split-KV ("3D")
// form: the KV range is cut into segments, each segment writes per-query-token
// partial softmax state (max, sum, weighted values), and a reduce kernel
// merges them.  The segments split only the key range some query row can
// see (with a sliding window, the last `window` keys rather than the whole
// context, most of which no row would read), and the main kernel and the
// reduce derive the same layout; per-head sink logits join the merge.
//
// Workspace (fp32): m[B, Tq, hq, S], l[B, Tq, hq, S], o[B, Tq, hq, S, dv],
// with m in natural-log units of the scaled scores.  A segment with no visible
// key for a row writes m = -inf, l = 0 and leaves o unwritten; the merge never
// reads o of such a segment.
#include <math.h>

#include "attention_common.cuh"

namespace dflash {

// The main kernels live in attention_tc.cu (GQA) and attention_mla_tc.cu
// (MLA latent); this file holds the merge, the segment count and dispatch.

// ----------------------------------------------------------- merge
// One CTA per output row (r, i, h), VEC value dims per thread (one for head
// dims up to 128, four for the 512-wide latent rows).  Segments are merged
// in batches of 32 (20 for 512-wide rows) with a running maximum (online
// log-sum-exp).  Lane j of every warp holds segment j's m and l, so the batch
// maximum and the denominator are warp reductions and each thread keeps only
// its own O elements.  The CTAs are small enough for the whole grid to be
// resident at once (56 registers a thread; for the latent 128 threads a row
// of 112 registers, whose 512 one-dim threads a row took two waves), so it
// starts the moment the main kernel completes.  All loads of a batch are
// issued before any is used (one memory round trip for up to one batch of
// segments).  The sink
// starts the running state as an extra logit with no value.  O of an empty
// segment (m_s = -inf) is loaded but never used (selected away), so a NaN
// there cannot leak.
template <int VEC>
struct MergeVec {
  float v[VEC];
};
template <int VEC>
__device__ __forceinline__ MergeVec<VEC> merge_load(const float *p) {
  MergeVec<VEC> r;
  if constexpr (VEC == 4) {
    const float4 t = __ldcg(reinterpret_cast<const float4 *>(p));
    r.v[0] = t.x;
    r.v[1] = t.y;
    r.v[2] = t.z;
    r.v[3] = t.w;
  } else {
#pragma unroll
    for (int e = 0; e < VEC; ++e) r.v[e] = __ldcg(p + e);
  }
  return r;
}

template <int DV, int VEC>
__global__ void __launch_bounds__(DV / VEC) attn_merge_kernel(const AttnParams p) {
  griddep_launch();
  griddep_wait();
  constexpr int kBatch = DV >= 512 ? 20 : 32;
  const int row = blockIdx.x;  // (r * Tq + i) * hq + h
  const int h = row % p.hq;
  const int d0 = threadIdx.x * VEC, lane = threadIdx.x & 31;
  const size_t base = static_cast<size_t>(row) * p.S;
  const int S = p.S;
  float M = p.sinks ? p.sinks[h] : -INFINITY;
  float den = p.sinks ? 1.f : 0.f;
  float acc[VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
  for (int s0 = 0; s0 < S; s0 += kBatch) {
    const bool in = lane < kBatch && s0 + lane < S;
    const float mj = in ? __ldcg(p.ws_m + base + s0 + lane) : -INFINITY;
    const float lj = in ? __ldcg(p.ws_l + base + s0 + lane) : 0.f;
    MergeVec<VEC> ov[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      if (s0 + j < S) {
        ov[j] = merge_load<VEC>(p.ws_o + (base + s0 + j) * DV + d0);
      } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) ov[j].v[e] = 0.f;
      }
    }
    const float Mn = fmaxf(M, warp_max(mj));
    if (Mn == -INFINITY) continue;
    const float sc = (M == -INFINITY) ? 0.f : __expf(M - Mn);
    const bool live = mj != -INFINITY;
    const float wj = live ? __expf(mj - Mn) : 0.f;
    const unsigned live_mask = __ballot_sync(0xffffffffu, live);
    den = den * sc + warp_sum(wj * lj);
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[e] *= sc;
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const float w = __shfl_sync(0xffffffffu, wj, j);
      const bool lj_live = ((live_mask >> j) & 1u) != 0;
#pragma unroll
      for (int e = 0; e < VEC; ++e) acc[e] += lj_live ? w * ov[j].v[e] : 0.f;
    }
    M = Mn;
  }
  uint16_t *o = p.out + static_cast<size_t>(row) * DV + d0;
  if constexpr (VEC == 4) {
    float f[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) f[e] = den > 0.f ? acc[e] / den : 0.f;
    *reinterpret_cast<uint2 *>(o) = make_uint2(ptx::pack_bf16x2(f[0], f[1]), ptx::pack_bf16x2(f[2], f[3]));
  } else {
#pragma unroll
    for (int e = 0; e < VEC; ++e) o[e] = f32_to_bf16_rn(den > 0.f ? acc[e] / den : 0.f);
  }
}

int attention_num_segments(const dflash_geom &g, int B, int Tq) {
  const int heads = (g.kind == DFLASH_KIND_GQA) ? g.nkv : 1;
  const int rows = Tq * (g.hq / (heads > 0 ? heads : 1));
  // query rows per CTA: 128 for GQA, 64 for the MLA latent (512-wide values)
  const int tile_rows = (g.kind == DFLASH_KIND_GQA) ? 128 : mla_rows_per_cta();
  const int row_tiles = (rows + tile_rows - 1) / tile_rows;
  // the tensor-core kernels run one CTA per SM
  const long long slots = static_cast<long long>(device_sm_count());
  const long long ctas = static_cast<long long>(B) * heads * row_tiles;
  int S = static_cast<int>(slots / (ctas > 0 ? ctas : 1));
  if (B >= 4) {
    // Requests of a batch differ in length, and each gets the same number of
    // segments: about 1.5 waves of CTAs let the block scheduler even out the
    // load (measured on the mixed-length batch workload, B = 4..16).
    S = static_cast<int>((3 * slots + ctas) / (2 * ctas));
  }
  if (S < 1) S = 1;
  const long long max_tiles =
      (static_cast<long long>(g.max_pages) * g.page_size + kAttnTileKeys - 1) / kAttnTileKeys;
  if (S > max_tiles) S = static_cast<int>(max_tiles > 0 ? max_tiles : 1);
  return S;
}

size_t attention_workspace_bytes(const dflash_geom &g, int B, int Tq, int S) {
  if (S <= 0) S = attention_num_segments(g, B, Tq);
  const int dv = (g.kind == DFLASH_KIND_GQA) ? g.head_dim : g.latent_dim;
  const size_t rows = static_cast<size_t>(B) * Tq * g.hq * S;
  size_t off = align_up(rows * sizeof(float), 256) * 2;
  off += rows * dv * sizeof(float);
  return align_up(off, 256);
}

cudaError_t launch_block_attention(const dflash_geom &g, int B, int layer, int Tq, const void *q,
                                   const void *q_rope, const void *pool, const int32_t *tbl,
                                   const int32_t *kv_len, int32_t window, const float *sinks,
                                   float scale, int mask_mode, int S, void *ws, void *out,
                                   int32_t *st, cudaStream_t s) {
  return launch_block_scatter_attention(g, B, layer, Tq, nullptr, nullptr, nullptr, nullptr,
                                        nullptr, q, q_rope, pool, tbl, kv_len, window, sinks,
                                        scale, mask_mode, S, ws, out, st, s);
}

cudaError_t launch_block_scatter_attention(const dflash_geom &g, int B, int layer, int Tq,
                                           const void *blk_k, const void *blk_v,
                                           const int32_t *blk_page, const int32_t *blk_slot,
                                           const uint8_t *blk_mask, const void *q,
                                           const void *q_rope, const void *pool,
                                           const int32_t *tbl, const int32_t *kv_len,
                                           int32_t window, const float *sinks, float scale,
                                           int mask_mode, int S, void *ws, void *out, int32_t *st,
                                           cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  if (S <= 0) S = attention_num_segments(g, B, Tq);
  AttnParams p = make_attn_params(g, B, layer, Tq, q, q_rope, pool, tbl, kv_len, window, sinks,
                                  scale, mask_mode, S, ws, out, st);
  p.blk_k = static_cast<const uint4 *>(blk_k);
  p.blk_v = static_cast<const uint4 *>(blk_v);
  p.blk_page = blk_page;
  p.blk_slot = blk_slot;
  p.blk_mask = blk_mask;
  cudaError_t e;
  if (g.kind == DFLASH_KIND_GQA)
    e = launch_attn_tc(p, g, s);
  else
    e = launch_attn_mla_tc(p, g, s);
  if (e != cudaSuccess) return e;
  return launch_attn_merge(p, s);
}

cudaError_t launch_attn_merge(const AttnParams &p, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(p.B * p.Tq * p.hq);
  cfg.blockDim = dim3(p.dv >= 512 ? p.dv / 4 : p.dv);
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (p.dv) {
    case 64: return cudaLaunchKernelEx(&cfg, attn_merge_kernel<64, 1>, p);
    case 128: return cudaLaunchKernelEx(&cfg, attn_merge_kernel<128, 1>, p);
    case 512: return cudaLaunchKernelEx(&cfg, attn_merge_kernel<512, 4>, p);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dflash
