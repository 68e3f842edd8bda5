// scatter.cu -- per-layer block K/V (GQA) or block latent (MLA) scatter into
// the paged pool at the DraftBlockPlacement.
//
// Follows TensorRT-LLM issue #20548 (Proposal: each layer writes its block
// latents into the pool) and PR #20550 (Description: that write becomes one
// scatter kernel per layer in place of an index_put; the follow-up commit's
// DraftBlockPlacement supplies page, slot and mask).  One CTA per block row;
// 16-byte vector copies.
#include "dflash_internal.cuh"

namespace dflash {
namespace {

constexpr int kScatterThreads = 256;
constexpr int kScatterVecs = 4;  // 16-byte vectors a thread holds: rows up to 16 KB

__global__ void __launch_bounds__(kScatterThreads) block_scatter_kernel(
    const uint4 *blk_k, const uint4 *blk_v, const int32_t *page, const int32_t *slot,
    const uint8_t *mask, uint16_t *pool, int kind, int nkv, int hd, int W, int P, int NP, int layer,
    int32_t *st) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int row = blockIdx.x;  // r * T + i
  const bool gqa = kind == DFLASH_KIND_GQA;
  const int vph = hd / 8;                      // vectors per head row (GQA)
  const int nv = gqa ? 2 * nkv * vph : W / 8;  // vectors of the block row
  // source vector t of the row: GQA [K heads | V heads], MLA one latent row
  auto src = [&](int t) -> uint4 {
    if (!gqa) return blk_k[static_cast<size_t>(row) * nv + t];
    const int kv = t / (nkv * vph);
    const int rem = t - kv * nkv * vph;
    return (kv == 0 ? blk_k : blk_v)[static_cast<size_t>(row) * nkv * vph + rem];
  };
  auto dst = [&](int t, int pg, int sl) -> uint4 * {
    if (!gqa)
      return reinterpret_cast<uint4 *>(pool + ((static_cast<size_t>(layer) * NP + pg) * P + sl) * W) + t;
    const int kv = t / (nkv * vph);
    const int rem = t - kv * nkv * vph;
    const int h = rem / vph, e = rem % vph;
    return reinterpret_cast<uint4 *>(
               pool + ((((static_cast<size_t>(layer) * NP + pg) * 2 + kv) * nkv + h) * P + sl) * hd) +
           e;
  };
  // The first vectors of the row are loaded before the destination is known:
  // those loads do not depend on it, so they overlap the mask / page / slot
  // lookups, which are all issued before the mask is tested (one memory
  // round trip in all).
  uint4 v[kScatterVecs];
#pragma unroll
  for (int u = 0; u < kScatterVecs; ++u) {
    const int t = threadIdx.x + u * kScatterThreads;
    if (t < nv) v[u] = src(t);
  }
  const uint8_t placed = mask[row];
  const int pg = page[row], sl = slot[row];
  if (!placed) return;
  if (pg < 0 || pg >= NP || sl < 0 || sl >= P) {
    if (threadIdx.x == 0) raise_status(st, DFLASH_DEV_BAD_PAGE);
    return;
  }
#pragma unroll
  for (int u = 0; u < kScatterVecs; ++u) {
    const int t = threadIdx.x + u * kScatterThreads;
    if (t < nv) *dst(t, pg, sl) = v[u];
  }
  for (int t = threadIdx.x + kScatterVecs * kScatterThreads; t < nv; t += kScatterThreads)
    *dst(t, pg, sl) = src(t);
}

}  // namespace

cudaError_t launch_block_scatter(const dflash_geom &g, int B, int layer, const void *blk_k,
                                 const void *blk_v, const int32_t *page, const int32_t *slot,
                                 const uint8_t *mask, void *pool, int32_t *st, cudaStream_t s) {
  const int rows = B * g.block_size;
  if (rows == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(rows);
  cfg.blockDim = dim3(kScatterThreads);
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, block_scatter_kernel, static_cast<const uint4 *>(blk_k),
                            static_cast<const uint4 *>(blk_v), page, slot, mask,
                            static_cast<uint16_t *>(pool), static_cast<int>(g.kind), g.nkv,
                            g.head_dim, g.latent_dim + g.rope_dim, g.page_size, g.num_pool_pages,
                            layer, st);
}

}  // namespace dflash
