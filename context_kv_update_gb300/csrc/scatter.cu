// scatter.cu -- per-layer block K/V (GQA) or block latent (MLA) scatter into
// the paged pool at the DraftBlockPlacement.
//
// Follows TensorRT-LLM issue #20548 (Proposal: each layer writes its block
// latents into the pool) and PR #20550 (Description: that write becomes one
// scatter kernel per layer in place of an index_put; the follow-up commit's
// DraftBlockPlacement supplies page, slot and mask).  One CTA per block row; 16-byte vector copies.
#include "dflash_internal.cuh"

namespace dflash {
namespace {

__global__ void __launch_bounds__(256) block_scatter_kernel(
    const uint4 *blk_k, const uint4 *blk_v, const int32_t *page, const int32_t *slot,
    const uint8_t *mask, uint16_t *pool, int kind, int nkv, int hd, int W, int P, int NP, int layer,
    int32_t *st) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int row = blockIdx.x;  // r * T + i
  if (!mask[row]) return;
  const int pg = page[row], sl = slot[row];
  if (pg < 0 || pg >= NP || sl < 0 || sl >= P) {
    if (threadIdx.x == 0) raise_status(st, DFLASH_DEV_BAD_PAGE);
    return;
  }
  if (kind == DFLASH_KIND_GQA) {
    const int vec_per_head = hd / 8;
    const int total = 2 * nkv * vec_per_head;
    for (int t = threadIdx.x; t < total; t += blockDim.x) {
      const int kv = t / (nkv * vec_per_head);
      const int rem = t - kv * nkv * vec_per_head;
      const int h = rem / vec_per_head, e = rem % vec_per_head;
      const uint4 *src = (kv == 0 ? blk_k : blk_v) + (static_cast<size_t>(row) * nkv + h) * vec_per_head + e;
      uint4 *dst = reinterpret_cast<uint4 *>(
          pool + ((((static_cast<size_t>(layer) * NP + pg) * 2 + kv) * nkv + h) * P + sl) * hd);
      dst[e] = *src;
    }
  } else {
    const int vec = W / 8;
    uint4 *dst =
        reinterpret_cast<uint4 *>(pool + ((static_cast<size_t>(layer) * NP + pg) * P + sl) * W);
    for (int t = threadIdx.x; t < vec; t += blockDim.x) dst[t] = blk_k[static_cast<size_t>(row) * vec + t];
  }
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
  cfg.blockDim = dim3(256);
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
