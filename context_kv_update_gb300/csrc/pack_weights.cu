// pack_weights.cu -- dflash_pack_weights: build the stacked projection weights
// the context update reads from the per-layer tensors a model holds.
//
// TensorRT-LLM PR #13995, commits "migrate draft path to per-layer cached K/V
// pool" (one GEMM stacked across the drafter layers) and "fuse cross-layer
// k_norm" (the per-layer k_norm weights stacked once, so one RMSNorm launch
// covers every layer).  Here the stacking is a one-time device copy:
//   GQA  w_kv[l] = [k_proj_l ; v_proj_l]  ([2][nkv * hd][D] per layer),
//        gamma_k[l] = k_norm_l            ([hd] per layer);
//   MLA  w_kv[l] = the latent projection of layer l ([latent + rope][D]),
//        gamma_k[l] = its latent norm gain ([latent]).
// Rows move as 16-byte vectors; nothing is converted, so the packed bytes are
// the inputs' bytes.
#include "dflash_internal.cuh"
#include "sm100_ptx.cuh"

namespace dflash {
namespace {

constexpr int kMaxPackLayers = 64;

struct PackParams {
  const uint4 *w_k[kMaxPackLayers];
  const uint4 *w_v[kMaxPackLayers];  // GQA only
  const uint16_t *gain[kMaxPackLayers];
  uint4 *w_kv;
  uint16_t *gamma;
  long long units_per_layer;  // 16-byte units of one layer's packed rows
  long long units_half;       // GQA: units of k_proj (= v_proj); MLA: units_per_layer
  int L, gain_width;
};

__global__ void __launch_bounds__(256) pack_weights_kernel(const PackParams p) {
  ptx::griddep_launch();
  ptx::griddep_wait();
  const long long total = p.units_per_layer * p.L;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long u = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; u < total;
       u += stride) {
    const int l = static_cast<int>(u / p.units_per_layer);
    const long long w = u - static_cast<long long>(l) * p.units_per_layer;
    const uint4 *src = (w < p.units_half) ? p.w_k[l] + w : p.w_v[l] + (w - p.units_half);
    p.w_kv[u] = __ldg(src);
  }
  const long long gtotal = static_cast<long long>(p.gain_width) * p.L;
  for (long long u = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; u < gtotal;
       u += stride) {
    const int l = static_cast<int>(u / p.gain_width);
    p.gamma[u] = p.gain[l][u - static_cast<long long>(l) * p.gain_width];
  }
}

size_t packed_rows_per_layer(const dflash_geom &g) {
  return g.kind == DFLASH_KIND_GQA ? static_cast<size_t>(2) * g.nkv * g.head_dim
                                   : static_cast<size_t>(g.latent_dim) + g.rope_dim;
}

}  // namespace

size_t packed_kv_bytes(const dflash_geom &g) {
  return static_cast<size_t>(g.num_layers) * packed_rows_per_layer(g) * g.d_model * 2;
}

size_t packed_gamma_bytes(const dflash_geom &g) {
  const size_t w = g.kind == DFLASH_KIND_GQA ? g.head_dim : g.latent_dim;
  return static_cast<size_t>(g.num_layers) * w * 2;
}

int max_pack_layers() { return kMaxPackLayers; }

cudaError_t launch_pack_weights(const dflash_geom &g, const dflash_layer_weights *layers,
                                void *w_kv, void *gamma, cudaStream_t s) {
  PackParams p = {};
  const bool gqa = g.kind == DFLASH_KIND_GQA;
  p.L = g.num_layers;
  p.units_per_layer = static_cast<long long>(packed_rows_per_layer(g)) * g.d_model / 8;
  p.units_half = gqa ? p.units_per_layer / 2 : p.units_per_layer;
  p.gain_width = gqa ? g.head_dim : g.latent_dim;
  for (int l = 0; l < g.num_layers; ++l) {
    p.w_k[l] = static_cast<const uint4 *>(layers[l].w_k);
    p.w_v[l] = static_cast<const uint4 *>(gqa ? layers[l].w_v : layers[l].w_k);
    p.gain[l] = static_cast<const uint16_t *>(layers[l].k_norm);
  }
  p.w_kv = static_cast<uint4 *>(w_kv);
  p.gamma = static_cast<uint16_t *>(gamma);
  const long long total = p.units_per_layer * p.L;
  long long blocks = (total + 255) / 256;
  const long long cap = static_cast<long long>(device_sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pack_weights_kernel, p);
}

}  // namespace dflash
