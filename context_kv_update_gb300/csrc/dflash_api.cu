// dflash_api.cu -- the extern "C" entry points declared in include/dflash.h:
// argument validation, then the launchers of the other translation units.
// Nothing here allocates, synchronises or reads device memory.
#include <cmath>
#include <mutex>

#include "dflash_internal.cuh"

namespace dflash {

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
    return 1;
  return n;
}

void fill_rope_freqs(RopeFreqs *rf, int dim, double theta) {
  for (int j = 0; j < dim / 2 && j < kMaxHeadDim / 2; ++j)
    rf->f[j] = std::pow(theta, -2.0 * static_cast<double>(j) / static_cast<double>(dim));
}

namespace {

bool geom_ok(const dflash_geom *g) {
  if (!g) return false;
  if (g->num_layers < 1 || g->d_in < 1 || g->d_model < 1 || g->hq < 1 || g->page_size < 1 ||
      g->max_pages < 1 || g->num_pool_pages < 1 || g->block_size < 1)
    return false;
  if (g->kind == DFLASH_KIND_GQA) {
    if (g->nkv < 1 || g->head_dim < 8 || g->hq % g->nkv != 0) return false;
  } else if (g->kind == DFLASH_KIND_MLA) {
    if (g->latent_dim < 8 || g->rope_dim < 2) return false;
  } else {
    return false;
  }
  if (!(g->rope_theta > 0.0) || !(g->eps_hidden >= 0.0) || !(g->eps_k >= 0.0)) return false;
  return true;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? DFLASH_OK : DFLASH_ERR_CUDA; }

}  // namespace
}  // namespace dflash

using namespace dflash;

extern "C" {

int dflash_abi_version(void) { return 1; }

const char *dflash_status_string(int code) {
  switch (code) {
    case DFLASH_OK: return "ok";
    case DFLASH_ERR_INVALID_ARG: return "invalid argument";
    case DFLASH_ERR_UNSUPPORTED_GEOM: return "unsupported geometry";
    case DFLASH_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case DFLASH_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

}  // extern "C"

extern "C" int dflash_step_bookkeeping(const dflash_geom *g, int B, const int32_t *raw_offsets,
                                       int64_t off_row_stride, int32_t off_div,
                                       const int32_t *accepted_tokens, int64_t acc_row_stride,
                                       const int32_t *n_accepted, const int32_t *ctx_len_pre,
                                       const uint8_t *valid, int32_t max_ctx,
                                       int32_t mask_token_id, const dflash_step_outputs *out,
                                       int32_t *dev_status, dflash_stream_t stream) {
  if (!g || B < 0 || off_div < 1 || !out) return DFLASH_ERR_INVALID_ARG;
  if (g->max_pages < 1 || g->page_size < 1 || g->block_size < 1) return DFLASH_ERR_INVALID_ARG;
  if (B == 0) return DFLASH_OK;
  if (!raw_offsets || !accepted_tokens || !n_accepted || !ctx_len_pre) return DFLASH_ERR_INVALID_ARG;
  if (off_row_stride < g->max_pages || acc_row_stride < g->block_size) return DFLASH_ERR_INVALID_ARG;
  if (max_ctx < 0) return DFLASH_ERR_INVALID_ARG;
  const dflash_step_outputs &o = *out;
  if (!o.n_pages || !o.block_table || !o.alloc_limit || !o.bonus || !o.emb_ids || !o.ctx_pos ||
      !o.q_pos || !o.ctx_dst_page || !o.ctx_dst_slot || !o.ctx_wmask || !o.blk_page ||
      !o.blk_slot || !o.blk_mask || !o.ctx_len_new || !o.seq_lens)
    return DFLASH_ERR_INVALID_ARG;
  return cuda_status(launch_bookkeeping(*g, B, raw_offsets, off_row_stride, off_div,
                                        accepted_tokens, acc_row_stride, n_accepted, ctx_len_pre,
                                        valid, max_ctx, mask_token_id, o, dev_status,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" void dflash_test_attention_skip_tile(int tile) {
  attention_test_skip_tile(tile < 0 ? -1 : tile);
}

extern "C" size_t dflash_packed_kv_bytes(const dflash_geom *g) {
  if (!geom_ok(g)) return 0;
  return packed_kv_bytes(*g);
}

extern "C" size_t dflash_packed_gamma_bytes(const dflash_geom *g) {
  if (!geom_ok(g)) return 0;
  return packed_gamma_bytes(*g);
}

extern "C" int dflash_pack_weights(const dflash_geom *g, const dflash_layer_weights *layers,
                                   void *w_kv, void *gamma_k, dflash_stream_t stream) {
  if (!geom_ok(g) || !layers || !w_kv || !gamma_k) return DFLASH_ERR_INVALID_ARG;
  if (g->num_layers > max_pack_layers() || g->d_model % 8 != 0) return DFLASH_ERR_UNSUPPORTED_GEOM;
  const bool gqa = g->kind == DFLASH_KIND_GQA;
  if (!aligned16(w_kv) || (reinterpret_cast<uintptr_t>(gamma_k) & 1u)) return DFLASH_ERR_INVALID_ARG;
  for (int l = 0; l < g->num_layers; ++l) {
    const dflash_layer_weights &w = layers[l];
    if (!w.w_k || !w.k_norm || !aligned16(w.w_k) || (reinterpret_cast<uintptr_t>(w.k_norm) & 1u))
      return DFLASH_ERR_INVALID_ARG;
    if (gqa ? (!w.w_v || !aligned16(w.w_v)) : (w.w_v != nullptr)) return DFLASH_ERR_INVALID_ARG;
  }
  return cuda_status(
      launch_pack_weights(*g, layers, w_kv, gamma_k, reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" int dflash_strict_accept(int B, int K, const int32_t *draft, int64_t draft_row_stride,
                                    const int32_t *target, int64_t target_row_stride,
                                    int32_t *n_accepted, int32_t *accepted,
                                    dflash_stream_t stream) {
  if (B < 0 || K < 0) return DFLASH_ERR_INVALID_ARG;
  if (B == 0) return DFLASH_OK;
  if (!target || !n_accepted || !accepted || (K > 0 && !draft)) return DFLASH_ERR_INVALID_ARG;
  if (draft_row_stride < K || target_row_stride < K + 1) return DFLASH_ERR_INVALID_ARG;
  return cuda_status(launch_strict_accept(B, K, draft, draft_row_stride, target,
                                          target_row_stride, n_accepted, accepted,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" int dflash_embedding_gather(int n, const int32_t *ids, const void *table, int vocab,
                                       int dim, void *out, int32_t *dev_status,
                                       dflash_stream_t stream) {
  if (n < 0 || vocab < 1) return DFLASH_ERR_INVALID_ARG;
  if (dim < 8 || dim % 8 != 0) return DFLASH_ERR_UNSUPPORTED_GEOM;
  if (n == 0) return DFLASH_OK;
  if (!ids || !table || !out || !aligned16(table) || !aligned16(out)) return DFLASH_ERR_INVALID_ARG;
  return cuda_status(launch_embedding_gather(n, ids, table, vocab, dim, out, dev_status,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" size_t dflash_ctx_workspace_bytes(const dflash_geom *g, int B) {
  if (!geom_ok(g) || B < 0) return 0;
  return ctx_workspace_bytes(*g, B);
}

namespace {

// Geometry the context update (fused or split) supports.
int update_geom_status(const dflash_geom *g) {
  if (g->d_in % 64 != 0 || g->d_model % 64 != 0) return DFLASH_ERR_UNSUPPORTED_GEOM;
  // the hidden RMSNorm spreads a row over at most 8 CTAs of 1024 columns
  if (g->d_in > 8192 || g->d_model > 8192) return DFLASH_ERR_UNSUPPORTED_GEOM;
  if (g->kind == DFLASH_KIND_GQA) {
    if (g->head_dim % 8 != 0 || g->head_dim > kMaxHeadDim || g->head_dim % 2 != 0)
      return DFLASH_ERR_UNSUPPORTED_GEOM;
  } else {
    if (g->latent_dim + g->rope_dim > 1024 || g->rope_dim % 2 != 0 || g->rope_dim > kMaxHeadDim ||
        (g->latent_dim + g->rope_dim) % 8 != 0)
      return DFLASH_ERR_UNSUPPORTED_GEOM;
  }
  return DFLASH_OK;
}

bool weights_ok(const dflash_weights *w) {
  return w->w_fc && w->gamma_h && w->w_kv && w->gamma_k && aligned16(w->w_fc) && aligned16(w->w_kv);
}

bool aligned256(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

}  // namespace

extern "C" int dflash_ctx_kv_update(const dflash_geom *g, int B, const void *hidden,
                                    int hidden_dtype, const int32_t *n_accepted, int32_t *ctx_len,
                                    const int32_t *alloc_limit, const int32_t *block_table,
                                    const uint8_t *valid, const dflash_weights *w, void *kv_pool,
                                    void *workspace, size_t ws_bytes, int32_t *dev_status,
                                    dflash_stream_t stream) {
  if (!geom_ok(g) || B < 0 || !w) return DFLASH_ERR_INVALID_ARG;
  if (hidden_dtype != DFLASH_DTYPE_BF16 && hidden_dtype != DFLASH_DTYPE_F32)
    return DFLASH_ERR_INVALID_ARG;
  if (const int gs = update_geom_status(g)) return gs;
  if (B == 0) return DFLASH_OK;
  if (!hidden || !n_accepted || !ctx_len || !alloc_limit || !block_table || !kv_pool || !workspace)
    return DFLASH_ERR_INVALID_ARG;
  if (!weights_ok(w) || !aligned16(hidden) || !aligned16(kv_pool) || !aligned256(workspace))
    return DFLASH_ERR_INVALID_ARG;
  if (ws_bytes < ctx_workspace_bytes(*g, B)) return DFLASH_ERR_WORKSPACE_TOO_SMALL;
  return cuda_status(launch_ctx_kv_update(*g, B, hidden, hidden_dtype, n_accepted, ctx_len,
                                          alloc_limit, block_table, valid, *w, kv_pool, workspace,
                                          dev_status, reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" size_t dflash_ctx_prefill_workspace_bytes(const dflash_geom *g, int B, int n_rows) {
  if (!geom_ok(g) || B < 0 || n_rows < 0 || n_rows > kMaxPrefillRows) return 0;
  return ctx_prefill_workspace_bytes(*g, B, n_rows);
}

extern "C" int dflash_ctx_kv_prefill(const dflash_geom *g, int B, int n_rows, const void *hidden,
                                     int hidden_dtype, const int32_t *cu_rows, int32_t *ctx_len,
                                     const int32_t *alloc_limit, const int32_t *block_table,
                                     const uint8_t *valid, const dflash_weights *w,
                                     void *kv_pool, void *workspace, size_t ws_bytes,
                                     int32_t *dev_status, dflash_stream_t stream) {
  if (!geom_ok(g) || B < 0 || n_rows < 0 || !w) return DFLASH_ERR_INVALID_ARG;
  if (n_rows > kMaxPrefillRows) return DFLASH_ERR_UNSUPPORTED_GEOM;
  if (hidden_dtype != DFLASH_DTYPE_BF16 && hidden_dtype != DFLASH_DTYPE_F32)
    return DFLASH_ERR_INVALID_ARG;
  if (const int gs = update_geom_status(g)) return gs;
  if (B == 0) return DFLASH_OK;
  if (!cu_rows || !ctx_len || !alloc_limit || !block_table || !kv_pool || !workspace ||
      (n_rows > 0 && !hidden))
    return DFLASH_ERR_INVALID_ARG;
  if (!weights_ok(w) || (hidden && !aligned16(hidden)) || !aligned16(kv_pool) ||
      !aligned256(workspace))
    return DFLASH_ERR_INVALID_ARG;
  if (ws_bytes < ctx_prefill_workspace_bytes(*g, B, n_rows)) return DFLASH_ERR_WORKSPACE_TOO_SMALL;
  return cuda_status(launch_ctx_kv_prefill(*g, B, n_rows, hidden, hidden_dtype, cu_rows, ctx_len,
                                           alloc_limit, block_table, valid, *w, kv_pool, workspace,
                                           dev_status, reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" size_t dflash_ctx_staged_bytes(const dflash_geom *g, int B) {
  if (!geom_ok(g) || B < 0) return 0;
  return ctx_staged_bytes(*g, B);
}

extern "C" int dflash_ctx_kv_project(const dflash_geom *g, int B, const void *hidden,
                                     int hidden_dtype, const int32_t *ctx_len,
                                     const dflash_weights *w, void *staged, size_t staged_bytes,
                                     void *workspace, size_t ws_bytes, int32_t *dev_status,
                                     dflash_stream_t stream) {
  if (!geom_ok(g) || B < 0 || !w) return DFLASH_ERR_INVALID_ARG;
  if (hidden_dtype != DFLASH_DTYPE_BF16 && hidden_dtype != DFLASH_DTYPE_F32)
    return DFLASH_ERR_INVALID_ARG;
  if (const int gs = update_geom_status(g)) return gs;
  if (B == 0) return DFLASH_OK;
  if (!hidden || !ctx_len || !staged || !workspace) return DFLASH_ERR_INVALID_ARG;
  if (!weights_ok(w) || !aligned16(hidden) || !aligned256(staged) || !aligned256(workspace))
    return DFLASH_ERR_INVALID_ARG;
  if (ws_bytes < ctx_workspace_bytes(*g, B) || staged_bytes < ctx_staged_bytes(*g, B))
    return DFLASH_ERR_WORKSPACE_TOO_SMALL;
  return cuda_status(launch_ctx_kv_project(*g, B, hidden, hidden_dtype, ctx_len, *w, staged,
                                           workspace, dev_status,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" int dflash_ctx_kv_commit(const dflash_geom *g, int B, const void *staged,
                                    size_t staged_bytes, const int32_t *n_accepted,
                                    int32_t *ctx_len, const int32_t *alloc_limit,
                                    const int32_t *block_table, const uint8_t *valid,
                                    void *kv_pool, int32_t *dev_status, dflash_stream_t stream) {
  if (!geom_ok(g) || B < 0) return DFLASH_ERR_INVALID_ARG;
  if (const int gs = update_geom_status(g)) return gs;
  if (B == 0) return DFLASH_OK;
  if (!staged || !n_accepted || !ctx_len || !alloc_limit || !block_table || !kv_pool)
    return DFLASH_ERR_INVALID_ARG;
  if (!aligned256(staged) || !aligned16(kv_pool)) return DFLASH_ERR_INVALID_ARG;
  if (staged_bytes < ctx_staged_bytes(*g, B)) return DFLASH_ERR_WORKSPACE_TOO_SMALL;
  return cuda_status(launch_ctx_kv_commit(*g, B, staged, n_accepted, ctx_len, alloc_limit,
                                          block_table, valid, kv_pool, dev_status,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" int dflash_q_norm_rope(const dflash_geom *g, int B, int Tq, const void *q_in,
                                  const void *gamma_q, const int32_t *q_pos, void *q_out,
                                  int32_t *dev_status, dflash_stream_t stream) {
  (void)dev_status;  // nothing in the rows can be out of range
  if (!geom_ok(g) || B < 0 || Tq < 1) return DFLASH_ERR_INVALID_ARG;
  const bool gqa = g->kind == DFLASH_KIND_GQA;
  const int dim = gqa ? g->head_dim : g->rope_dim;
  if (dim < 2 || dim % 2 != 0 || dim > kMaxHeadDim) return DFLASH_ERR_UNSUPPORTED_GEOM;
  // GQA: norm + rotation of the head rows; MLA: rotation of the rope part only
  if (gqa != (gamma_q != nullptr)) return DFLASH_ERR_INVALID_ARG;
  if (B == 0) return DFLASH_OK;
  if (!q_in || !q_pos || !q_out) return DFLASH_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q_in) | reinterpret_cast<uintptr_t>(q_out) |
       reinterpret_cast<uintptr_t>(gamma_q)) & 1u)
    return DFLASH_ERR_INVALID_ARG;
  return cuda_status(launch_q_norm_rope(*g, B * Tq, q_in, gamma_q, q_pos, q_out,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" int dflash_block_kv_scatter(const dflash_geom *g, int B, int layer, const void *blk_k,
                                       const void *blk_v, const int32_t *blk_page,
                                       const int32_t *blk_slot, const uint8_t *blk_mask,
                                       void *kv_pool, int32_t *dev_status,
                                       dflash_stream_t stream) {
  if (!geom_ok(g) || B < 0 || layer < 0 || layer >= g->num_layers) return DFLASH_ERR_INVALID_ARG;
  if (B == 0) return DFLASH_OK;
  if (const int st = block_scatter_args_status(*g, blk_k, blk_v, blk_page, blk_slot, blk_mask,
                                               kv_pool))
    return st;
  return cuda_status(launch_block_scatter(*g, B, layer, blk_k, blk_v, blk_page, blk_slot, blk_mask,
                                          kv_pool, dev_status,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" int dflash_attention_num_segments(const dflash_geom *g, int B, int Tq) {
  if (!geom_ok(g) || B < 1 || Tq < 1) return 0;
  return attention_num_segments(*g, B, Tq);
}

extern "C" size_t dflash_attention_workspace_bytes(const dflash_geom *g, int B, int Tq,
                                                   int num_segments) {
  if (!geom_ok(g) || B < 0 || Tq < 1 || num_segments < 0) return 0;
  return attention_workspace_bytes(*g, B, Tq, num_segments);
}

namespace dflash {

// Host-side checks of a block-attention call, shared by the workspace and the
// allocation-free entry points: first the arguments (geometry, indices,
// modes, scale -- resolving scale <= 0 to the method's default), then the
// buffer pointers.  B == 0 passes both (nothing to do).
int attention_args_status(const dflash_geom *g, int B, int layer, int Tq, const void *q_rope,
                          int32_t window, float *scale, int mask_mode, int num_segments) {
  if (!geom_ok(g) || B < 0 || Tq < 1 || layer < 0 || layer >= g->num_layers || window < 0 ||
      num_segments < 0)
    return DFLASH_ERR_INVALID_ARG;
  if (mask_mode != DFLASH_MASK_CAUSAL_TAIL && mask_mode != DFLASH_MASK_BLOCK_BIDIR)
    return DFLASH_ERR_INVALID_ARG;
  if (!std::isfinite(*scale)) return DFLASH_ERR_INVALID_ARG;
  if (g->kind == DFLASH_KIND_GQA) {
    if (g->head_dim != 64 && g->head_dim != 128) return DFLASH_ERR_UNSUPPORTED_GEOM;
    if (q_rope) return DFLASH_ERR_INVALID_ARG;
  } else {
    if (g->latent_dim != 512 || g->rope_dim != 64) return DFLASH_ERR_UNSUPPORTED_GEOM;
    if (B > 0 && !q_rope) return DFLASH_ERR_INVALID_ARG;
  }
  if (!(*scale > 0.f)) *scale = default_attention_scale(*g);
  const int P = g->page_size;
  if (P % 8 != 0 || !(kAttnTileKeys % P == 0 || P % kAttnTileKeys == 0))
    return DFLASH_ERR_UNSUPPORTED_GEOM;
  // TMA row coordinates of the pool are signed 32-bit
  const long long pool_rows = static_cast<long long>(g->num_layers) * g->num_pool_pages * P *
                              (g->kind == DFLASH_KIND_GQA ? 2LL * g->nkv : 1LL);
  if (pool_rows >= (1LL << 31)) return DFLASH_ERR_UNSUPPORTED_GEOM;
  return DFLASH_OK;
}

int attention_ptrs_status(int B, const void *q, const void *q_rope, const void *kv_pool,
                          const int32_t *block_table, const int32_t *kv_len, const void *out) {
  if (B == 0) return DFLASH_OK;
  if (!q || !kv_pool || !block_table || !kv_len || !out) return DFLASH_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv_pool) || !aligned16(out) || (q_rope && !aligned16(q_rope)))
    return DFLASH_ERR_INVALID_ARG;
  return DFLASH_OK;
}

// Pointers and row widths of a block scatter (standalone or fused).
int block_scatter_args_status(const dflash_geom &g, const void *blk_k, const void *blk_v,
                              const int32_t *blk_page, const int32_t *blk_slot,
                              const uint8_t *blk_mask, const void *kv_pool) {
  if (!blk_k || !blk_page || !blk_slot || !blk_mask || !kv_pool) return DFLASH_ERR_INVALID_ARG;
  if (g.kind == DFLASH_KIND_GQA) {
    if (!blk_v || !aligned16(blk_v)) return DFLASH_ERR_INVALID_ARG;
    if (g.head_dim % 8 != 0) return DFLASH_ERR_UNSUPPORTED_GEOM;
  } else {
    if (blk_v) return DFLASH_ERR_INVALID_ARG;
    if ((g.latent_dim + g.rope_dim) % 8 != 0) return DFLASH_ERR_UNSUPPORTED_GEOM;
  }
  if (!aligned16(blk_k) || !aligned16(kv_pool)) return DFLASH_ERR_INVALID_ARG;
  return DFLASH_OK;
}

float default_attention_scale(const dflash_geom &g) {
  // GQA: 1/sqrt(head_dim).  MLA: the absorbed-latent form keeps the scale of
  // the unabsorbed head, a 128-wide no-rope part plus the rope part.
  const double d = (g.kind == DFLASH_KIND_GQA) ? g.head_dim : 128.0 + g.rope_dim;
  return static_cast<float>(1.0 / std::sqrt(d));
}

}  // namespace dflash

extern "C" int dflash_block_attention(const dflash_geom *g, int B, int layer, int Tq,
                                      const void *q, const void *q_rope, const void *kv_pool,
                                      const int32_t *block_table, const int32_t *kv_len,
                                      int32_t window, const float *sinks, float scale,
                                      int mask_mode, int num_segments, void *workspace,
                                      size_t ws_bytes, void *out, int32_t *dev_status,
                                      dflash_stream_t stream) {
  if (const int st =
          attention_args_status(g, B, layer, Tq, q_rope, window, &scale, mask_mode, num_segments))
    return st;
  if (B == 0) return DFLASH_OK;
  if (const int st = attention_ptrs_status(B, q, q_rope, kv_pool, block_table, kv_len, out))
    return st;
  if (!workspace || !aligned16(workspace)) return DFLASH_ERR_INVALID_ARG;
  const int S = num_segments > 0 ? num_segments : attention_num_segments(*g, B, Tq);
  if (ws_bytes < attention_workspace_bytes(*g, B, Tq, S)) return DFLASH_ERR_WORKSPACE_TOO_SMALL;
  return cuda_status(launch_block_attention(*g, B, layer, Tq, q, q_rope, kv_pool, block_table,
                                            kv_len, window, sinks, scale, mask_mode, S, workspace,
                                            out, dev_status,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" int dflash_block_scatter_attention(
    const dflash_geom *g, int B, int layer, int Tq, const void *blk_k, const void *blk_v,
    const int32_t *blk_page, const int32_t *blk_slot, const uint8_t *blk_mask, const void *q,
    const void *q_rope, void *kv_pool, const int32_t *block_table, const int32_t *kv_len,
    int32_t window, const float *sinks, float scale, int mask_mode, int num_segments,
    void *workspace, size_t ws_bytes, void *out, int32_t *dev_status, dflash_stream_t stream) {
  if (const int st =
          attention_args_status(g, B, layer, Tq, q_rope, window, &scale, mask_mode, num_segments))
    return st;
  if (Tq != g->block_size) return DFLASH_ERR_INVALID_ARG;
  if (B == 0) return DFLASH_OK;
  if (const int st = attention_ptrs_status(B, q, q_rope, kv_pool, block_table, kv_len, out))
    return st;
  if (const int st =
          block_scatter_args_status(*g, blk_k, blk_v, blk_page, blk_slot, blk_mask, kv_pool))
    return st;
  if (!workspace || !aligned16(workspace)) return DFLASH_ERR_INVALID_ARG;
  const int S = num_segments > 0 ? num_segments : attention_num_segments(*g, B, Tq);
  if (ws_bytes < attention_workspace_bytes(*g, B, Tq, S)) return DFLASH_ERR_WORKSPACE_TOO_SMALL;
  return cuda_status(launch_block_scatter_attention(
      *g, B, layer, Tq, blk_k, blk_v, blk_page, blk_slot, blk_mask, q, q_rope, kv_pool,
      block_table, kv_len, window, sinks, scale, mask_mode, S, workspace, out, dev_status,
      reinterpret_cast<cudaStream_t>(stream)));
}
