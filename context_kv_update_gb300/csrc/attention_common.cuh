// attention_common.cuh -- parameters, masks and the window-rebased segment
// layout shared by the split-KV attention kernels and the merge.
#pragma once

#include <math.h>

#include "dflash_internal.cuh"
#include "sm100_ptx.cuh"

namespace dflash {

using ptx::griddep_launch;
using ptx::griddep_wait;

struct AttnParams {
  int kind, B, Tq, hq, nkv, G, layer, NP, P, M;
  int dq, drope, dqk, dv, W;  // q width, q_rope width, score width, value width, latent row
  int window, mask_mode, S;
  float scale;
  const uint16_t *q, *q_rope, *pool;
  const int32_t *tbl, *kv_len;
  const float *sinks;
  float *ws_m, *ws_l, *ws_o;
  uint16_t *out;
  int32_t *st;
  // Fused block scatter (blk_k null: none).  Block rows [B, Tq] of this
  // layer: GQA K and V [B, Tq, nkv, hd], MLA latents [B, Tq, W] (blk_v null),
  // placed at (blk_page, blk_slot) where blk_mask is set.
  const uint4 *blk_k, *blk_v;
  const int32_t *blk_page, *blk_slot;
  const uint8_t *blk_mask;
};

inline AttnParams make_attn_params(const dflash_geom &g, int B, int layer, int Tq, const void *q,
                                   const void *q_rope, const void *pool, const int32_t *tbl,
                                   const int32_t *kv_len, int32_t window, const float *sinks,
                                   float scale, int mask_mode, int S, void *ws, void *out,
                                   int32_t *st) {
  AttnParams p;
  p.kind = g.kind;
  p.B = B;
  p.Tq = Tq;
  p.hq = g.hq;
  p.nkv = (g.kind == DFLASH_KIND_GQA) ? g.nkv : 1;
  p.G = g.hq / p.nkv;
  p.layer = layer;
  p.NP = g.num_pool_pages;
  p.P = g.page_size;
  p.M = g.max_pages;
  if (g.kind == DFLASH_KIND_GQA) {
    p.dq = g.head_dim;
    p.drope = 0;
    p.dv = g.head_dim;
    p.W = g.head_dim;
  } else {
    p.dq = g.latent_dim;
    p.drope = g.rope_dim;
    p.dv = g.latent_dim;
    p.W = g.latent_dim + g.rope_dim;
  }
  p.dqk = p.dq + p.drope;
  p.window = window;
  p.mask_mode = mask_mode;
  p.S = S;
  p.scale = scale;
  p.q = static_cast<const uint16_t *>(q);
  p.q_rope = static_cast<const uint16_t *>(q_rope);
  p.pool = static_cast<const uint16_t *>(pool);
  p.tbl = tbl;
  p.kv_len = kv_len;
  p.sinks = sinks;
  const size_t rows = static_cast<size_t>(B) * Tq * g.hq * S;
  char *w = static_cast<char *>(ws);
  p.ws_m = reinterpret_cast<float *>(w);
  p.ws_l = reinterpret_cast<float *>(w + align_up(rows * sizeof(float), 256));
  p.ws_o = reinterpret_cast<float *>(w + 2 * align_up(rows * sizeof(float), 256));
  p.out = static_cast<uint16_t *>(out);
  p.st = st;
  p.blk_k = p.blk_v = nullptr;
  p.blk_page = p.blk_slot = nullptr;
  p.blk_mask = nullptr;
  return p;
}

cudaError_t launch_attn_merge(const AttnParams &p, cudaStream_t s);
cudaError_t launch_attn_tc(const AttnParams &a, const dflash_geom &g, cudaStream_t s);
cudaError_t launch_attn_mla_tc(const AttnParams &a, const dflash_geom &g, cudaStream_t s);
int mla_rows_per_cta();

// kv_len of request r, clamped to [0, M*P] (flagging out-of-range values).
__device__ __forceinline__ int clamped_kv_len(const AttnParams &p, int r, bool report) {
  int kl = p.kv_len[r];
  const long long cap = static_cast<long long>(p.M) * p.P;
  if (kl < 0 || kl > cap) {
    if (report) raise_status(p.st, DFLASH_DEV_KV_LEN_RANGE);
    kl = kl < 0 ? 0 : static_cast<int>(cap);
  }
  return kl;
}

// Visible keys [lo, hi] of query token i (hi < lo: none).
__device__ __forceinline__ void row_key_range(const AttnParams &p, int kv_len, int i, int *lo,
                                              int *hi) {
  const int pos = kv_len - p.Tq + i;
  *hi = (p.mask_mode == DFLASH_MASK_CAUSAL_TAIL) ? pos : kv_len - 1;
  int l = 0;
  if (p.window > 0) {
    const int w0 = pos - p.window + 1;
    l = w0 > 0 ? w0 : 0;
  }
  *lo = l;
}

// Key range [k0, k1) of segment s of request r: the union of the block's
// visible ranges, [lo_0, kv_len), re-based to start at its first key tile
// and cut into S runs of whole tiles.
struct SegRange {
  int kv_len, k0, k1, t0, t1;
};
// The same from a given (already clamped) kv_len.
__device__ __forceinline__ SegRange segment_range_for(const AttnParams &p, int kv_len, int s) {
  SegRange sr;
  sr.kv_len = kv_len;
  sr.k0 = sr.k1 = sr.t0 = sr.t1 = 0;
  if (sr.kv_len <= 0) return sr;
  int lo0, hi0;
  row_key_range(p, sr.kv_len, 0, &lo0, &hi0);
  const int tile_lo = lo0 / kAttnTileKeys;
  const int tile_hi = (sr.kv_len - 1) / kAttnTileKeys + 1;
  const int ntiles = tile_hi - tile_lo;
  const int per = (ntiles + p.S - 1) / p.S;
  sr.t0 = tile_lo + s * per;
  sr.t1 = min(tile_hi, sr.t0 + per);
  if (sr.t0 >= sr.t1) {
    sr.t0 = sr.t1 = 0;
    return sr;
  }
  sr.k0 = max(lo0, sr.t0 * kAttnTileKeys);
  sr.k1 = min(sr.kv_len, sr.t1 * kAttnTileKeys);
  return sr;
}
__device__ __forceinline__ SegRange segment_range(const AttnParams &p, int r, int s) {
  return segment_range_for(p, clamped_kv_len(p, r, s == 0 && blockIdx.y == 0 && threadIdx.x == 0),
                           s);
}

// Fused block scatter.  The block's row (r, i) holds the key at position
// kv_len - Tq + i (the last Tq keys, which every window sees), so the CTAs
// whose segment range [k0, k1) covers that position are the ones that read
// it: each of them writes the rows of its own range (the row tiles of a
// segment write the same bytes) before its copies of those keys are issued.
// Rows at positions no segment reads (kv_len < Tq) are written by the CTAs of
// segment 0, row tile 0.  GQA: head kvh's K and V rows; MLA: the latent row.
// Warp-wide (the producer warp, before its first copy); each lane ends with a
// proxy fence, so tensor copies issued after the warp's next __syncwarp read
// the new rows.  Only the kernels' scatter instantiations carry this code.
// What the scatter reads of the call, gathered from the kernel parameters
// (constant bank) once.  Measured: an out-of-line scatter reading the fields
// through a reference to the parameters made the CTAs holding the block's
// rows finish ~15 us late; passed by value, ~0.4 us slower than inline.
struct BlockScatterArgs {
  const uint4 *blk_k, *blk_v;
  const int32_t *page, *slot;
  const uint8_t *mask;
  uint16_t *pool;
  int32_t *st;
  int Tq, W, nkv, NP, P, layer;
  int lo0;  // first visible key of the block's first row (row_key_range)
  bool gqa;
};

__device__ __forceinline__ BlockScatterArgs block_scatter_args(const AttnParams &p,
                                                               const SegRange &sr) {
  BlockScatterArgs a;
  a.blk_k = p.blk_k;
  a.blk_v = p.blk_v;
  a.page = p.blk_page;
  a.slot = p.blk_slot;
  a.mask = p.blk_mask;
  a.pool = const_cast<uint16_t *>(p.pool);
  a.st = p.st;
  a.Tq = p.Tq;
  a.W = p.W;
  a.nkv = p.nkv;
  a.NP = p.NP;
  a.P = p.P;
  a.layer = p.layer;
  int hi0 = 0;
  a.lo0 = 0;
  if (sr.kv_len > 0) row_key_range(p, sr.kv_len, 0, &a.lo0, &hi0);
  a.gqa = p.kind == DFLASH_KIND_GQA;
  return a;
}

__device__ __forceinline__ void block_scatter_rows(const BlockScatterArgs a, int r, int kvh,
                                                   const SegRange sr, bool first_cta, int lane) {
  constexpr int kBatch = 8;  // 16-byte vectors a lane has in flight
  const int kl = sr.kv_len, lo0 = a.lo0;
  // Most CTAs hold none of the block's rows: they skip the loop and the fence.
  const bool any_covered = kl > 0 && max(kl - a.Tq, sr.k0) < min(kl, sr.k1);
  const bool any_uncovered = first_cta && (kl <= 0 || kl - a.Tq < lo0);
  if (!any_covered && !any_uncovered) return;
  const bool gqa = a.gqa;
  const int vw = a.W / 8;               // vectors of one cache row
  const int vrow = gqa ? 2 * vw : vw;   // vectors of one block row (GQA: K, V)
  const int total = a.Tq * vrow;
  for (int t0 = 0; t0 < total; t0 += 32 * kBatch) {
    // every load of the batch is issued before any is used
    uint4 v[kBatch];
    int pg[kBatch], sl[kBatch];
    uint8_t placed[kBatch];
    bool mine[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int t = t0 + 32 * u + lane;
      const int i = t / vrow, e = t - i * vrow;
      const int pos = kl - a.Tq + i;
      const bool covered = kl > 0 && pos >= lo0;
      mine[u] = t < total && (covered ? (pos >= sr.k0 && pos < sr.k1) : first_cta);
      placed[u] = 0;
      if (mine[u]) {
        const int64_t k = static_cast<int64_t>(r) * a.Tq + i;
        const int kv = gqa && e >= vw ? 1 : 0, ee = e - kv * vw;
        v[u] = gqa ? (kv ? a.blk_v : a.blk_k)[(k * a.nkv + kvh) * vw + ee] : a.blk_k[k * vw + ee];
        placed[u] = a.mask[k];
        pg[u] = a.page[k];
        sl[u] = a.slot[k];
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (!placed[u]) continue;
      if (pg[u] < 0 || pg[u] >= a.NP || sl[u] < 0 || sl[u] >= a.P) {
        raise_status(a.st, DFLASH_DEV_BAD_PAGE);
        continue;
      }
      const int t = t0 + 32 * u + lane;
      const int e = t % vrow;
      const int kv = gqa && e >= vw ? 1 : 0, ee = e - kv * vw;
      const size_t row = gqa ? ((((static_cast<size_t>(a.layer) * a.NP + pg[u]) * 2 + kv) * a.nkv +
                                 kvh) * a.P + sl[u])
                             : ((static_cast<size_t>(a.layer) * a.NP + pg[u]) * a.P + sl[u]);
      reinterpret_cast<uint4 *>(a.pool + row * a.W)[ee] = v[u];
    }
  }
  ptx::fence_proxy_async_global();
}

// Cache rows of key j (GQA: K and V of head kvh; MLA: the latent row twice).
// False when the table maps j outside the pool (flagged).
__device__ __forceinline__ bool key_rows(const AttnParams &p, int r, int kvh, int j,
                                         const uint16_t **krow, const uint16_t **vrow) {
  const int lp = j / p.P;
  const int page = p.tbl[static_cast<int64_t>(r) * p.M + lp];
  if (page < 0 || page >= p.NP) {
    raise_status(p.st, DFLASH_DEV_BAD_PAGE);
    return false;
  }
  const int slot = j - lp * p.P;
  if (p.kind == DFLASH_KIND_GQA) {
    const size_t base = ((static_cast<size_t>(p.layer) * p.NP + page) * 2) * p.nkv;
    *krow = p.pool + (((base + 0 * p.nkv) + kvh) * p.P + slot) * static_cast<size_t>(p.dq);
    *vrow = p.pool + (((base + 1 * p.nkv) + kvh) * p.P + slot) * static_cast<size_t>(p.dq);
  } else {
    *krow = p.pool + ((static_cast<size_t>(p.layer) * p.NP + page) * p.P + slot) *
                         static_cast<size_t>(p.W);
    *vrow = *krow;
  }
  return true;
}

}  // namespace dflash
