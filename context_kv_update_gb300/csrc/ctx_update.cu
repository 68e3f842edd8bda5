// ctx_update.cu -- the per-step context-KV update.
//
// Follows TensorRT-LLM PR #20550 (Description, TLLM_DFLASH_OVERLAP_CONTEXT_
// PROJECTION: the fc projection, hidden norm, latent projection and norm +
// RoPE of the generation tokens, then the masked write of the accepted rows) and PR #13995 ("migrate draft path to
// per-layer cached K/V pool": one GEMM stacked across the drafter layers on
// the newly accepted K+1 rows; "fuse cross-layer k_norm and avoid mask-mul
// alloc": one RMSNorm over [N, L, nkv, hd] with stacked per-layer weights and
// a shared eps; "match RoPE between context and query": one cos/sin
// convention).
//
// Launch chain on the caller's stream:
//   prep      fp32 -> bf16 of the hidden rows (fp32 hidden only)
//   gemm      Y1 = X W_fc^T            (weights streamed once)
//   norm      hn = bf16(bf16(Y1) * gamma_h / rms), ctx_len snapshot
//   gemm      Y2 = hn W_kv^T           (all layers' K/V rows in one pass)
//   epilogue  k RMSNorm + RoPE (GQA) / latent RMSNorm + RoPE (MLA), masked
//             paged bf16 store, ctx_len advance
// Y1 and Y2 stay as the GEMMs' per-CTA partial tiles; the norm and the
// epilogue add them up as they read (gemm_out_issue / gemm_out_finish).
#include <algorithm>

#include "dflash_internal.cuh"
#include "gemm_tc.cuh"

namespace dflash {
namespace {

// ----------------------------------------------------------- workspace map
struct CtxWs {
  int32_t *ctx_snap;  // [B]
  uint16_t *x;        // [Npad, D_in] bf16 (fp32 hidden converted)
  uint16_t *hn;       // [Npad, D]    bf16
  float *part1;       // fc partial tiles (Y1)
  float *part2;       // K/V (or latent) partial tiles (Y2)
  size_t bytes;
};

struct CtxDims {
  int N, Npad, D_in, D, Wrows;
};

CtxDims ctx_dims_rows(const dflash_geom &g, int N) {
  CtxDims d;
  d.N = N;
  d.Npad = static_cast<int>(align_up(static_cast<size_t>(d.N > 0 ? d.N : 1), 16));
  d.D_in = g.d_in;
  d.D = g.d_model;
  d.Wrows = (g.kind == DFLASH_KIND_GQA) ? g.num_layers * 2 * g.nkv * g.head_dim
                                        : g.num_layers * (g.latent_dim + g.rope_dim);
  return d;
}

CtxDims ctx_dims(const dflash_geom &g, int B) { return ctx_dims_rows(g, B * g.block_size); }

// B requests, N rows (the decode update's N = B * T)
CtxWs ctx_ws_map_rows(const dflash_geom &g, int B, int N, void *base) {
  const CtxDims d = ctx_dims_rows(g, N);
  char *p = static_cast<char *>(base);
  size_t off = 0;
  CtxWs w;
  w.ctx_snap = reinterpret_cast<int32_t *>(p + off);
  off = align_up(off + sizeof(int32_t) * (B > 0 ? B : 1), 256);
  w.x = reinterpret_cast<uint16_t *>(p + off);
  off = align_up(off + sizeof(uint16_t) * d.Npad * d.D_in, 256);
  w.hn = reinterpret_cast<uint16_t *>(p + off);
  off = align_up(off + sizeof(uint16_t) * d.Npad * d.D, 256);
  w.part1 = reinterpret_cast<float *>(p + off);
  off = align_up(off + gemm_partial_bytes(d.D, d.D_in, d.Npad), 256);
  w.part2 = reinterpret_cast<float *>(p + off);
  off = align_up(off + gemm_partial_bytes(d.Wrows, d.D, d.Npad), 256);
  w.bytes = off;
  return w;
}

CtxWs ctx_ws_map(const dflash_geom &g, int B, void *base) {
  return ctx_ws_map_rows(g, B, B * g.block_size, base);
}

// ------------------------------------------------------------------ prep
__global__ void prep_kernel(const float *hidden_f32, uint16_t *x, int n_elems, int row_elems,
                            int n_pad_rows) {
  griddep_launch();
  griddep_wait();
  const int tid = blockIdx.x * blockDim.x + threadIdx.x;
  const int total = n_pad_rows * row_elems;
  for (int e = tid; e < total; e += gridDim.x * blockDim.x)
    x[e] = e < n_elems ? f32_to_bf16_rn(hidden_f32[e]) : static_cast<uint16_t>(0);
}

// ----------------------------------------------------- hidden RMSNorm
// hn = bf16(h * gamma_h / rms(h)), h = bf16(Y1 row).  A cluster of G CTAs
// normalises one row, each CTA `cols` consecutive columns; the row's sum of
// squares is added up across the cluster through distributed shared memory,
// in rank order (deterministic).  Each thread issues the loads of all its
// columns' partials before adding any.  The CTAs are small (128 threads), so
// they share the SMs with the GEMMs: the K/V GEMM's CTAs start and prefetch
// their weights while this kernel runs.  CTA (0, 0) also snapshots ctx_len
// for the epilogue, which advances it.
constexpr int kNormThreads = 128;
constexpr int kNormMaxCols = 8 * kNormThreads;  // columns per CTA
constexpr int kClusterNormMaxRows = 256;        // beyond: the row-per-CTA kernel

__global__ void __launch_bounds__(kNormThreads) hidden_norm_kernel(
    const GemmOut y, const uint16_t *gamma, uint16_t *hn, int D, int cols, float eps,
    const int32_t *ctx_len, int32_t *ctx_snap, int B) {
  constexpr int E = kNormMaxCols / kNormThreads;
  __shared__ float red[kNormThreads / 32];
  __shared__ float s_part;
  __shared__ int parts[E + 1];  // partial count of each 128-column tile the CTA covers
  griddep_launch();
  const int x = blockIdx.x, n = blockIdx.y, tid = threadIdx.x;
  const int c0 = x * cols, c1 = min(D, c0 + cols);
  float gv[E];
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const int col = c0 + i * kNormThreads + tid;
    gv[i] = col < c1 ? bf16_to_f32(gamma[col]) : 0.f;  // independent of the previous kernel
  }
  griddep_wait();
  if (n == 0 && x == 0)
    for (int r = tid; r < B; r += kNormThreads) ctx_snap[r] = ctx_len[r];
  const int nt = n / y.ntile, nr = n - nt * y.ntile;
  const unsigned tb = static_cast<unsigned>(nt) * y.mtiles + static_cast<unsigned>(c0 >> 7);
  if (c1 > c0 && tid <= ((c1 - 1) >> 7) - (c0 >> 7)) parts[tid] = gemm_tile_parts(y, tb + tid);
  __syncthreads();
  GemmOutLoad ld[E];
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const int col = c0 + i * kNormThreads + tid;
    const int j = (col >> 7) - (c0 >> 7);
    gemm_out_issue(y, tb + j, col < c1 ? parts[j] : 0, nr, col & 127, ld[i]);
  }
  float h[E], ss = 0.f;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    h[i] = bf16_to_f32(f32_to_bf16_rn(gemm_out_finish(y, ld[i])));
    ss += h[i] * h[i];
  }
  ss = warp_sum(ss);
  if ((tid & 31) == 0) red[tid >> 5] = ss;
  __syncthreads();
  if (tid == 0) {
    float t = 0.f;
    for (int w = 0; w < kNormThreads / 32; ++w) t += red[w];
    s_part = t;
  }
  ptx::cluster_sync();  // every CTA's s_part is written
  // lane r reads CTA r's part (one round trip for all); the butterfly sum
  // leaves the same total in every lane of every warp
  const int lane = tid & 31;
  const float tot =
      warp_sum(lane < static_cast<int>(gridDim.x) ? ptx::ld_dsmem_f32(&s_part, lane) : 0.f);
  ptx::cluster_arrive();  // done reading the other CTAs' s_part
  const float inv = rsqrtf(tot / static_cast<float>(D) + eps);
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const int col = c0 + i * kNormThreads + tid;
    if (col < c1) hn[static_cast<size_t>(n) * D + col] = f32_to_bf16_rn(h[i] * inv * gv[i]);
  }
  ptx::cluster_wait();  // no CTA leaves while another may still read its s_part
}

// The same norm for many rows (prefill): one 256-thread CTA per row and no
// cluster -- with thousands of rows there is parallelism enough, and a
// cluster per row would serialise on cluster scheduling.  Each thread holds
// up to 32 columns; the partials are read in batches of 8 columns.
constexpr int kRowNormThreads = 256;
constexpr int kRowNormMaxCols = 32;  // per thread: d_model <= 8192

__global__ void __launch_bounds__(kRowNormThreads) hidden_norm_rows_kernel(
    const GemmOut y, const uint16_t *gamma, uint16_t *hn, int D, float eps,
    const int32_t *ctx_len, int32_t *ctx_snap, int B) {
  __shared__ float red[32];
  griddep_launch();
  griddep_wait();
  const int n = blockIdx.x, tid = threadIdx.x;
  if (n == 0)
    for (int r = tid; r < B; r += kRowNormThreads) ctx_snap[r] = ctx_len[r];
  const int nt = n / y.ntile, nr = n - nt * y.ntile;
  const int per = (D + kRowNormThreads - 1) / kRowNormThreads;
  float h[kRowNormMaxCols];
  float ss = 0.f;
#pragma unroll
  for (int b0 = 0; b0 < kRowNormMaxCols; b0 += 8) {
    if (b0 < per) {
      GemmOutLoad ld[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int col = (b0 + k) * kRowNormThreads + tid;
        const unsigned t = static_cast<unsigned>(nt) * y.mtiles + static_cast<unsigned>(col >> 7);
        gemm_out_issue(y, t, (b0 + k < per && col < D) ? gemm_tile_parts(y, t) : 0, nr, col & 127,
                       ld[k]);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float v = bf16_to_f32(f32_to_bf16_rn(gemm_out_finish(y, ld[k])));
        h[b0 + k] = v;
        ss += v * v;
      }
    }
  }
  const float tot = block_sum(ss, red);
  const float inv = rsqrtf(tot / static_cast<float>(D) + eps);
#pragma unroll
  for (int k = 0; k < kRowNormMaxCols; ++k) {
    const int col = k * kRowNormThreads + tid;
    if (k < per && col < D)
      hn[static_cast<size_t>(n) * D + col] = f32_to_bf16_rn(h[k] * inv * bf16_to_f32(gamma[col]));
  }
}

// ----------------------------------------------------------- write mask
struct MaskArgs {
  const int32_t *n_acc;
  const int32_t *ctx_snap;
  const int32_t *alloc_limit;
  const int32_t *tbl;
  const uint8_t *valid;
  const int32_t *cu_rows;  // prefill: request r owns rows cu_rows[r] .. cu_rows[r+1]-1
  int T, M, P, NP, B;
  int32_t *st;
};

// Request and in-request index of GEMM row n: (n / T, n % T) for the decode
// update, a binary search of cu_rows for the prefill store.  False when the
// prefill row lies in no request's range (cu_rows inconsistent with the row
// count; the row is skipped).
__device__ __forceinline__ bool row_of(const MaskArgs &m, int n, int *r, int *i) {
  if (!m.cu_rows) {
    *r = n / m.T;
    *i = n % m.T;
    return true;
  }
  int lo = 0, hi = m.B - 1;  // the last request whose first row is <= n
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (m.cu_rows[mid] <= n) lo = mid; else hi = mid - 1;
  }
  const int a = m.cu_rows[lo], b = m.cu_rows[lo + 1];
  *r = lo;
  *i = n - a;
  return n >= a && n < b;
}

// Destination of context row (r, i), or false when the row is not written.
__device__ __forceinline__ bool ctx_row_dest(const MaskArgs &m, int r, int i, int *page, int *slot,
                                             int *pos, bool report) {
  // the row's scalars are independent loads, issued together
  const int n = m.cu_rows ? i + 1 : m.n_acc[r];  // prefill: every row of the request
  const int c = m.ctx_snap[r];
  const int A = m.alloc_limit[r];
  const bool live = m.valid ? (m.valid[r] != 0) : true;
  if (!live || n < 1 || (!m.cu_rows && n > m.T) || c < 0 || i >= n) return false;
  const int p = c + i;
  if (p >= A) return false;
  const int lp = p / m.P;
  if (lp >= m.M) return false;
  const int pg = m.tbl[static_cast<int64_t>(r) * m.M + lp];
  if (pg < 0) return false;
  if (pg >= m.NP) {
    if (report) raise_status(m.st, DFLASH_DEV_BAD_PAGE);
    return false;
  }
  *page = pg;
  *slot = p % m.P;
  *pos = p;
  return true;
}

// Advance of ctx_len[r] from the pre-step length c (the snapshot).
__device__ __forceinline__ void advance_ctx_len(const MaskArgs &m, int32_t *ctx_len, int B) {
  for (int r = threadIdx.x; r < B; r += blockDim.x) {
    const int c = m.ctx_snap[r];
    if (m.cu_rows) {  // prefill: all of the request's rows
      const int nn = max(0, m.cu_rows[r + 1] - m.cu_rows[r]);
      const bool live = (m.valid ? (m.valid[r] != 0) : true) && c >= 0;
      const long long s = static_cast<long long>(c) + nn;
      const int A = m.alloc_limit[r];
      ctx_len[r] = live ? static_cast<int>(s < A ? s : A) : 0;
      continue;
    }
    const int nn = m.n_acc[r];
    const bool live = (m.valid ? (m.valid[r] != 0) : true) && nn >= 1 && nn <= m.T && c >= 0;
    const long long s = static_cast<long long>(c) + nn;
    const int A = m.alloc_limit[r];
    ctx_len[r] = live ? static_cast<int>(s < A ? s : A) : 0;
  }
}

// ------------------------------------------------------ GQA epilogue
// grid (N rows, L*2*nkv heads), block = head_dim / 2 threads rounded up to a
// warp: thread t holds columns t and t + hd/2 of the head -- a rotate-half
// pair, so one cos/sin serves both and RoPE needs no exchange.  kStaged =
// false: the fused update (write-masked paged store, ctx_len advance).
// kStaged = true: the projection half of a split update -- every row, RoPE at
// c + i, the bf16 values to staged[n][col] (no mask, no store to the pool).
template <bool kStaged>
__global__ void epilogue_gqa_kernel(const GemmOut y, const MaskArgs m, const RopeFreqs rf,
                                    const uint16_t *gamma_k, uint16_t *pool, uint16_t *staged,
                                    int L, int nkv, int hd, float eps, int32_t *ctx_len, int B) {
  __shared__ float red[32];
  __shared__ __align__(16) uint16_t obuf[kMaxHeadDim];  // the bf16 row, stored as 16-byte vectors
  griddep_launch();
  griddep_wait();
  const int n = blockIdx.x;
  const int head = blockIdx.y;  // ((l * 2 + kv) * nkv + h)
  const int t = threadIdx.x, half = hd >> 1;
  const bool act = t < half;
  // the Y2 loads go out first, overlapping the destination lookup
  GemmOutLoad ld0, ld1;
  {
    const int c0 = head * hd + (act ? t : 0), c1 = c0 + half;
    const int nt = n / y.ntile, nr = n - nt * y.ntile;
    const unsigned t0 = static_cast<unsigned>(nt) * y.mtiles + (c0 >> 7);
    const unsigned t1 = static_cast<unsigned>(nt) * y.mtiles + (c1 >> 7);
    gemm_out_issue(y, t0, act ? gemm_tile_parts(y, t0) : 0, nr, c0 & 127, ld0);
    gemm_out_issue(y, t1, act ? gemm_tile_parts(y, t1) : 0, nr, c1 & 127, ld1);
  }
  // ctx_len advance; every reader of the pre-step value uses the snapshot
  if (!kStaged && n == 0 && head == 0) advance_ctx_len(m, ctx_len, B);
  int r, i;
  if (!row_of(m, n, &r, &i)) return;
  int page = 0, slot = 0, pos;
  if (kStaged) {
    pos = m.ctx_snap[r] + i;
  } else if (!ctx_row_dest(m, r, i, &page, &slot, &pos, head == 0 && t == 0)) {
    return;
  }
  const int l = head / (2 * nkv);
  const int kv = (head / nkv) & 1;
  const int h = head % nkv;
  float v0 = gemm_out_finish(y, ld0), v1 = gemm_out_finish(y, ld1);
  if (kv == 0) {
    const float ss = block_sum(act ? v0 * v0 + v1 * v1 : 0.f, red);
    const float inv = rsqrtf(ss / static_cast<float>(hd) + eps);
    if (act) {
      const float k0 = v0 * inv * bf16_to_f32(gamma_k[static_cast<size_t>(l) * hd + t]);
      const float k1 = v1 * inv * bf16_to_f32(gamma_k[static_cast<size_t>(l) * hd + t + half]);
      float c, s;
      rope_cos_sin(pos, rf.f[t], &c, &s);
      v0 = k0 * c - k1 * s;
      v1 = k1 * c + k0 * s;
    }
  }
  if (act) {
    obuf[t] = f32_to_bf16_rn(v0);
    obuf[t + half] = f32_to_bf16_rn(v1);
  }
  __syncthreads();
  if (t < hd / 8) {  // head_dim % 8 == 0: the row leaves as 16-byte vectors
    uint16_t *row =
        kStaged ? staged + static_cast<size_t>(n) * L * 2 * nkv * hd + head * hd
                : pool + ((((static_cast<size_t>(l) * m.NP + page) * 2 + kv) * nkv + h) * m.P +
                          slot) * hd;
    reinterpret_cast<uint4 *>(row)[t] = reinterpret_cast<const uint4 *>(obuf)[t];
  }
}

// ------------------------------------------------------ MLA epilogue
// grid (N rows, L), block = lat / 2 + rope / 2 threads rounded up to a warp:
// thread t < lat/2 holds latent columns t and t + lat/2; thread lat/2 + j
// holds the rope pair j, j + rope/2.  kStaged as for GQA.
template <bool kStaged>
__global__ void epilogue_mla_kernel(const GemmOut y, const MaskArgs m, const RopeFreqs rf,
                                    const uint16_t *gamma_kv, uint16_t *pool, uint16_t *staged,
                                    int L, int lat, int rope, float eps, int32_t *ctx_len, int B) {
  __shared__ float red[32];
  __shared__ __align__(16) uint16_t obuf[1024];  // lat + rope <= 1024
  griddep_launch();
  griddep_wait();
  const int n = blockIdx.x;
  const int l = blockIdx.y;
  const int t = threadIdx.x;
  const int W = lat + rope, hl = lat >> 1, hr = rope >> 1;
  const bool is_lat = t < hl, is_rope = !is_lat && t < hl + hr;
  const int ca = is_lat ? t : (is_rope ? lat + (t - hl) : 0);
  const int cb = is_lat ? t + hl : ca + hr;
  GemmOutLoad ld0, ld1;
  {
    const int nt = n / y.ntile, nr = n - nt * y.ntile;
    const int g0 = l * W + ca, g1 = l * W + cb;
    const unsigned t0 = static_cast<unsigned>(nt) * y.mtiles + (g0 >> 7);
    const unsigned t1 = static_cast<unsigned>(nt) * y.mtiles + (g1 >> 7);
    const bool act = is_lat || is_rope;
    gemm_out_issue(y, t0, act ? gemm_tile_parts(y, t0) : 0, nr, g0 & 127, ld0);
    gemm_out_issue(y, t1, act ? gemm_tile_parts(y, t1) : 0, nr, g1 & 127, ld1);
  }
  if (!kStaged && n == 0 && l == 0) advance_ctx_len(m, ctx_len, B);
  int r, i;
  if (!row_of(m, n, &r, &i)) return;
  int page = 0, slot = 0, pos;
  if (kStaged) {
    pos = m.ctx_snap[r] + i;
  } else if (!ctx_row_dest(m, r, i, &page, &slot, &pos, l == 0 && t == 0)) {
    return;
  }
  const float v0 = gemm_out_finish(y, ld0), v1 = gemm_out_finish(y, ld1);
  const float ss = block_sum(is_lat ? v0 * v0 + v1 * v1 : 0.f, red);
  float o0 = 0.f, o1 = 0.f;
  if (is_lat) {
    const float inv = rsqrtf(ss / static_cast<float>(lat) + eps);
    o0 = v0 * inv * bf16_to_f32(gamma_kv[static_cast<size_t>(l) * lat + ca]);
    o1 = v1 * inv * bf16_to_f32(gamma_kv[static_cast<size_t>(l) * lat + cb]);
  } else if (is_rope) {
    float c, s;
    rope_cos_sin(pos, rf.f[t - hl], &c, &s);
    o0 = v0 * c - v1 * s;
    o1 = v1 * c + v0 * s;
  }
  if (is_lat || is_rope) {
    obuf[ca] = f32_to_bf16_rn(o0);
    obuf[cb] = f32_to_bf16_rn(o1);
  }
  __syncthreads();
  if (t < W / 8) {  // (lat + rope) % 8 == 0: the row leaves as 16-byte vectors
    uint16_t *row = kStaged ? staged + static_cast<size_t>(n) * L * W + static_cast<size_t>(l) * W
                            : pool + ((static_cast<size_t>(l) * m.NP + page) * m.P + slot) * W;
    reinterpret_cast<uint4 *>(row)[t] = reinterpret_cast<const uint4 *>(obuf)[t];
  }
}

// ------------------------------------------------------------ commit
// The store half of a split update: staged rows -> pool at the write-masked
// rows, then the ctx_len advance, both from the pre-step lengths the
// projection recorded (so no CTA reads ctx_len while another writes it).
// grid (N rows, L), 16-byte vectors of one layer's K and V rows (or latent).
__global__ void commit_kernel(const uint4 *staged, const MaskArgs m, uint16_t *pool, int kind,
                              int L, int nkv, int hd, int W, int32_t *ctx_len, int B) {
  griddep_launch();
  griddep_wait();
  const int n = blockIdx.x, l = blockIdx.y;
  if (n == 0 && l == 0) advance_ctx_len(m, ctx_len, B);
  int r, i;
  row_of(m, n, &r, &i);
  int page, slot, pos;
  if (!ctx_row_dest(m, r, i, &page, &slot, &pos, l == 0 && threadIdx.x == 0)) return;
  const bool gqa = kind == DFLASH_KIND_GQA;
  const int vph = hd / 8;                            // vectors per head row (GQA)
  const int lv = gqa ? 2 * nkv * vph : W / 8;        // vectors of one layer's row
  const uint4 *src = staged + (static_cast<size_t>(n) * L + l) * lv;
  uint4 *base = reinterpret_cast<uint4 *>(pool);
  for (int t = threadIdx.x; t < lv; t += blockDim.x) {
    size_t dst;
    if (gqa) {
      const int kv = t / (nkv * vph);
      const int rem = t - kv * nkv * vph;
      const int h = rem / vph, e = rem % vph;
      dst = ((((static_cast<size_t>(l) * m.NP + page) * 2 + kv) * nkv + h) * m.P + slot) * vph + e;
    } else {
      dst = ((static_cast<size_t>(l) * m.NP + page) * m.P + slot) * (W / 8) + t;
    }
    base[dst] = src[t];
  }
}

}  // namespace

size_t ctx_workspace_bytes(const dflash_geom &g, int B) { return ctx_ws_map(g, B, nullptr).bytes; }

namespace {

// The launch chain prep -> fc GEMM -> hidden norm -> K/V GEMM -> epilogue.
// staged == nullptr: the fused update.  Otherwise the projection half of a
// split update: the norm records the pre-step ctx_len in staged_c and the
// epilogue writes every row's values to staged (mask arguments unused).
cudaError_t launch_ctx_chain(const dflash_geom &g, int B, const void *hidden, int hidden_dtype,
                             const int32_t *n_acc, int32_t *ctx_len, const int32_t *alloc_limit,
                             const int32_t *tbl, const uint8_t *valid, const dflash_weights &w,
                             void *pool, void *ws, int32_t *st, int32_t *staged_c,
                             uint16_t *staged, cudaStream_t s, int rows = -1,
                             const int32_t *cu_rows = nullptr) {
  const int N = rows >= 0 ? rows : B * g.block_size;
  const CtxDims d = ctx_dims_rows(g, N);
  const CtxWs W = ctx_ws_map_rows(g, B, N, ws);
  const bool split = staged != nullptr;
  int32_t *snap = split ? staged_c : W.ctx_snap;
  cudaError_t e;

  // prep: fp32 hidden -> bf16
  const bool f32 = hidden_dtype == DFLASH_DTYPE_F32;
  if (f32) {
    const int threads = 256;
    int blocks = (d.Npad * d.D_in + threads - 1) / threads;
    if (blocks > 4 * device_sm_count()) blocks = 4 * device_sm_count();
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(threads);
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((e = cudaLaunchKernelEx(&cfg, prep_kernel, static_cast<const float *>(hidden), W.x,
                                d.N * d.D_in, d.D_in, d.Npad)) != cudaSuccess)
      return e;
  }
  const uint16_t *X = f32 ? W.x : static_cast<const uint16_t *>(hidden);

  // fc GEMM
  GemmOut y1, y2;
  if ((e = launch_gemm(X, d.N, d.D_in, static_cast<const uint16_t *>(w.w_fc), d.D, W.part1, st,
                       /*pdl=*/true, s, &y1)) != cudaSuccess)
    return e;

  // hidden RMSNorm: a cluster of G CTAs per row for decode-sized row counts,
  // one CTA per row beyond (prefill)
  if (d.N > kClusterNormMaxRows) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(d.N);
    cfg.blockDim = dim3(kRowNormThreads);
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (d.D > kRowNormThreads * kRowNormMaxCols) return cudaErrorInvalidValue;
    if ((e = cudaLaunchKernelEx(&cfg, hidden_norm_rows_kernel, y1,
                                static_cast<const uint16_t *>(w.gamma_h), W.hn, d.D,
                                static_cast<float>(g.eps_hidden),
                                static_cast<const int32_t *>(ctx_len), snap, B)) != cudaSuccess)
      return e;
  } else {
    int G = (d.D + 511) / 512;
    if (G > 8) G = 8;
    const int cols = (d.D + G - 1) / G;  // <= kNormMaxCols, as d_model <= 8192
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.gridDim = dim3(G, d.N);
    cfg.blockDim = dim3(kNormThreads);
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = G;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (cols > kNormMaxCols) return cudaErrorInvalidValue;
    if ((e = cudaLaunchKernelEx(&cfg, hidden_norm_kernel, y1,
                                static_cast<const uint16_t *>(w.gamma_h), W.hn, d.D, cols,
                                static_cast<float>(g.eps_hidden), static_cast<const int32_t *>(ctx_len),
                                snap, B)) != cudaSuccess)
      return e;
  }

  // stacked K/V (or latent) GEMM over every layer
  if ((e = launch_gemm(W.hn, d.N, d.D, static_cast<const uint16_t *>(w.w_kv), d.Wrows, W.part2, st,
                       /*pdl=*/true, s, &y2)) != cudaSuccess)
    return e;

  // epilogue
  MaskArgs m;
  m.n_acc = n_acc;
  m.ctx_snap = snap;
  m.alloc_limit = alloc_limit;
  m.tbl = tbl;
  m.valid = valid;
  m.cu_rows = cu_rows;
  m.T = g.block_size;
  m.M = g.max_pages;
  m.P = g.page_size;
  m.NP = g.num_pool_pages;
  m.B = B;
  m.st = st;
  RopeFreqs rf;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.stream = s;
  uint16_t *pool16 = static_cast<uint16_t *>(pool);
  if (g.kind == DFLASH_KIND_GQA) {
    fill_rope_freqs(&rf, g.head_dim, g.rope_theta);
    cfg.gridDim = dim3(d.N, g.num_layers * 2 * g.nkv);
    cfg.blockDim = dim3(std::max(32, (g.head_dim / 2 + 31) / 32 * 32));
    e = cudaLaunchKernelEx(&cfg, split ? epilogue_gqa_kernel<true> : epilogue_gqa_kernel<false>, y2,
                           m, rf, static_cast<const uint16_t *>(w.gamma_k), pool16, staged,
                           g.num_layers, g.nkv, g.head_dim, static_cast<float>(g.eps_k), ctx_len, B);
  } else {
    fill_rope_freqs(&rf, g.rope_dim, g.rope_theta);
    cfg.gridDim = dim3(d.N, g.num_layers);
    cfg.blockDim = dim3((g.latent_dim / 2 + g.rope_dim / 2 + 31) / 32 * 32);
    e = cudaLaunchKernelEx(&cfg, split ? epilogue_mla_kernel<true> : epilogue_mla_kernel<false>, y2,
                           m, rf, static_cast<const uint16_t *>(w.gamma_k), pool16, staged,
                           g.num_layers, g.latent_dim, g.rope_dim, static_cast<float>(g.eps_k),
                           ctx_len, B);
  }
  return e;
}

// staged buffer: int32 pre-step ctx_len [B], then bf16 rows [B * T][Wrows]
size_t staged_rows_offset(int B) { return align_up(sizeof(int32_t) * (B > 0 ? B : 1), 256); }

}  // namespace

cudaError_t launch_ctx_kv_update(const dflash_geom &g, int B, const void *hidden, int hidden_dtype,
                                 const int32_t *n_acc, int32_t *ctx_len, const int32_t *alloc_limit,
                                 const int32_t *tbl, const uint8_t *valid, const dflash_weights &w,
                                 void *pool, void *ws, int32_t *st, cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  return launch_ctx_chain(g, B, hidden, hidden_dtype, n_acc, ctx_len, alloc_limit, tbl, valid, w,
                          pool, ws, st, nullptr, nullptr, s);
}

size_t ctx_prefill_workspace_bytes(const dflash_geom &g, int B, int rows) {
  return ctx_ws_map_rows(g, B, rows, nullptr).bytes;
}

cudaError_t launch_ctx_kv_prefill(const dflash_geom &g, int B, int rows, const void *hidden,
                                  int hidden_dtype, const int32_t *cu_rows, int32_t *ctx_len,
                                  const int32_t *alloc_limit, const int32_t *tbl,
                                  const uint8_t *valid, const dflash_weights &w, void *pool,
                                  void *ws, int32_t *st, cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  return launch_ctx_chain(g, B, hidden, hidden_dtype, nullptr, ctx_len, alloc_limit, tbl, valid, w,
                          pool, ws, st, nullptr, nullptr, s, rows, cu_rows);
}

size_t ctx_staged_bytes(const dflash_geom &g, int B) {
  const CtxDims d = ctx_dims(g, B);
  return staged_rows_offset(B) + sizeof(uint16_t) * static_cast<size_t>(d.N) * d.Wrows;
}

cudaError_t launch_ctx_kv_project(const dflash_geom &g, int B, const void *hidden, int hidden_dtype,
                                  const int32_t *ctx_len, const dflash_weights &w, void *staged,
                                  void *ws, int32_t *st, cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  char *sb = static_cast<char *>(staged);
  return launch_ctx_chain(g, B, hidden, hidden_dtype, nullptr, const_cast<int32_t *>(ctx_len),
                          nullptr, nullptr, nullptr, w, nullptr, ws, st,
                          reinterpret_cast<int32_t *>(sb),
                          reinterpret_cast<uint16_t *>(sb + staged_rows_offset(B)), s);
}

cudaError_t launch_ctx_kv_commit(const dflash_geom &g, int B, const void *staged,
                                 const int32_t *n_acc, int32_t *ctx_len, const int32_t *alloc_limit,
                                 const int32_t *tbl, const uint8_t *valid, void *pool, int32_t *st,
                                 cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  const CtxDims d = ctx_dims(g, B);
  const char *sb = static_cast<const char *>(staged);
  MaskArgs m;
  m.n_acc = n_acc;
  m.ctx_snap = reinterpret_cast<const int32_t *>(sb);
  m.alloc_limit = alloc_limit;
  m.tbl = tbl;
  m.valid = valid;
  m.cu_rows = nullptr;
  m.T = g.block_size;
  m.M = g.max_pages;
  m.P = g.page_size;
  m.NP = g.num_pool_pages;
  m.B = B;
  m.st = st;
  const bool gqa = g.kind == DFLASH_KIND_GQA;
  const int W = g.latent_dim + g.rope_dim;
  const int lv = gqa ? 2 * g.nkv * (g.head_dim / 8) : W / 8;
  int threads = lv < 256 ? ((lv + 31) / 32) * 32 : 256;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(d.N, g.num_layers);
  cfg.blockDim = dim3(threads);
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, commit_kernel,
                            reinterpret_cast<const uint4 *>(sb + staged_rows_offset(B)), m,
                            static_cast<uint16_t *>(pool), static_cast<int>(g.kind), g.num_layers,
                            g.nkv, g.head_dim, W, ctx_len, B);
}

}  // namespace dflash
