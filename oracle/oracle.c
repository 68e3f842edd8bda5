/*
 * oracle.c -- plain, slow CPU oracle of the DFlash/DSpark drafter decode-step
 * hot path.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg are the only callers.  The product path never
 * links, loads or calls this file; it shares no code, header, table or helper
 * with the CUDA library.
 *
 * Every floating-point reduction accumulates in double.  bf16 values are
 * widened exactly; a value is rounded to bf16 only at the rounding points the
 * method defines (listed on each function).  Loops are written in the order
 * of the definitions, with no blocking, fusion or reordering.
 *
 * Sources (page title, part of the page):
 *  - TensorRT-LLM issue #20548 "DFlash / MLA DSpark decode spends ~0.2 ms per
 *    step in small bookkeeping kernels", Proposal: the bookkeeping groups.
 *  - TensorRT-LLM PR #20550, Description (TLLM_DFLASH_FUSED_PROLOGUE) and the
 *    follow-up commit "spec_tail_kernels.py": block-table decode (offsets
 *    clamped, then divided), bonus token, query / RoPE positions, destination
 *    pages / offsets / write mask, ctx_len advance with the dummy slot
 *    emptied, advertised context length, seq_lens, DraftBlockPlacement.
 *  - TensorRT-LLM PR #13995 "DFlash performance optimizations", commits
 *    "migrate draft path to per-layer cached K/V pool" (one stacked GEMM over
 *    the drafter layers), "match RoPE between context and query", "fuse
 *    cross-layer k_norm and avoid mask-mul alloc" (one RMSNorm over
 *    [N, L, nkv, hd] with stacked per-layer weights, shared eps).
 *  - vLLM PR #54092, Purpose item 2 and Changes item 2: split-KV over
 *    segments for small uniform q, sliding window with per-head sinks, the
 *    segments over the keys the window leaves visible, the reduce over them.
 *
 * Readings where the pages are silent:
 *  - n_pages counts the non-negative raw offsets of a row; the decoded table
 *    is max(offset, 0) / div with floor division.
 *  - alloc limit A = min(max_ctx, n_pages * P); advance c' = min(c + n, A).
 *  - a row is a dummy when valid == 0, n is outside [1, T] or c < 0: all its
 *    masks are 0, positions 0, ids mask_id, c' = 0, seq_len = 0, n_pages = 0.
 *  - rounding points of the update: x -> bf16, h = bf16(W_fc x),
 *    hn = bf16(h * g_h / rms(h)); K/V projection unrounded; k-norm and RoPE
 *    in full precision; stored values rounded to bf16 once.
 *  - RoPE is the rotate-half (NeoX) pairing, f_j = theta^(-2j/rot_dim).
 *  - sinks are per-head logits that join the softmax denominator only.
 *  - CAUSAL_TAIL: query i of Tq sits at p_i = kv_len - Tq + i and sees keys
 *    j <= p_i; BLOCK_BIDIR: it sees every key j < kv_len.  A window W > 0
 *    further restricts to p_i - j < W.  An empty key set yields 0.
 *  - split update: the projection covers every row of the block at c + i
 *    and records c; the commit masks and advances from the recorded c.
 *  - the query norm uses the key norm's eps; MLA rotates only the rope part.
 *  - strict acceptance compares each draft with the target's token at the
 *    same position; the first mismatch (or the position after the last
 *    draft) supplies the bonus, accepted[n - 1].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_MASK_CAUSAL_TAIL 0
#define OR_MASK_BLOCK_BIDIR 1

/* device-status style flags reported by the oracle bookkeeping */
#define OR_ST_BAD_NACCEPTED 1
#define OR_ST_BAD_CTX_LEN 2
#define OR_ST_CTX_OUTRUN 4
#define OR_ST_BAD_PAGE 8

/* ------------------------------------------------------------------ bf16 */

double oracle_bf16_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Round to nearest even: double -> float (RNE), then float -> bf16 (RNE). */
uint16_t oracle_double_to_bf16(double x) {
  float f = (float)x;
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7f800000u) == 0x7f800000u) {
    uint16_t hi = (uint16_t)(u >> 16);
    if (u & 0x007fffffu) hi |= 0x0040u; /* keep NaN a NaN */
    return hi;
  }
  uint32_t keep_lsb = (u >> 16) & 1u;
  u += 0x7fffu + keep_lsb;
  return (uint16_t)(u >> 16);
}

static double round_bf16(double x) { return oracle_bf16_to_double(oracle_double_to_bf16(x)); }

/* ------------------------------------------------------- building blocks */

/* y[m] = sum_k W[m, k] * x[k], W row-major [Mrows, K] bf16, x double. */
void oracle_matvec_bf16(const uint16_t *W, int Mrows, int K, const double *x, double *y) {
  for (int m = 0; m < Mrows; ++m) {
    double acc = 0.0;
    const uint16_t *row = W + (size_t)m * K;
    for (int k = 0; k < K; ++k) acc += oracle_bf16_to_double(row[k]) * x[k];
    y[m] = acc;
  }
}

/* out = x * g / sqrt(mean(x^2) + eps)   (RMSNorm with gain g; g may be NULL = 1) */
void oracle_rmsnorm(const double *x, const double *g, int n, double eps, double *out) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  double inv = 1.0 / sqrt(ss / (double)n + eps);
  for (int i = 0; i < n; ++i) out[i] = x[i] * inv * (g ? g[i] : 1.0);
}

/* Rotate-half RoPE over n (even) dims at position pos:
 *   f_j = theta^(-2j/n), a = pos * f_j,
 *   out[j]       = x[j] cos a - x[j+n/2] sin a
 *   out[j + n/2] = x[j+n/2] cos a + x[j] sin a            (j < n/2) */
void oracle_rope_neox(const double *x, int n, double pos, double theta, double *out) {
  int half = n / 2;
  for (int j = 0; j < half; ++j) {
    double f = pow(theta, -2.0 * (double)j / (double)n);
    double a = pos * f;
    double c = cos(a), s = sin(a);
    double x0 = x[j], x1 = x[j + half];
    out[j] = x0 * c - x1 * s;
    out[j + half] = x1 * c + x0 * s;
  }
}

/* ----------------------------------------------------------- bookkeeping */

/* Block-table decode, gen-request prologue, write mask / destinations,
 * ctx_len advance and block placement for B requests (all int32, exact).
 * off: raw offsets [B, M] with row stride off_stride (elements).
 * acc: accepted tokens [B, T] with row stride acc_stride.
 * valid may be NULL (every row live).  Outputs are dense [B] / [B, T] /
 * [B, M].  Returns the OR of the status flags raised. */
int oracle_bookkeeping(int B, int T, int M, int P, int off_div, int max_ctx, int mask_id,
                       const int32_t *off, int64_t off_stride, const int32_t *acc,
                       int64_t acc_stride, const int32_t *n_acc, const int32_t *ctx_pre,
                       const uint8_t *valid, int32_t *n_pages, int32_t *tbl,
                       int32_t *alloc_limit, int32_t *bonus, int32_t *emb, int32_t *ctx_pos,
                       int32_t *q_pos, int32_t *dst_page, int32_t *dst_slot, uint8_t *wmask,
                       int32_t *blk_page, int32_t *blk_slot, uint8_t *blk_mask,
                       int32_t *ctx_new, int32_t *seq_lens) {
  int status = 0;
  for (int r = 0; r < B; ++r) {
    const int32_t *orow = off + (int64_t)r * off_stride;
    const int32_t *arow = acc + (int64_t)r * acc_stride;
    int n = n_acc[r];
    int c = ctx_pre[r];
    int live = valid ? (valid[r] != 0) : 1;
    int ok = live;
    if (live && (n < 1 || n > T)) { status |= OR_ST_BAD_NACCEPTED; ok = 0; }
    if (live && c < 0) { status |= OR_ST_BAD_CTX_LEN; ok = 0; }

    /* block-table decode: count of non-negative offsets, clamp-and-divide */
    int count = 0;
    for (int j = 0; j < M; ++j) {
      int v = orow[j];
      if (v >= 0) count += 1;
      tbl[(int64_t)r * M + j] = (v > 0 ? v : 0) / off_div;
    }
    int np = ok ? count : 0;
    n_pages[r] = np;
    long long cap = (long long)np * P;
    int A = ok ? (int)(cap < max_ctx ? cap : max_ctx) : 0;
    alloc_limit[r] = A;

    int b = ok ? arow[n - 1] : mask_id;
    bonus[r] = b;
    for (int i = 0; i < T; ++i) emb[(int64_t)r * T + i] = (i == 0) ? b : mask_id;

    /* context rows */
    for (int i = 0; i < T; ++i) {
      int64_t k = (int64_t)r * T + i;
      int p = ok ? c + i : 0;
      ctx_pos[k] = p;
      int w = 0;
      if (ok && i < n && p < A) {
        int lp = p / P;
        if (lp < M && orow[lp] >= 0) w = 1;
      }
      wmask[k] = (uint8_t)w;
      dst_page[k] = w ? tbl[(int64_t)r * M + p / P] : -1;
      dst_slot[k] = w ? p % P : -1;
    }

    /* advance and advertised length */
    int cn = 0;
    if (ok) {
      long long s = (long long)c + n;
      cn = (int)(s < A ? s : A);
      if (c > A) status |= OR_ST_CTX_OUTRUN;
    }
    ctx_new[r] = cn;
    seq_lens[r] = ok ? cn + T : 0;

    /* block placement for the block's own positions */
    for (int i = 0; i < T; ++i) {
      int64_t k = (int64_t)r * T + i;
      int p = ok ? cn + i : 0;
      q_pos[k] = p;
      int w = 0;
      if (ok && (long long)p < cap) {
        int lp = p / P;
        if (lp < M && orow[lp] >= 0) w = 1;
      }
      blk_mask[k] = (uint8_t)w;
      blk_page[k] = w ? tbl[(int64_t)r * M + p / P] : -1;
      blk_slot[k] = w ? p % P : -1;
    }
  }
  return status;
}

/* ---------------------------------------------------- context-KV update */

static int row_valid(const uint8_t *valid, int r, int n, int c, int T) {
  int live = valid ? (valid[r] != 0) : 1;
  return live && n >= 1 && n <= T && c >= 0;
}

/* Write mask of context row i of request r, and its physical page. */
static int ctx_row_dest(int ok, int i, int n, int c, int A, const int32_t *tbl_row, int M, int P,
                        int num_pool_pages, int *page, int *slot) {
  if (!ok || i >= n) return 0;
  int p = c + i;
  if (p >= A) return 0;
  int lp = p / P;
  if (lp >= M) return 0;
  int pg = tbl_row[lp];
  if (pg < 0 || pg >= num_pool_pages) return 0;
  *page = pg;
  *slot = p % P;
  return 1;
}

/* x (one hidden row) -> hn = bf16(bf16(W_fc x) * g_h / rms), as doubles. */
static void fc_hidden_norm(const void *hidden_row, int hidden_is_f32, int D_in, int D,
                           const uint16_t *w_fc, const uint16_t *g_h, double eps_h, double *x,
                           double *h, double *g, double *hn) {
  for (int k = 0; k < D_in; ++k) {
    double v = hidden_is_f32 ? (double)((const float *)hidden_row)[k]
                             : oracle_bf16_to_double(((const uint16_t *)hidden_row)[k]);
    x[k] = round_bf16(v);
  }
  oracle_matvec_bf16(w_fc, D, D_in, x, h);
  for (int d = 0; d < D; ++d) {
    h[d] = round_bf16(h[d]);
    g[d] = oracle_bf16_to_double(g_h[d]);
  }
  oracle_rmsnorm(h, g, D, eps_h, hn);
  for (int d = 0; d < D; ++d) hn[d] = round_bf16(hn[d]);
}

/* Exposed for the tests: hn rows (bf16 bits) for every hidden row. */
void oracle_fc_hidden_norm(int rows, const void *hidden, int hidden_is_f32, int D_in, int D,
                           const uint16_t *w_fc, const uint16_t *g_h, double eps_h,
                           uint16_t *hn_out) {
  double *x = malloc(sizeof(double) * D_in);
  double *h = malloc(sizeof(double) * D);
  double *g = malloc(sizeof(double) * D);
  double *hn = malloc(sizeof(double) * D);
  size_t esz = hidden_is_f32 ? 4 : 2;
  for (int r = 0; r < rows; ++r) {
    const char *row = (const char *)hidden + (size_t)r * D_in * esz;
    fc_hidden_norm(row, hidden_is_f32, D_in, D, w_fc, g_h, eps_h, x, h, g, hn);
    for (int d = 0; d < D; ++d) hn_out[(size_t)r * D + d] = oracle_double_to_bf16(hn[d]);
  }
  free(x); free(h); free(g); free(hn);
}

/* GQA context-KV update.
 * hidden [B, T, D_in] (fp32 when hidden_is_f32 else bf16), w_fc [D, D_in],
 * g_h [D], w_kv [L, 2, nkv, hd, D] (k rows then v rows per layer), g_k [L, hd],
 * tbl [B, M] (entry < 0: unmapped), pool [L][NP][2][nkv][P][hd] bf16 (updated
 * in place at the write-masked rows only), ctx_out[r] = advanced ctx_len. */
int oracle_ctx_kv_update_gqa(int B, int T, int L, int D_in, int D, int nkv, int hd, int P, int M,
                             int num_pool_pages, double theta, double eps_h, double eps_k,
                             const void *hidden, int hidden_is_f32, const int32_t *n_acc,
                             const int32_t *ctx_in, int32_t *ctx_out, const int32_t *alloc_limit,
                             const int32_t *tbl, const uint8_t *valid, const uint16_t *w_fc,
                             const uint16_t *g_h, const uint16_t *w_kv, const uint16_t *g_k,
                             uint16_t *pool) {
  size_t esz = hidden_is_f32 ? 4 : 2;
#pragma omp parallel
  {
    double *x = malloc(sizeof(double) * D_in);
    double *h = malloc(sizeof(double) * D);
    double *g = malloc(sizeof(double) * D);
    double *hn = malloc(sizeof(double) * D);
    double *t = malloc(sizeof(double) * hd);
    double *kn = malloc(sizeof(double) * hd);
    double *kr = malloc(sizeof(double) * hd);
    double *gk = malloc(sizeof(double) * hd);
#pragma omp for schedule(dynamic, 1)
    for (int rt = 0; rt < B * T; ++rt) {
      int r = rt / T, i = rt % T;
      int n = n_acc[r], c = ctx_in[r];
      int ok = row_valid(valid, r, n, c, T);
      int page, slot;
      if (!ctx_row_dest(ok, i, n, c, alloc_limit[r], tbl + (int64_t)r * M, M, P,
                        num_pool_pages, &page, &slot))
        continue;
      const char *row = (const char *)hidden + (size_t)rt * D_in * esz;
      fc_hidden_norm(row, hidden_is_f32, D_in, D, w_fc, g_h, eps_h, x, h, g, hn);
      double pos = (double)(c + i);
      for (int l = 0; l < L; ++l) {
        for (int d = 0; d < hd; ++d) gk[d] = oracle_bf16_to_double(g_k[(size_t)l * hd + d]);
        for (int kv = 0; kv < 2; ++kv) {
          for (int hh = 0; hh < nkv; ++hh) {
            const uint16_t *W = w_kv + ((((size_t)l * 2 + kv) * nkv + hh) * hd) * (size_t)D;
            oracle_matvec_bf16(W, hd, D, hn, t);
            uint16_t *dst =
                pool + (((((size_t)l * num_pool_pages + page) * 2 + kv) * nkv + hh) * P + slot) *
                           (size_t)hd;
            if (kv == 0) {
              oracle_rmsnorm(t, gk, hd, eps_k, kn);
              oracle_rope_neox(kn, hd, pos, theta, kr);
              for (int d = 0; d < hd; ++d) dst[d] = oracle_double_to_bf16(kr[d]);
            } else {
              for (int d = 0; d < hd; ++d) dst[d] = oracle_double_to_bf16(t[d]);
            }
          }
        }
      }
    }
    free(x); free(h); free(g); free(hn); free(t); free(kn); free(kr); free(gk);
  }
  for (int r = 0; r < B; ++r) {
    int n = n_acc[r], c = ctx_in[r];
    int ok = row_valid(valid, r, n, c, T);
    long long s = (long long)c + n;
    ctx_out[r] = ok ? (int)(s < alloc_limit[r] ? s : alloc_limit[r]) : 0;
  }
  return 0;
}

/* MLA (single latent) context update.  w_dkv [L, lat+rope, D], g_kv [L, lat];
 * pool [L][NP][P][lat+rope] bf16.  Stored row = bf16(RMSNorm(c[0:lat]) * g) ||
 * bf16(RoPE(c[lat:lat+rope], pos)). */
int oracle_ctx_kv_update_mla(int B, int T, int L, int D_in, int D, int lat, int rope, int P, int M,
                             int num_pool_pages, double theta, double eps_h, double eps_k,
                             const void *hidden, int hidden_is_f32, const int32_t *n_acc,
                             const int32_t *ctx_in, int32_t *ctx_out, const int32_t *alloc_limit,
                             const int32_t *tbl, const uint8_t *valid, const uint16_t *w_fc,
                             const uint16_t *g_h, const uint16_t *w_dkv, const uint16_t *g_kv,
                             uint16_t *pool) {
  size_t esz = hidden_is_f32 ? 4 : 2;
  int W = lat + rope;
#pragma omp parallel
  {
    double *x = malloc(sizeof(double) * D_in);
    double *h = malloc(sizeof(double) * D);
    double *g = malloc(sizeof(double) * D);
    double *hn = malloc(sizeof(double) * D);
    double *cc = malloc(sizeof(double) * W);
    double *ln = malloc(sizeof(double) * lat);
    double *gl = malloc(sizeof(double) * lat);
    double *rr = malloc(sizeof(double) * rope);
#pragma omp for schedule(dynamic, 1)
    for (int rt = 0; rt < B * T; ++rt) {
      int r = rt / T, i = rt % T;
      int n = n_acc[r], c = ctx_in[r];
      int ok = row_valid(valid, r, n, c, T);
      int page, slot;
      if (!ctx_row_dest(ok, i, n, c, alloc_limit[r], tbl + (int64_t)r * M, M, P,
                        num_pool_pages, &page, &slot))
        continue;
      const char *row = (const char *)hidden + (size_t)rt * D_in * esz;
      fc_hidden_norm(row, hidden_is_f32, D_in, D, w_fc, g_h, eps_h, x, h, g, hn);
      double pos = (double)(c + i);
      for (int l = 0; l < L; ++l) {
        oracle_matvec_bf16(w_dkv + (size_t)l * W * D, W, D, hn, cc);
        for (int d = 0; d < lat; ++d) gl[d] = oracle_bf16_to_double(g_kv[(size_t)l * lat + d]);
        oracle_rmsnorm(cc, gl, lat, eps_k, ln);
        oracle_rope_neox(cc + lat, rope, pos, theta, rr);
        uint16_t *dst = pool + (((size_t)l * num_pool_pages + page) * P + slot) * (size_t)W;
        for (int d = 0; d < lat; ++d) dst[d] = oracle_double_to_bf16(ln[d]);
        for (int d = 0; d < rope; ++d) dst[lat + d] = oracle_double_to_bf16(rr[d]);
      }
    }
    free(x); free(h); free(g); free(hn); free(cc); free(ln); free(gl); free(rr);
  }
  for (int r = 0; r < B; ++r) {
    int n = n_acc[r], c = ctx_in[r];
    int ok = row_valid(valid, r, n, c, T);
    long long s = (long long)c + n;
    ctx_out[r] = ok ? (int)(s < alloc_limit[r] ? s : alloc_limit[r]) : 0;
  }
  return 0;
}

/* ------------------------------------------- prefill context store */
/* TensorRT-LLM PR #20550, Description (TLLM_DFLASH_FUSED_PROLOGUE): the
 * single-latent _store_context_kv_paged scatter used by prefill.  Every
 * prompt row of a request goes through the decode update's context
 * projection (fc, hidden RMSNorm, per-layer K/V or latent projection, k or
 * latent RMSNorm, RoPE at its position) and is stored into the paged pool; no
 * acceptance mask applies.  Rows of request r are hidden rows
 * cu_rows[r] .. cu_rows[r+1]-1 and sit at positions c_r + i (c_r = ctx_in[r]);
 * a row is stored when the request is live (valid, c_r >= 0), c_r + i is
 * below alloc_limit[r] and its page is mapped inside the pool.  ctx_out[r] =
 * live ? min(c_r + n_r, alloc_limit[r]) : 0.  kind 0 = GQA (w_kv [L, 2, nkv,
 * hd, D], g_k [L, hd], pool [L][NP][2][nkv][P][hd]); kind 1 = MLA (w_kv
 * [L, lat + rope, D], g_k [L, lat], pool [L][NP][P][lat + rope]). */
int oracle_ctx_kv_prefill(int kind, int B, int L, int D_in, int D, int nkv, int hd, int lat,
                          int rope, int P, int M, int num_pool_pages, double theta, double eps_h,
                          double eps_k, const void *hidden, int hidden_is_f32,
                          const int32_t *cu_rows, const int32_t *ctx_in, int32_t *ctx_out,
                          const int32_t *alloc_limit, const int32_t *tbl, const uint8_t *valid,
                          const uint16_t *w_fc, const uint16_t *g_h, const uint16_t *w_kv,
                          const uint16_t *g_k, uint16_t *pool) {
  size_t esz = hidden_is_f32 ? 4 : 2;
  int N = cu_rows[B];
  int W = kind == 0 ? hd : lat + rope;
  int GW = kind == 0 ? hd : lat;
  for (int r = 0; r < B; ++r)
    if (cu_rows[r + 1] < cu_rows[r]) return -1;
#pragma omp parallel
  {
    double *x = malloc(sizeof(double) * D_in);
    double *h = malloc(sizeof(double) * D);
    double *g = malloc(sizeof(double) * D);
    double *hn = malloc(sizeof(double) * D);
    double *t = malloc(sizeof(double) * W);
    double *nrm = malloc(sizeof(double) * GW);
    double *rot = malloc(sizeof(double) * W);
    double *gk = malloc(sizeof(double) * GW);
#pragma omp for schedule(dynamic, 1)
    for (int n = 0; n < N; ++n) {
      int r = 0;
      while (cu_rows[r + 1] <= n) ++r; /* the request holding hidden row n */
      int i = n - cu_rows[r];
      int c = ctx_in[r];
      int live = (valid ? valid[r] != 0 : 1) && c >= 0;
      int page, slot;
      if (!ctx_row_dest(live, i, i + 1, c, alloc_limit[r], tbl + (int64_t)r * M, M, P,
                        num_pool_pages, &page, &slot))
        continue;
      const char *row = (const char *)hidden + (size_t)n * D_in * esz;
      fc_hidden_norm(row, hidden_is_f32, D_in, D, w_fc, g_h, eps_h, x, h, g, hn);
      double pos = (double)(c + i);
      for (int l = 0; l < L; ++l) {
        for (int d = 0; d < GW; ++d) gk[d] = oracle_bf16_to_double(g_k[(size_t)l * GW + d]);
        if (kind == 0) {
          for (int kv = 0; kv < 2; ++kv)
            for (int hh = 0; hh < nkv; ++hh) {
              const uint16_t *Wm = w_kv + ((((size_t)l * 2 + kv) * nkv + hh) * hd) * (size_t)D;
              oracle_matvec_bf16(Wm, hd, D, hn, t);
              uint16_t *dst =
                  pool + (((((size_t)l * num_pool_pages + page) * 2 + kv) * nkv + hh) * P + slot) *
                             (size_t)hd;
              if (kv == 0) {
                oracle_rmsnorm(t, gk, hd, eps_k, nrm);
                oracle_rope_neox(nrm, hd, pos, theta, rot);
                for (int d = 0; d < hd; ++d) dst[d] = oracle_double_to_bf16(rot[d]);
              } else {
                for (int d = 0; d < hd; ++d) dst[d] = oracle_double_to_bf16(t[d]);
              }
            }
        } else {
          oracle_matvec_bf16(w_kv + (size_t)l * W * D, W, D, hn, t);
          oracle_rmsnorm(t, gk, lat, eps_k, nrm);
          oracle_rope_neox(t + lat, rope, pos, theta, rot);
          uint16_t *dst = pool + (((size_t)l * num_pool_pages + page) * P + slot) * (size_t)W;
          for (int d = 0; d < lat; ++d) dst[d] = oracle_double_to_bf16(nrm[d]);
          for (int d = 0; d < rope; ++d) dst[lat + d] = oracle_double_to_bf16(rot[d]);
        }
      }
    }
    free(x); free(h); free(g); free(hn); free(t); free(nrm); free(rot); free(gk);
  }
  for (int r = 0; r < B; ++r) {
    int c = ctx_in[r];
    int live = (valid ? valid[r] != 0 : 1) && c >= 0;
    long long s = (long long)c + (cu_rows[r + 1] - cu_rows[r]);
    ctx_out[r] = live ? (int)(s < alloc_limit[r] ? s : alloc_limit[r]) : 0;
  }
  return 0;
}

/* ------------------------------------------- split context-KV update */
/* TensorRT-LLM PR #20550, Description (TLLM_DFLASH_OVERLAP_CONTEXT_PROJECTION):
 * the context projection (fc, hidden norm, latent / K-V projection, norm and
 * RoPE) runs before acceptance, from the target hidden states and the
 * pre-step ctx_len alone; the accepted-mask write follows after the join.
 * Projection half: for EVERY row (no write mask) the values the update would
 * store, RoPE at c + i; staged_c[r] = the c used.  Staged row layout:
 * GQA [L][2][nkv][hd], MLA [L][lat + rope], bf16 bits. */
int oracle_ctx_kv_project_gqa(int B, int T, int L, int D_in, int D, int nkv, int hd,
                              double theta, double eps_h, double eps_k, const void *hidden,
                              int hidden_is_f32, const int32_t *ctx_in, const uint16_t *w_fc,
                              const uint16_t *g_h, const uint16_t *w_kv, const uint16_t *g_k,
                              int32_t *staged_c, uint16_t *staged) {
  size_t esz = hidden_is_f32 ? 4 : 2;
  size_t row_w = (size_t)L * 2 * nkv * hd;
  for (int r = 0; r < B; ++r) staged_c[r] = ctx_in[r];
#pragma omp parallel
  {
    double *x = malloc(sizeof(double) * D_in);
    double *h = malloc(sizeof(double) * D);
    double *g = malloc(sizeof(double) * D);
    double *hn = malloc(sizeof(double) * D);
    double *t = malloc(sizeof(double) * hd);
    double *kn = malloc(sizeof(double) * hd);
    double *kr = malloc(sizeof(double) * hd);
    double *gk = malloc(sizeof(double) * hd);
#pragma omp for schedule(dynamic, 1)
    for (int rt = 0; rt < B * T; ++rt) {
      int r = rt / T, i = rt % T;
      const char *row = (const char *)hidden + (size_t)rt * D_in * esz;
      fc_hidden_norm(row, hidden_is_f32, D_in, D, w_fc, g_h, eps_h, x, h, g, hn);
      double pos = (double)ctx_in[r] + i;
      for (int l = 0; l < L; ++l) {
        for (int d = 0; d < hd; ++d) gk[d] = oracle_bf16_to_double(g_k[(size_t)l * hd + d]);
        for (int kv = 0; kv < 2; ++kv) {
          for (int hh = 0; hh < nkv; ++hh) {
            const uint16_t *Wh = w_kv + ((((size_t)l * 2 + kv) * nkv + hh) * hd) * (size_t)D;
            oracle_matvec_bf16(Wh, hd, D, hn, t);
            uint16_t *dst = staged + (size_t)rt * row_w + (((size_t)l * 2 + kv) * nkv + hh) * hd;
            if (kv == 0) {
              oracle_rmsnorm(t, gk, hd, eps_k, kn);
              oracle_rope_neox(kn, hd, pos, theta, kr);
              for (int d = 0; d < hd; ++d) dst[d] = oracle_double_to_bf16(kr[d]);
            } else {
              for (int d = 0; d < hd; ++d) dst[d] = oracle_double_to_bf16(t[d]);
            }
          }
        }
      }
    }
    free(x); free(h); free(g); free(hn); free(t); free(kn); free(kr); free(gk);
  }
  return 0;
}

int oracle_ctx_kv_project_mla(int B, int T, int L, int D_in, int D, int lat, int rope,
                              double theta, double eps_h, double eps_k, const void *hidden,
                              int hidden_is_f32, const int32_t *ctx_in, const uint16_t *w_fc,
                              const uint16_t *g_h, const uint16_t *w_dkv, const uint16_t *g_kv,
                              int32_t *staged_c, uint16_t *staged) {
  size_t esz = hidden_is_f32 ? 4 : 2;
  int W = lat + rope;
  for (int r = 0; r < B; ++r) staged_c[r] = ctx_in[r];
#pragma omp parallel
  {
    double *x = malloc(sizeof(double) * D_in);
    double *h = malloc(sizeof(double) * D);
    double *g = malloc(sizeof(double) * D);
    double *hn = malloc(sizeof(double) * D);
    double *cc = malloc(sizeof(double) * W);
    double *ln = malloc(sizeof(double) * lat);
    double *gl = malloc(sizeof(double) * lat);
    double *rr = malloc(sizeof(double) * rope);
#pragma omp for schedule(dynamic, 1)
    for (int rt = 0; rt < B * T; ++rt) {
      int r = rt / T, i = rt % T;
      const char *row = (const char *)hidden + (size_t)rt * D_in * esz;
      fc_hidden_norm(row, hidden_is_f32, D_in, D, w_fc, g_h, eps_h, x, h, g, hn);
      double pos = (double)ctx_in[r] + i;
      for (int l = 0; l < L; ++l) {
        oracle_matvec_bf16(w_dkv + (size_t)l * W * D, W, D, hn, cc);
        for (int d = 0; d < lat; ++d) gl[d] = oracle_bf16_to_double(g_kv[(size_t)l * lat + d]);
        oracle_rmsnorm(cc, gl, lat, eps_k, ln);
        oracle_rope_neox(cc + lat, rope, pos, theta, rr);
        uint16_t *dst = staged + ((size_t)rt * L + l) * W;
        for (int d = 0; d < lat; ++d) dst[d] = oracle_double_to_bf16(ln[d]);
        for (int d = 0; d < rope; ++d) dst[lat + d] = oracle_double_to_bf16(rr[d]);
      }
    }
    free(x); free(h); free(g); free(hn); free(cc); free(ln); free(gl); free(rr);
  }
  return 0;
}

/* Store half (after the join): the write-masked paged store of the staged
 * rows and the ctx_len advance, both from the c the projection recorded.
 * kind 0 = GQA (pool [L][NP][2][nkv][P][hd]), 1 = MLA (pool [L][NP][P][W]). */
int oracle_ctx_kv_commit(int kind, int B, int T, int L, int nkv, int hd, int W, int P, int M,
                         int num_pool_pages, const int32_t *staged_c, const uint16_t *staged,
                         const int32_t *n_acc, int32_t *ctx_out, const int32_t *alloc_limit,
                         const int32_t *tbl, const uint8_t *valid, uint16_t *pool) {
  size_t row_w = kind == 0 ? (size_t)L * 2 * nkv * hd : (size_t)L * W;
  for (int rt = 0; rt < B * T; ++rt) {
    int r = rt / T, i = rt % T;
    int n = n_acc[r], c = staged_c[r];
    int ok = row_valid(valid, r, n, c, T);
    int page, slot;
    if (!ctx_row_dest(ok, i, n, c, alloc_limit[r], tbl + (int64_t)r * M, M, P, num_pool_pages,
                      &page, &slot))
      continue;
    const uint16_t *src = staged + (size_t)rt * row_w;
    for (int l = 0; l < L; ++l) {
      if (kind == 0) {
        for (int kv = 0; kv < 2; ++kv)
          for (int hh = 0; hh < nkv; ++hh) {
            uint16_t *dst =
                pool + (((((size_t)l * num_pool_pages + page) * 2 + kv) * nkv + hh) * P + slot) *
                           (size_t)hd;
            memcpy(dst, src + (((size_t)l * 2 + kv) * nkv + hh) * hd, sizeof(uint16_t) * hd);
          }
      } else {
        uint16_t *dst = pool + (((size_t)l * num_pool_pages + page) * P + slot) * (size_t)W;
        memcpy(dst, src + (size_t)l * W, sizeof(uint16_t) * W);
      }
    }
  }
  for (int r = 0; r < B; ++r) {
    int n = n_acc[r], c = staged_c[r];
    int ok = row_valid(valid, r, n, c, T);
    long long s = (long long)c + n;
    ctx_out[r] = ok ? (int)(s < alloc_limit[r] ? s : alloc_limit[r]) : 0;
  }
  return 0;
}

/* ------------------------------------------ either side of the path */
/* TensorRT-LLM PR #20550, follow-up commit "spec_tail_kernels.py": strict
 * acceptance of a uniform-width draft.  Request r drafted K tokens
 * draft[r, 0..K-1]; the target produced K + 1 tokens target[r, 0..K] at the
 * same positions.  Drafts are accepted while they equal the target's token;
 * the target's token at the first disagreement (or after the last draft) is
 * the bonus.  n_acc[r] = 1 + (leading matches) in [1, K + 1];
 * accepted[r, i] = target[r, i] for i < n_acc[r], -1 after. */
int oracle_strict_accept(int B, int K, const int32_t *draft, const int32_t *target,
                         int32_t *n_acc, int32_t *accepted) {
  for (int r = 0; r < B; ++r) {
    int m = 0;
    while (m < K && draft[(size_t)r * K + m] == target[(size_t)r * (K + 1) + m]) ++m;
    n_acc[r] = m + 1;
    for (int i = 0; i <= K; ++i)
      accepted[(size_t)r * (K + 1) + i] = i <= m ? target[(size_t)r * (K + 1) + i] : -1;
  }
  return 0;
}

/* TensorRT-LLM PR #13995, commit "fuse query-input build in pure Torch +
 * fused embedding lookup": the noise block's input rows are one embedding
 * lookup over its ids ([bonus, mask_id, ...]).  out[k, :] = table[ids[k], :]
 * for k < n (bf16 bits); an id outside [0, V) gives a zero row and returns 1. */
int oracle_embedding_gather(int n, int V, int D, const int32_t *ids, const uint16_t *table,
                            uint16_t *out) {
  int bad = 0;
  for (int k = 0; k < n; ++k) {
    int id = ids[k];
    if (id < 0 || id >= V) {
      memset(out + (size_t)k * D, 0, sizeof(uint16_t) * D);
      bad = 1;
      continue;
    }
    memcpy(out + (size_t)k * D, table + (size_t)id * D, sizeof(uint16_t) * D);
  }
  return bad;
}

/* ------------------------------------------------------- query side */
/* TensorRT-LLM PR #13995, commits "use fused qk-norm+rope on non-YaRN draft"
 * and "match RoPE between context and query": the drafter's query rows get
 * RMSNorm (gain gamma, eps) and the same rotate-half RoPE as the context keys,
 * at the query positions.  q_in / q_out [rows][heads][dim] bf16 bits,
 * pos [rows]; do_norm = 0 applies the rotation only (the MLA rope part). */
int oracle_q_norm_rope(int rows, int heads, int dim, int do_norm, double theta, double eps,
                       const uint16_t *q_in, const uint16_t *gamma, const int32_t *pos,
                       uint16_t *q_out) {
  double *x = malloc(sizeof(double) * dim);
  double *g = malloc(sizeof(double) * dim);
  double *n = malloc(sizeof(double) * dim);
  double *o = malloc(sizeof(double) * dim);
  for (int d = 0; d < dim; ++d) g[d] = do_norm ? oracle_bf16_to_double(gamma[d]) : 1.0;
  for (int r = 0; r < rows; ++r) {
    for (int h = 0; h < heads; ++h) {
      size_t base = ((size_t)r * heads + h) * dim;
      for (int d = 0; d < dim; ++d) x[d] = oracle_bf16_to_double(q_in[base + d]);
      if (do_norm)
        oracle_rmsnorm(x, g, dim, eps, n);
      else
        memcpy(n, x, sizeof(double) * dim);
      oracle_rope_neox(n, dim, (double)pos[r], theta, o);
      for (int d = 0; d < dim; ++d) q_out[base + d] = oracle_double_to_bf16(o[d]);
    }
  }
  free(x); free(g); free(n); free(o);
  return 0;
}

/* --------------------------------------------------- block KV scatter */

/* GQA: blk_k / blk_v [B, T, nkv, hd] -> pool layer `layer` at the placement. */
int oracle_block_kv_scatter_gqa(int B, int T, int nkv, int hd, int P, int num_pool_pages,
                                int layer, const uint16_t *blk_k, const uint16_t *blk_v,
                                const int32_t *blk_page, const int32_t *blk_slot,
                                const uint8_t *blk_mask, uint16_t *pool) {
  for (int r = 0; r < B; ++r)
    for (int i = 0; i < T; ++i) {
      int64_t k = (int64_t)r * T + i;
      if (!blk_mask[k]) continue;
      int pg = blk_page[k], sl = blk_slot[k];
      if (pg < 0 || pg >= num_pool_pages || sl < 0 || sl >= P) return -1;
      for (int kv = 0; kv < 2; ++kv)
        for (int h = 0; h < nkv; ++h) {
          const uint16_t *src = (kv == 0 ? blk_k : blk_v) + ((size_t)k * nkv + h) * hd;
          uint16_t *dst =
              pool + (((((size_t)layer * num_pool_pages + pg) * 2 + kv) * nkv + h) * P + sl) *
                         (size_t)hd;
          memcpy(dst, src, sizeof(uint16_t) * hd);
        }
    }
  return 0;
}

/* MLA: blk_latent [B, T, W] -> pool layer `layer` at the placement. */
int oracle_block_latent_scatter_mla(int B, int T, int W, int P, int num_pool_pages, int layer,
                                    const uint16_t *blk_lat, const int32_t *blk_page,
                                    const int32_t *blk_slot, const uint8_t *blk_mask,
                                    uint16_t *pool) {
  for (int r = 0; r < B; ++r)
    for (int i = 0; i < T; ++i) {
      int64_t k = (int64_t)r * T + i;
      if (!blk_mask[k]) continue;
      int pg = blk_page[k], sl = blk_slot[k];
      if (pg < 0 || pg >= num_pool_pages || sl < 0 || sl >= P) return -1;
      memcpy(pool + (((size_t)layer * num_pool_pages + pg) * P + sl) * (size_t)W,
             blk_lat + (size_t)k * W, sizeof(uint16_t) * W);
    }
  return 0;
}

/* ------------------------------------------------------------ attention */

/* Visible key range [lo, hi] of query i (hi < lo: empty). */
static void key_range(int kv_len, int Tq, int i, int window, int mask_mode, int *lo, int *hi) {
  int p = kv_len - Tq + i;
  int h = (mask_mode == OR_MASK_CAUSAL_TAIL) ? p : kv_len - 1;
  int l = 0;
  if (window > 0) {
    int w0 = p - window + 1;
    l = w0 > 0 ? w0 : 0;
  }
  *lo = l;
  *hi = h;
}

/* Key j of request r: pointer to its cache row (GQA K or V of head kvh, or
 * the MLA latent row), or NULL when the table maps it outside the pool. */
static const uint16_t *gqa_row(const uint16_t *pool, const int32_t *tbl_row, int j, int P,
                               int num_pool_pages, int layer, int kv, int nkv, int kvh, int hd) {
  int pg = tbl_row[j / P];
  if (pg < 0 || pg >= num_pool_pages) return NULL;
  return pool + (((((size_t)layer * num_pool_pages + pg) * 2 + kv) * nkv + kvh) * P + j % P) *
                    (size_t)hd;
}

static const uint16_t *mla_row(const uint16_t *pool, const int32_t *tbl_row, int j, int P,
                               int num_pool_pages, int layer, int W) {
  int pg = tbl_row[j / P];
  if (pg < 0 || pg >= num_pool_pages) return NULL;
  return pool + (((size_t)layer * num_pool_pages + pg) * P + j % P) * (size_t)W;
}

/* Softmax-weighted sum over one (r, i, h) with an optional sink logit.
 * scores[n], values fetched by callback-free index arrays: the caller passes
 * value rows. */
static void softmax_combine(int nk, const double *s, const uint16_t *const *vrows, int dv,
                            int has_sink, double sink, double *out) {
  for (int d = 0; d < dv; ++d) out[d] = 0.0;
  if (nk == 0) return;
  double m = has_sink ? sink : -INFINITY;
  for (int k = 0; k < nk; ++k)
    if (s[k] > m) m = s[k];
  double den = has_sink ? exp(sink - m) : 0.0;
  for (int k = 0; k < nk; ++k) {
    double e = exp(s[k] - m);
    den += e;
    for (int d = 0; d < dv; ++d) out[d] += e * oracle_bf16_to_double(vrows[k][d]);
  }
  for (int d = 0; d < dv; ++d) out[d] /= den;
}

/* GQA block attention, direct definition.
 * q [B, Tq, hq, hd] bf16; pool as in the update; tbl [B, M]; kv_len [B];
 * sinks [hq] fp32 or NULL; out [B, Tq, hq, hd] double.  Returns -1 when a
 * visible key maps outside the pool or kv_len exceeds M*P. */
int oracle_attention_gqa(int B, int Tq, int hq, int nkv, int hd, int P, int M,
                         int num_pool_pages, int layer, const uint16_t *q, const uint16_t *pool,
                         const int32_t *tbl, const int32_t *kv_len, int window,
                         const float *sinks, double scale, int mask_mode, double *out) {
  int G = hq / nkv;
  int bad = 0;
  for (int r = 0; r < B; ++r)
    if (kv_len[r] < 0 || (long long)kv_len[r] > (long long)M * P) return -1;
#pragma omp parallel for collapse(3) schedule(dynamic, 1) reduction(| : bad)
  for (int r = 0; r < B; ++r)
    for (int i = 0; i < Tq; ++i)
      for (int h = 0; h < hq; ++h) {
        int kvh = h / G;
        int lo, hi;
        key_range(kv_len[r], Tq, i, window, mask_mode, &lo, &hi);
        int nk = hi >= lo ? hi - lo + 1 : 0;
        double *s = malloc(sizeof(double) * (nk > 0 ? nk : 1));
        const uint16_t **vr = malloc(sizeof(void *) * (nk > 0 ? nk : 1));
        const uint16_t *qv = q + (((size_t)r * Tq + i) * hq + h) * hd;
        for (int k = 0; k < nk; ++k) {
          int j = lo + k;
          const uint16_t *kr =
              gqa_row(pool, tbl + (int64_t)r * M, j, P, num_pool_pages, layer, 0, nkv, kvh, hd);
          const uint16_t *vv =
              gqa_row(pool, tbl + (int64_t)r * M, j, P, num_pool_pages, layer, 1, nkv, kvh, hd);
          if (!kr || !vv) { bad = 1; s[k] = 0; vr[k] = qv; continue; }
          double dot = 0.0;
          for (int d = 0; d < hd; ++d)
            dot += oracle_bf16_to_double(qv[d]) * oracle_bf16_to_double(kr[d]);
          s[k] = scale * dot;
          vr[k] = vv;
        }
        softmax_combine(nk, s, vr, hd, sinks != NULL, sinks ? (double)sinks[h] : 0.0,
                        out + (((size_t)r * Tq + i) * hq + h) * hd);
        free(s);
        free(vr);
      }
  return bad ? -1 : 0;
}

/* MLA absorbed-latent block attention, direct definition.
 * q_lat [B, Tq, hq, lat], q_rope [B, Tq, hq, rope]; pool [L][NP][P][lat+rope];
 * score = scale * (<q_lat, c> + <q_rope, r>); value = c (lat dims);
 * out [B, Tq, hq, lat] double. */
int oracle_attention_mla(int B, int Tq, int hq, int lat, int rope, int P, int M,
                         int num_pool_pages, int layer, const uint16_t *q_lat,
                         const uint16_t *q_rope, const uint16_t *pool, const int32_t *tbl,
                         const int32_t *kv_len, int window, const float *sinks, double scale,
                         int mask_mode, double *out) {
  int W = lat + rope;
  int bad = 0;
  for (int r = 0; r < B; ++r)
    if (kv_len[r] < 0 || (long long)kv_len[r] > (long long)M * P) return -1;
#pragma omp parallel for collapse(3) schedule(dynamic, 1) reduction(| : bad)
  for (int r = 0; r < B; ++r)
    for (int i = 0; i < Tq; ++i)
      for (int h = 0; h < hq; ++h) {
        int lo, hi;
        key_range(kv_len[r], Tq, i, window, mask_mode, &lo, &hi);
        int nk = hi >= lo ? hi - lo + 1 : 0;
        double *s = malloc(sizeof(double) * (nk > 0 ? nk : 1));
        const uint16_t **vr = malloc(sizeof(void *) * (nk > 0 ? nk : 1));
        const uint16_t *ql = q_lat + (((size_t)r * Tq + i) * hq + h) * lat;
        const uint16_t *qr = q_rope + (((size_t)r * Tq + i) * hq + h) * rope;
        for (int k = 0; k < nk; ++k) {
          int j = lo + k;
          const uint16_t *row =
              mla_row(pool, tbl + (int64_t)r * M, j, P, num_pool_pages, layer, W);
          if (!row) { bad = 1; s[k] = 0; vr[k] = ql; continue; }
          double dot = 0.0;
          for (int d = 0; d < lat; ++d)
            dot += oracle_bf16_to_double(ql[d]) * oracle_bf16_to_double(row[d]);
          for (int d = 0; d < rope; ++d)
            dot += oracle_bf16_to_double(qr[d]) * oracle_bf16_to_double(row[lat + d]);
          s[k] = scale * dot;
          vr[k] = row;
        }
        softmax_combine(nk, s, vr, lat, sinks != NULL, sinks ? (double)sinks[h] : 0.0,
                        out + (((size_t)r * Tq + i) * hq + h) * lat);
        free(s);
        free(vr);
      }
  return bad ? -1 : 0;
}

/* GQA block attention, split-KV form: the visible span of request r,
 * [min_i lo_i, max_i hi_i], is cut into S equal slices of ceil(span / S)
 * keys (the last may be short or empty).  Each slice yields, per (i, h),
 * m_s = max score, l_s = sum e^(s - m_s), o_s = sum e^(s - m_s) v over the
 * visible keys it holds; empty slices (m_s = -inf) are skipped.  The merge is
 * out = sum_s e^(m_s - M) o_s / (sum_s e^(m_s - M) l_s + e^(sink - M)),
 * M = max(max_s m_s, sink). */
int oracle_attention_gqa_split(int B, int Tq, int hq, int nkv, int hd, int P, int M,
                               int num_pool_pages, int layer, const uint16_t *q,
                               const uint16_t *pool, const int32_t *tbl, const int32_t *kv_len,
                               int window, const float *sinks, double scale, int mask_mode,
                               int S, double *out) {
  int G = hq / nkv;
  if (S < 1) return -1;
  for (int r = 0; r < B; ++r) {
    if (kv_len[r] < 0 || (long long)kv_len[r] > (long long)M * P) return -1;
    int span_lo = 0, span_hi = -1;
    for (int i = 0; i < Tq; ++i) {
      int lo, hi;
      key_range(kv_len[r], Tq, i, window, mask_mode, &lo, &hi);
      if (i == 0 || lo < span_lo) span_lo = lo;
      if (i == 0 || hi > span_hi) span_hi = hi;
    }
    int span = span_hi >= span_lo ? span_hi - span_lo + 1 : 0;
    int seg = span > 0 ? (span + S - 1) / S : 0;
    double *ms = malloc(sizeof(double) * S);
    double *ls = malloc(sizeof(double) * S);
    double *os = malloc(sizeof(double) * (size_t)S * hd);
    for (int i = 0; i < Tq; ++i)
      for (int h = 0; h < hq; ++h) {
        int kvh = h / G;
        int lo, hi;
        key_range(kv_len[r], Tq, i, window, mask_mode, &lo, &hi);
        const uint16_t *qv = q + (((size_t)r * Tq + i) * hq + h) * hd;
        for (int sI = 0; sI < S; ++sI) {
          int a = span_lo + sI * seg, b = a + seg - 1;
          if (b > span_hi) b = span_hi;
          if (a < lo) a = lo;
          if (b > hi) b = hi;
          ms[sI] = -INFINITY;
          ls[sI] = 0.0;
          for (int d = 0; d < hd; ++d) os[(size_t)sI * hd + d] = 0.0;
          if (seg == 0 || b < a) continue;
          for (int j = a; j <= b; ++j) {
            const uint16_t *kr = gqa_row(pool, tbl + (int64_t)r * M, j, P, num_pool_pages,
                                         layer, 0, nkv, kvh, hd);
            if (!kr) { free(ms); free(ls); free(os); return -1; }
            double dot = 0.0;
            for (int d = 0; d < hd; ++d)
              dot += oracle_bf16_to_double(qv[d]) * oracle_bf16_to_double(kr[d]);
            if (scale * dot > ms[sI]) ms[sI] = scale * dot;
          }
          for (int j = a; j <= b; ++j) {
            const uint16_t *kr = gqa_row(pool, tbl + (int64_t)r * M, j, P, num_pool_pages,
                                         layer, 0, nkv, kvh, hd);
            const uint16_t *vv = gqa_row(pool, tbl + (int64_t)r * M, j, P, num_pool_pages,
                                         layer, 1, nkv, kvh, hd);
            double dot = 0.0;
            for (int d = 0; d < hd; ++d)
              dot += oracle_bf16_to_double(qv[d]) * oracle_bf16_to_double(kr[d]);
            double e = exp(scale * dot - ms[sI]);
            ls[sI] += e;
            for (int d = 0; d < hd; ++d) os[(size_t)sI * hd + d] += e * oracle_bf16_to_double(vv[d]);
          }
        }
        double Mx = sinks ? (double)sinks[h] : -INFINITY;
        for (int sI = 0; sI < S; ++sI)
          if (ms[sI] > Mx) Mx = ms[sI];
        double *o = out + (((size_t)r * Tq + i) * hq + h) * hd;
        for (int d = 0; d < hd; ++d) o[d] = 0.0;
        if (Mx == -INFINITY) continue;
        double den = sinks ? exp((double)sinks[h] - Mx) : 0.0;
        for (int sI = 0; sI < S; ++sI) {
          if (ms[sI] == -INFINITY) continue;
          double w = exp(ms[sI] - Mx);
          den += w * ls[sI];
          for (int d = 0; d < hd; ++d) o[d] += w * os[(size_t)sI * hd + d];
        }
        for (int d = 0; d < hd; ++d) o[d] = den > 0 ? o[d] / den : 0.0;
      }
    free(ms);
    free(ls);
    free(os);
  }
  return 0;
}

/* Thread count the OpenMP runtime would use (1 when built without it). */
int oracle_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  extern void omp_set_num_threads(int);
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
