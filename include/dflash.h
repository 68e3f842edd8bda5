/*
 * dflash.h -- C ABI of the GB300 (sm_103a) drafter decode-step library.
 *
 * The library implements the data-parallel hot path of one decode step of a
 * DFlash / DSpark block drafter:
 *   1. the bookkeeping around the context-KV update (block-table decode,
 *      bonus / mask embedding ids, query and context positions, write masks,
 *      ctx_len advance, block placement);
 *   2. the context-KV update itself (fc -> hidden RMSNorm -> stacked per-layer
 *      K/V or latent projection -> k RMSNorm + RoPE -> masked paged store);
 *   3. the block-KV scatter and the decode-shaped split-KV block attention.
 *
 * Conventions shared by every call
 *  - All pointers named as device buffers are device pointers the caller owns
 *    and keeps alive until the work on `stream` has finished.  No call
 *    allocates memory, synchronises the host, or reads a device value on the
 *    host.  The calls of the decode step (bookkeeping, context update,
 *    scatter, attention) may be captured in a CUDA graph; each makes its
 *    one-time per-device set-up on its first eager call.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *    enqueued asynchronously; a return of DFLASH_OK means "validated and
 *    enqueued", not "finished".  The device current on the calling thread
 *    must be the device of `stream` (launch limits, SM counts and the
 *    allocation-free scratch are looked up for the current device).
 *  - bf16 means IEEE bfloat16 (1-8-7).  Every tensor is dense row-major in the
 *    stated shape unless a row stride is given.  Device buffers read with
 *    vector loads or TMA (KV pool, weights, hidden, q, block K/V, workspace)
 *    must be 16-byte aligned.
 *  - Per-request scalars (n_accepted, ctx_len, kv_len, ...) live in device
 *    arrays and are read on the device only.
 *  - Errors: a call returns a dflash_status_code.  Host-detectable problems
 *    (null pointers, bad geometry, misalignment, small workspace) return an
 *    error and enqueue nothing; there is no fallback path.  Problems in device
 *    data (a page id outside the pool, n_accepted outside [1, T], kv_len
 *    beyond the table) never fault: the affected row is masked or clamped and
 *    a DFLASH_DEV_* bit is OR-ed into *dev_status when dev_status is non-NULL.
 *
 * KV pool layouts (one plane per drafter layer, pages shared by all layers)
 *  - GQA: bf16 [L][num_pool_pages][2][nkv][page_size][head_dim]; index 0 of
 *    the third axis is K, 1 is V.  One (layer, page, K|V, head) block is
 *    page_size * head_dim contiguous values.
 *  - MLA: bf16 [L][num_pool_pages][page_size][latent_dim + rope_dim]; one
 *    latent row per token: RMS-normed latent then the rotated rope part.
 *
 * Sources (page title and part):
 *  [TRT-20548] TensorRT-LLM issue #20548, Proposal.
 *  [TRT-20550] TensorRT-LLM PR #20550, Description and the follow-up commit
 *              "spec_tail_kernels.py".
 *  [TRT-13995] TensorRT-LLM PR #13995 "DFlash performance optimizations",
 *              commits "migrate draft path to per-layer cached K/V pool",
 *              "fuse cross-layer k_norm", "match RoPE between context and
 *              query", "fuse query-input build", "drop K-1 filler tokens".
 *  [VLLM-54092] vLLM PR #54092, Purpose item 2 and Changes item 2.
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DFLASH_API __attribute__((visibility("default")))
#else
#define DFLASH_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without including the CUDA headers. */
typedef struct CUstream_st *dflash_stream_t;

/* Return codes. */
enum dflash_status_code {
  DFLASH_OK = 0,
  DFLASH_ERR_INVALID_ARG = 1,        /* null / misaligned pointer, bad count or index */
  DFLASH_ERR_UNSUPPORTED_GEOM = 2,   /* geometry outside what the kernels implement */
  DFLASH_ERR_WORKSPACE_TOO_SMALL = 3,
  DFLASH_ERR_CUDA = 4                /* a CUDA runtime / driver call failed */
};

/* Bits OR-ed into *dev_status by device code. */
#define DFLASH_DEV_BAD_NACCEPTED 1u   /* live row with n_accepted outside [1, T]: treated as dummy */
#define DFLASH_DEV_BAD_CTX_LEN 2u     /* live row with ctx_len < 0: treated as dummy */
#define DFLASH_DEV_CTX_OUTRUN 4u      /* ctx_len already beyond the allocation limit */
#define DFLASH_DEV_BAD_PAGE 8u        /* table entry outside [0, num_pool_pages): row/key masked */
#define DFLASH_DEV_KV_LEN_RANGE 16u   /* kv_len < 0 or > max_pages * page_size: clamped */
#define DFLASH_DEV_WAIT_TIMEOUT 32u   /* an on-chip pipeline wait hit its iteration limit */
#define DFLASH_DEV_BAD_TOKEN 64u      /* embedding id outside [0, vocab): zero row written */

enum dflash_kind { DFLASH_KIND_GQA = 0, DFLASH_KIND_MLA = 1 };
enum dflash_mask_mode { DFLASH_MASK_CAUSAL_TAIL = 0, DFLASH_MASK_BLOCK_BIDIR = 1 };
enum dflash_dtype { DFLASH_DTYPE_BF16 = 0, DFLASH_DTYPE_F32 = 1 };

/* Drafter geometry.  Filled once by the caller. */
typedef struct dflash_geom {
  int32_t kind;            /* DFLASH_KIND_GQA or DFLASH_KIND_MLA */
  int32_t num_layers;      /* L: drafter layers sharing one page table */
  int32_t d_in;            /* fc input width (target hidden size) */
  int32_t d_model;         /* fc output width = drafter hidden size */
  int32_t hq;              /* query heads */
  int32_t nkv;             /* KV heads (GQA); 1 for MLA */
  int32_t head_dim;        /* GQA head dim: even multiple of 8 up to 256 for the
                              update, 64 or 128 for the attention */
  int32_t latent_dim;      /* MLA latent width (512) */
  int32_t rope_dim;        /* MLA rotated width (64) */
  int32_t page_size;       /* P: tokens per page */
  int32_t max_pages;       /* M: entries per block-table row */
  int32_t num_pool_pages;  /* pages in each layer plane of the pool */
  int32_t block_size;      /* T = K + 1 rows per request (bonus + K drafts) */
  int32_t reserved0;
  double rope_theta;       /* RoPE base */
  double eps_hidden;       /* eps of the hidden RMSNorm */
  double eps_k;            /* eps of the k (or latent) RMSNorm, shared by all layers */
} dflash_geom;

/* Weights of the context projection, packed once by the caller.  All bf16.
 *  w_fc    [d_model, d_in]
 *  gamma_h [d_model]
 *  w_kv    GQA: [L][2][nkv][head_dim][d_model]  (K rows, then V rows, per layer)
 *          MLA: [L][latent_dim + rope_dim][d_model]
 *  gamma_k GQA: [L][head_dim] (shared by the heads of a layer)
 *          MLA: [L][latent_dim]
 * The stacking of every layer's K/V projection into one matrix is what lets
 * one GEMM serve all drafter layers [TRT-13995, "per-layer cached K/V pool";
 * "fuse cross-layer k_norm": stacked k_norm weights, one eps]. */
typedef struct dflash_weights {
  const void *w_fc;
  const void *gamma_h;
  const void *w_kv;
  const void *gamma_k;
} dflash_weights;

/* One drafter layer's projection weights as a model holds them (device,
 * bf16, row-major), the input of dflash_pack_weights.
 *  w_k     GQA: k_proj [nkv * head_dim, d_model]
 *          MLA: the latent (down) projection [latent_dim + rope_dim, d_model]
 *  w_v     GQA: v_proj [nkv * head_dim, d_model]; MLA: NULL
 *  k_norm  GQA: the k RMSNorm gain [head_dim]; MLA: the latent RMSNorm gain
 *          [latent_dim] */
typedef struct dflash_layer_weights {
  const void *w_k;
  const void *w_v;
  const void *k_norm;
} dflash_layer_weights;

/* Outputs of dflash_step_bookkeeping (all device, int32 unless noted;
 * [B] or [B, T] or [B, M] dense). */
typedef struct dflash_step_outputs {
  int32_t *n_pages;      /* [B]    pages the request owns (count of offsets >= 0) */
  int32_t *block_table;  /* [B, M] max(offset, 0) / off_div */
  int32_t *alloc_limit;  /* [B]    A = min(max_ctx, n_pages * P) */
  int32_t *bonus;        /* [B]    accepted[n-1] */
  int32_t *emb_ids;      /* [B, T] bonus, then mask_token_id */
  int32_t *ctx_pos;      /* [B, T] c + i (RoPE positions of the context rows) */
  int32_t *q_pos;        /* [B, T] c' + i (positions of the block's queries) */
  int32_t *ctx_dst_page; /* [B, T] physical page of context row i, -1 if masked */
  int32_t *ctx_dst_slot; /* [B, T] slot in that page, -1 if masked */
  uint8_t *ctx_wmask;    /* [B, T] 1 = row i is written */
  int32_t *blk_page;     /* [B, T] DraftBlockPlacement: page of q_pos, -1 if unplaced */
  int32_t *blk_slot;     /* [B, T] slot of q_pos, -1 if unplaced */
  uint8_t *blk_mask;     /* [B, T] 1 = placed (q_pos < n_pages * P on a mapped page) */
  int32_t *ctx_len_new;  /* [B]    c' = min(c + n, A) (advertised context length) */
  int32_t *seq_lens;     /* [B]    c' + T (kv_len of the block attention) */
} dflash_step_outputs;

/* ---------------------------------------------------------------------
 * dflash_pack_weights -- stack every drafter layer's K/V (GQA) or latent (MLA)
 * projection into the one matrix the context update's GEMM reads, and the
 * layers' norm gains into one array [TRT-13995, "per-layer cached K/V pool":
 * one GEMM stacked across the drafter layers; "fuse cross-layer k_norm": the
 * k_norm weights stacked once so one RMSNorm covers every layer].
 *
 * layers   HOST array of num_layers entries; each names that layer's device
 *          tensors (dflash_layer_weights).  w_k / w_v 16-byte aligned.
 * w_kv     device output, dflash_packed_kv_bytes(g) bytes, 16-byte aligned:
 *          GQA [L][2][nkv][head_dim][d_model] (row block 0 = w_k, 1 = w_v),
 *          MLA [L][latent_dim + rope_dim][d_model].
 * gamma_k  device output, dflash_packed_gamma_bytes(g) bytes: GQA
 *          [L][head_dim], MLA [L][latent_dim].
 * The copy is bit-exact (no conversion).  Done once at model load; the
 * outputs are the dflash_weights.w_kv / gamma_k of the context update.
 * Errors: DFLASH_ERR_INVALID_ARG (null or misaligned pointers),
 * DFLASH_ERR_UNSUPPORTED_GEOM (more than 64 layers, d_model not a multiple of
 * 8), DFLASH_ERR_CUDA.
 * ------------------------------------------------------------------- */
DFLASH_API size_t dflash_packed_kv_bytes(const dflash_geom *g);
DFLASH_API size_t dflash_packed_gamma_bytes(const dflash_geom *g);
DFLASH_API int dflash_pack_weights(const dflash_geom *g, const dflash_layer_weights *layers,
                                   void *w_kv, void *gamma_k, dflash_stream_t stream);

/* ---------------------------------------------------------------------
 * dflash_strict_accept -- acceptance of a uniform-width draft, one launch,
 * ahead of the bookkeeping [TRT-20550, follow-up commit "spec_tail_kernels.py":
 * strict acceptance of a uniform-width draft is one launch].
 *
 * Request r drafted K tokens draft[r, 0..K-1]; the target produced K + 1
 * tokens target[r, 0..K] at the same positions.  Drafts are accepted while
 * they equal the target's token; the target's token at the first
 * disagreement (or after the last draft) is the bonus:
 *   n_accepted[r] = 1 + (number of leading i with draft[r,i] == target[r,i]),
 *   accepted[r, i] = target[r, i] for i < n_accepted[r], -1 after.
 * So accepted[r, n - 1] is the bonus token dflash_step_bookkeeping reads, and
 * (accepted, K + 1, n_accepted) can be passed to it as (accepted_tokens,
 * acc_row_stride, n_accepted) with block_size = K + 1.
 *
 * draft       device int32, row r at draft + r * draft_row_stride (K entries).
 * target      device int32, row r at target + r * target_row_stride (K + 1).
 * n_accepted  device int32 [B] (out).  accepted  device int32 [B, K + 1] (out).
 * Errors: DFLASH_ERR_INVALID_ARG (null pointers, B < 0, K < 0, strides below
 * the row widths), DFLASH_ERR_CUDA.
 * ------------------------------------------------------------------- */
DFLASH_API int dflash_strict_accept(int B, int K, const int32_t *draft, int64_t draft_row_stride,
                                    const int32_t *target, int64_t target_row_stride,
                                    int32_t *n_accepted, int32_t *accepted,
                                    dflash_stream_t stream);

/* ---------------------------------------------------------------------
 * dflash_embedding_gather -- the noise block's input rows, one lookup over
 * the block's ids [TRT-13995, "fuse query-input build in pure Torch + fused
 * embedding lookup": one embed_tokens call over [bonus..., mask_token_id]].
 *
 * out[k, :] = table[ids[k], :] for k < n (e.g. ids = the bookkeeping's
 * emb_ids, n = B * T).  An id outside [0, vocab) writes a zero row and ORs
 * DFLASH_DEV_BAD_TOKEN into *dev_status.
 * ids    device int32 [n].  table  device bf16 [vocab, dim], 16-byte aligned.
 * out    device bf16 [n, dim], 16-byte aligned.
 * Errors: DFLASH_ERR_INVALID_ARG (null or misaligned pointers, n < 0,
 * vocab < 1), DFLASH_ERR_UNSUPPORTED_GEOM (dim not a positive multiple of 8),
 * DFLASH_ERR_CUDA.
 * ------------------------------------------------------------------- */
DFLASH_API int dflash_embedding_gather(int n, const int32_t *ids, const void *table, int vocab,
                                       int dim, void *out, int32_t *dev_status,
                                       dflash_stream_t stream);

/* ---------------------------------------------------------------------
 * dflash_step_bookkeeping -- one launch for the per-step bookkeeping groups
 * [TRT-20548 Proposal; TRT-20550 Description: the _refresh_ctx_block_tables
 * group, the generation prologue and the ctx_len advance, and the follow-up
 * commit: block-table decode from clamped, divided offsets, bonus token,
 * query and RoPE positions, destination pages / offsets / write mask, ctx_len advance
 * with the dummy slot emptied, advertised context length, seq_lens,
 * DraftBlockPlacement].
 *
 * raw_offsets     device int32, row r at raw_offsets + r*off_row_stride,
 *                 max_pages entries (a strided view is fine); negative = no page.
 * off_div         >= 1; decoded page = max(offset, 0) / off_div.
 * accepted_tokens device int32, row r at accepted_tokens + r*acc_row_stride,
 *                 block_size entries.
 * n_accepted      device int32 [B], accepted rows n (1..T) including the bonus.
 * ctx_len_pre     device int32 [B], context length c before the step.
 * valid           device uint8 [B] or NULL (all live); 0 = dummy slot.
 * A row is live when valid != 0, 1 <= n <= T and c >= 0; any other row is a
 * dummy: n_pages = alloc_limit = ctx_len_new = seq_lens = 0, positions 0,
 * masks 0, pages/slots -1, emb_ids and bonus = mask_token_id.  The decoded
 * table row is written for every row.
 * Errors: DFLASH_ERR_INVALID_ARG for null pointers, B < 0, off_div < 1,
 * strides below the row widths; DFLASH_ERR_CUDA when the launch fails.
 * ------------------------------------------------------------------- */
DFLASH_API int dflash_step_bookkeeping(const dflash_geom *g, int B, const int32_t *raw_offsets,
                            int64_t off_row_stride, int32_t off_div,
                            const int32_t *accepted_tokens, int64_t acc_row_stride,
                            const int32_t *n_accepted, const int32_t *ctx_len_pre,
                            const uint8_t *valid, int32_t max_ctx, int32_t mask_token_id,
                            const dflash_step_outputs *out, int32_t *dev_status,
                            dflash_stream_t stream);

/* ---------------------------------------------------------------------
 * dflash_ctx_workspace_bytes -- device scratch needed by dflash_ctx_kv_update
 * for B requests (depends on the geometry and the current device's SM count).
 * Returns 0 for an invalid geometry.
 * ------------------------------------------------------------------- */
DFLASH_API size_t dflash_ctx_workspace_bytes(const dflash_geom *g, int B);

/* ---------------------------------------------------------------------
 * dflash_ctx_kv_update -- the per-step context-KV update
 * [TRT-20548 Proposal: context-KV mask, clamp, paged write, ctx_len advance;
 * TRT-20550 Description, TLLM_DFLASH_OVERLAP_CONTEXT_PROJECTION: the fc
 * projection, hidden norm, latent projection and norm + RoPE; TRT-13995
 * "per-layer cached K/V pool" (one GEMM stacked across drafter layers on the
 * K+1 accepted rows),
 * "fuse cross-layer k_norm" (one RMSNorm over [N, L, nkv, hd], mask
 * multiply), "match RoPE between context and query" (one cos/sin
 * convention)].
 *
 * For every request r and row i < T with write mask
 *   w = live(r) && i < n_r && c_r + i < alloc_limit[r]
 *       && block_table[r, (c_r+i)/P] in [0, num_pool_pages),
 * computes  x = bf16(hidden[r, i]),  h = bf16(W_fc x),
 *           hn = bf16(h * gamma_h / sqrt(mean(h^2) + eps_hidden)),
 * then for every layer l (GQA, per KV head):
 *           k = W_k[l] hn,  v = W_v[l] hn   (fp32 accumulation),
 *           k' = RoPE(k * gamma_k[l] / sqrt(mean(k^2) + eps_k), c_r + i),
 * and stores bf16(k'), bf16(v) at (page, slot) = (block_table[r, p/P], p%P)
 * of layer l; (MLA) c = W_dkv[l] hn, stores bf16(RMSNorm(c[:lat]) * gamma)
 * || bf16(RoPE(c[lat:], p)).  RoPE is rotate-half with
 * f_j = rope_theta^(-2j/d), the angle p * f_j formed in double precision and
 * reduced modulo 2*pi before the fp32 sin/cos.  Rows with w = 0 are not
 * stored: every other pool entry is left bit-identical.  Finally, in place,
 * ctx_len[r] = live(r) ? min(c_r + n_r, alloc_limit[r]) : 0.
 *
 * hidden       device [B, T, d_in], bf16 or fp32 per hidden_dtype.
 * ctx_len      device int32 [B]: read as c (pre-step), overwritten with c'.
 * alloc_limit  device int32 [B] (e.g. from dflash_step_bookkeeping).
 * block_table  device int32 [B, max_pages] physical page ids (entry < 0 =
 *              unmapped, the row is masked).
 * valid        device uint8 [B] or NULL.
 * workspace    device scratch of at least dflash_ctx_workspace_bytes(g, B)
 *              bytes, 256-byte aligned; its contents are clobbered.
 * Errors: DFLASH_ERR_INVALID_ARG (null / misaligned pointers, B < 0, bad
 * dtype), DFLASH_ERR_UNSUPPORTED_GEOM (head_dim not a multiple of 8 or
 * > 256, d_in or d_model not a multiple of 64, MLA widths other than
 * 512 + 64), DFLASH_ERR_WORKSPACE_TOO_SMALL, DFLASH_ERR_CUDA.
 * ------------------------------------------------------------------- */
DFLASH_API int dflash_ctx_kv_update(const dflash_geom *g, int B, const void *hidden, int hidden_dtype,
                         const int32_t *n_accepted, int32_t *ctx_len,
                         const int32_t *alloc_limit, const int32_t *block_table,
                         const uint8_t *valid, const dflash_weights *w, void *kv_pool,
                         void *workspace, size_t ws_bytes, int32_t *dev_status,
                         dflash_stream_t stream);

/* ---------------------------------------------------------------------
 * dflash_ctx_kv_prefill -- the prefill-side context store: every prompt row
 * of every request through the context projection and into the paged pool
 * [TRT-20550 Description, TLLM_DFLASH_FUSED_PROLOGUE: the single-latent
 * _store_context_kv_paged scatter used by prefill].
 *
 * The rows of request r are hidden rows cu_rows[r] .. cu_rows[r+1]-1 (a
 * variable number per request; cu_rows[0] = 0, nondecreasing, cu_rows[B] =
 * n_rows).  Row i of request r sits at position p = c_r + i, c_r = ctx_len[r]
 * (0 for a fresh prompt, the chunk start for a chunked prefill), and gets the
 * values dflash_ctx_kv_update computes for an accepted row: x = bf16(hidden),
 * h = bf16(W_fc x), hn = bf16(RMSNorm(h)), per layer GQA k' = RoPE(RMSNorm(W_k
 * hn), p) and v = W_v hn, MLA bf16(RMSNorm(c[:lat])) || bf16(RoPE(c[lat:], p)).
 * It is stored when the request is live (valid != 0 and c_r >= 0), p is below
 * alloc_limit[r] and block_table[r, p / P] is a page inside the pool; nothing
 * else in the pool changes.  Then, in place, ctx_len[r] = live ?
 * min(c_r + n_r, alloc_limit[r]) : 0.  A row outside every request's range
 * (cu_rows inconsistent with n_rows) is skipped.
 *
 * n_rows      host int, 0 .. 65535 rows per call (chunk longer prompts).
 * hidden      device [n_rows, d_in], bf16 or fp32 per hidden_dtype.
 * cu_rows     device int32 [B + 1].
 * workspace   device scratch of dflash_ctx_prefill_workspace_bytes(g, B,
 *             n_rows) bytes (grows with n_rows), 256-byte aligned.
 * Other arguments as dflash_ctx_kv_update.  Errors: as dflash_ctx_kv_update,
 * plus DFLASH_ERR_UNSUPPORTED_GEOM for n_rows > 65535.
 * ------------------------------------------------------------------- */
DFLASH_API size_t dflash_ctx_prefill_workspace_bytes(const dflash_geom *g, int B, int n_rows);
DFLASH_API int dflash_ctx_kv_prefill(const dflash_geom *g, int B, int n_rows, const void *hidden,
                                     int hidden_dtype, const int32_t *cu_rows, int32_t *ctx_len,
                                     const int32_t *alloc_limit, const int32_t *block_table,
                                     const uint8_t *valid, const dflash_weights *w, void *kv_pool,
                                     void *workspace, size_t ws_bytes, int32_t *dev_status,
                                     dflash_stream_t stream);

/* ---------------------------------------------------------------------
 * Split context update: dflash_ctx_kv_project + dflash_ctx_kv_commit
 * [TRT-20550 Description, TLLM_DFLASH_OVERLAP_CONTEXT_PROJECTION: the
 * context projection of the generation tokens is forked onto an auxiliary
 * stream before sampling / acceptance and joined before the accepted-mask
 * write; it reads only the target hidden states and the pre-step ctx_len].
 *
 * dflash_ctx_kv_project computes, for EVERY row (r, i < T), the values
 * dflash_ctx_kv_update would store -- GQA bf16(k'), bf16(v) of every layer
 * and KV head, MLA the bf16 latent row -- with RoPE at c_r + i, and writes
 * them to `staged` together with the c_r it used.  n_accepted, the masks and
 * the pool are not needed, so it can run before acceptance.
 * dflash_ctx_kv_commit then does the write-masked paged store of the staged
 * rows and the ctx_len advance, exactly as dflash_ctx_kv_update: the pool and
 * ctx_len after project + commit are bit-identical to the fused call's.  The
 * advance starts from the c_r recorded by the projection.
 *
 * staged       device scratch of dflash_ctx_staged_bytes(g, B) bytes,
 *              256-byte aligned, owned by the caller: int32 c [B] at offset
 *              0, then bf16 rows [B * T][W] at offset round_up(4 B, 256),
 *              W = L * 2 * nkv * head_dim (GQA, per row [L][K|V][nkv][hd])
 *              or L * (latent_dim + rope_dim) (MLA, [L][latent | rope]).
 *              Written by project, read by commit; nothing else may write it
 *              in between.
 * workspace    (project) as for dflash_ctx_kv_update; a project and a fused
 *              update must not share a workspace concurrently.
 * ctx_len      project reads it (the pre-step lengths); commit overwrites it
 *              with c'.
 * Other arguments and errors as for dflash_ctx_kv_update;
 * DFLASH_ERR_WORKSPACE_TOO_SMALL also when staged_bytes is short.
 * ------------------------------------------------------------------- */
DFLASH_API size_t dflash_ctx_staged_bytes(const dflash_geom *g, int B);
DFLASH_API int dflash_ctx_kv_project(const dflash_geom *g, int B, const void *hidden,
                          int hidden_dtype, const int32_t *ctx_len, const dflash_weights *w,
                          void *staged, size_t staged_bytes, void *workspace, size_t ws_bytes,
                          int32_t *dev_status, dflash_stream_t stream);
DFLASH_API int dflash_ctx_kv_commit(const dflash_geom *g, int B, const void *staged,
                         size_t staged_bytes, const int32_t *n_accepted, int32_t *ctx_len,
                         const int32_t *alloc_limit, const int32_t *block_table,
                         const uint8_t *valid, void *kv_pool, int32_t *dev_status,
                         dflash_stream_t stream);

/* ---------------------------------------------------------------------
 * dflash_q_norm_rope -- the query side of one drafter layer
 * [TRT-13995 "use fused qk-norm+rope on non-YaRN draft", "match RoPE between
 * context and query": query norm and rotation in one kernel, with the cos/sin
 * the context keys are rotated with].
 *
 * GQA: for every request r, query token i < Tq and head h,
 *   q_out[r, i, h] = bf16(RoPE(q * gamma_q / sqrt(mean(q^2) + eps_k),
 *                               q_pos[r, i]))   over head_dim,
 * q = q_in[r, i, h]; eps is the geometry's eps_k and the rotation the
 * rotate-half RoPE of dflash_ctx_kv_update (same frequency table and angle
 * code, so a query and a context key at the same position get the same
 * cos/sin).  MLA: gamma_q must be NULL and only the rotation is applied, to
 * the rope part of the query (rows of rope_dim).
 *
 * q_in, q_out  device bf16 [B, Tq, hq, head_dim] (MLA: [B, Tq, hq, rope_dim]);
 *              q_out may equal q_in.
 * gamma_q      device bf16 [head_dim] (the layer's query-norm gain), or NULL
 *              for MLA.
 * q_pos        device int32 [B, Tq] (e.g. dflash_step_outputs.q_pos).
 * Errors: DFLASH_ERR_INVALID_ARG (null / odd pointers, gamma_q given for MLA
 * or missing for GQA), DFLASH_ERR_UNSUPPORTED_GEOM (an odd or > 256 rotated
 * width), DFLASH_ERR_CUDA.
 * ------------------------------------------------------------------- */
DFLASH_API int dflash_q_norm_rope(const dflash_geom *g, int B, int Tq, const void *q_in,
                       const void *gamma_q, const int32_t *q_pos, void *q_out,
                       int32_t *dev_status, dflash_stream_t stream);

/* ---------------------------------------------------------------------
 * dflash_block_kv_scatter -- write the block's own K/V (GQA) or latent rows
 * (MLA) of one layer into the pool at the DraftBlockPlacement
 * [TRT-20548 Proposal: each layer writes its block latents into the pool;
 * TRT-20550 Description: that write is one scatter kernel per layer].
 *
 * blk_k    GQA: device bf16 [B, T, nkv, head_dim]; MLA: [B, T, latent+rope].
 * blk_v    GQA: device bf16 [B, T, nkv, head_dim]; MLA: must be NULL.
 * blk_page, blk_slot  device int32 [B, T]; blk_mask device uint8 [B, T].
 * Rows with blk_mask = 0 are skipped; a placed row whose page is outside the
 * pool or slot outside [0, P) is skipped and flags DFLASH_DEV_BAD_PAGE.
 * Errors: DFLASH_ERR_INVALID_ARG, DFLASH_ERR_CUDA.
 * ------------------------------------------------------------------- */
DFLASH_API int dflash_block_kv_scatter(const dflash_geom *g, int B, int layer, const void *blk_k,
                            const void *blk_v, const int32_t *blk_page,
                            const int32_t *blk_slot, const uint8_t *blk_mask, void *kv_pool,
                            int32_t *dev_status, dflash_stream_t stream);

/* ---------------------------------------------------------------------
 * dflash_attention_num_segments -- the split count `num_segments = 0`
 * resolves to for this geometry and batch (a launch heuristic that fills the
 * GPU's SMs; it never depends on device data).
 * dflash_attention_workspace_bytes -- scratch for dflash_block_attention with
 * that many segments (0 = the automatic count).  0 for invalid arguments.
 * ------------------------------------------------------------------- */
DFLASH_API int dflash_attention_num_segments(const dflash_geom *g, int B, int Tq);
DFLASH_API size_t dflash_attention_workspace_bytes(const dflash_geom *g, int B, int Tq, int num_segments);

/* ---------------------------------------------------------------------
 * dflash_block_attention -- decode-shaped block attention of one drafter
 * layer over the paged cache, split over KV segments, with an optional
 * sliding window and per-head sink logits [VLLM-54092 Purpose 2 and
 * Changes 2: 3D split-KV for small uniform q (1 bonus + N drafts), per-query-
 * token segment buffers, segments over the keys the window leaves visible,
 * one layout for the main kernel and the reduce; sinks].
 *
 * For request r, query token i < Tq and head h (kv head h / (hq/nkv)):
 *   p_i = kv_len[r] - Tq + i,
 *   visible keys j: lo_i <= j <= hi_i with hi_i = p_i (CAUSAL_TAIL) or
 *   kv_len[r]-1 (BLOCK_BIDIR), lo_i = window > 0 ? max(0, p_i-window+1) : 0,
 *   s_j = scale * <q, k_j>,  M = max(max_j s_j, sink_h),
 *   out = sum_j e^(s_j-M) v_j / (sum_j e^(s_j-M) + e^(sink_h-M))
 * (no sink term when sinks == NULL; out = 0 when no key is visible).
 * Key j lives at page block_table[r, j/P], slot j%P of layer `layer`.
 * The visible span [lo_0, hi_{Tq-1}] is cut into num_segments slices of whole
 * 128-key tiles; each (request, kv head, slice) CTA -- one per 128 query rows
 * (64 for MLA) of the kv head's group, rows being (token, head) pairs --
 * writes a partial (max, sum, weighted values) to the workspace and a second
 * pass merges them (log-sum-exp) with the sink.
 *
 * GQA: q device bf16 [B, Tq, hq, head_dim]; q_rope NULL; out bf16
 *      [B, Tq, hq, head_dim].
 * MLA: q device bf16 [B, Tq, hq, latent] (absorbed latent query), q_rope
 *      bf16 [B, Tq, hq, rope]; s_j = scale*(<q, c_j> + <q_rope, r_j>),
 *      values c_j; out bf16 [B, Tq, hq, latent].
 * kv_len      device int32 [B] (seq_lens of the bookkeeping).
 * sinks       device fp32 [hq] or NULL.
 * scale       softmax scale; scale <= 0 selects the default, 1/sqrt(head_dim)
 *             for GQA and 1/sqrt(128 + rope_dim) for MLA (the scale of the
 *             unabsorbed head: a 128-wide no-rope part plus the rope part).
 * num_segments 0 = automatic, else >= 1.
 * workspace   device scratch >= dflash_attention_workspace_bytes(...), 16-byte
 *             aligned; clobbered.
 * Errors: DFLASH_ERR_INVALID_ARG (also: scale not finite, window < 0,
 * unknown mask_mode, a pointer not 16-byte aligned), DFLASH_ERR_UNSUPPORTED_GEOM
 * (hq not a multiple of nkv, GQA head_dim not 64 or 128, MLA dims not 512 + 64,
 * page_size not a multiple of 8 that divides 128 or is a multiple of 128, pool
 * rows >= 2^31), DFLASH_ERR_WORKSPACE_TOO_SMALL, DFLASH_ERR_CUDA.
 * ------------------------------------------------------------------- */
DFLASH_API int dflash_block_attention(const dflash_geom *g, int B, int layer, int Tq, const void *q,
                           const void *q_rope, const void *kv_pool,
                           const int32_t *block_table, const int32_t *kv_len, int32_t window,
                           const float *sinks, float scale, int mask_mode, int num_segments,
                           void *workspace, size_t ws_bytes, void *out, int32_t *dev_status,
                           dflash_stream_t stream);

/* ---------------------------------------------------------------------
 * dflash_block_scatter_attention -- dflash_block_kv_scatter followed by
 * dflash_block_attention on the same layer, in one launch pair (main kernel
 * + merge) instead of three: the two calls the pages run back to back for
 * every drafter layer [TRT-20550 Description: the per-layer block scatter;
 * VLLM-54092 Purpose 2: the split-KV block attention that reads it].
 *
 * Arguments: those of dflash_block_kv_scatter (blk_k, blk_v, blk_page,
 * blk_slot, blk_mask, kv_pool) and of dflash_block_attention, with
 * Tq == g->block_size.  The result -- the pool and `out` -- is the one the two
 * calls give in that order, provided the placement is the bookkeeping's: the
 * block's row i sits at the position kv_len[r] - Tq + i (dflash_step_outputs
 * blk_page / blk_slot / blk_mask with kv_len = seq_lens), and its pool slot is
 * read by this call at that position only (the block's pages are the
 * request's own).  Each attention CTA writes the block rows of its own key
 * range before it copies those keys; rows no range reads (kv_len < Tq) are
 * still written.  Those CTAs start copying later by the scatter's memory
 * round trips: the fused form is faster where their segment is shorter than
 * the others and the grid is one wave (a long context, few requests); with
 * one-tile segments or several waves the two calls are faster.
 * Errors: those of the two calls; DFLASH_ERR_INVALID_ARG also for
 * Tq != g->block_size.
 * ------------------------------------------------------------------- */
DFLASH_API int dflash_block_scatter_attention(
    const dflash_geom *g, int B, int layer, int Tq, const void *blk_k, const void *blk_v,
    const int32_t *blk_page, const int32_t *blk_slot, const uint8_t *blk_mask, const void *q,
    const void *q_rope, void *kv_pool, const int32_t *block_table, const int32_t *kv_len,
    int32_t window, const float *sinks, float scale, int mask_mode, int num_segments,
    void *workspace, size_t ws_bytes, void *out, int32_t *dev_status, dflash_stream_t stream);

/* ---------------------------------------------------------------------
 * dflash_block_attention_noalloc -- the same computation as
 * dflash_block_attention, for callers that cannot allocate device memory
 * where they run it: a plugin whose host framework owns every device buffer
 * and gives it no allocator, or a real-time loop that must not block in an
 * allocator.  The caller passes inputs and output as for
 * dflash_block_attention; the split-KV scratch comes from one fixed array
 * inside the library.  The pages describe no such entry point: it is a
 * convenience of this library, with no counterpart in the method.
 *
 * Scratch: a file-scope device array of
 * dflash_block_attention_noalloc_max_scratch_bytes() bytes (32 MiB), present
 * on every GPU that loads the library until the process exits.  A call whose
 * dflash_attention_workspace_bytes(g, B, Tq, num_segments) exceeds it returns
 * DFLASH_ERR_WORKSPACE_TOO_SMALL and launches nothing.  The array is shared by
 * every call and keeps the last call's contents; nothing in it has to start
 * at zero.  Calls whose GPU work overlaps (on other streams, for example) race
 * on it: serialise them.
 * Set-up: the first call on each device looks up the array's device address
 * (with that device current) and caches it.  The call allocates nothing and
 * calls no allocating routine.
 * Errors: the argument checks of dflash_block_attention come first and give
 * the same codes; then DFLASH_ERR_WORKSPACE_TOO_SMALL for a problem larger
 * than the fixed scratch, and DFLASH_ERR_CUDA when the address look-up fails.
 * The scratch address is that of the current device, which must be the
 * device of `stream`.
 * ------------------------------------------------------------------- */
DFLASH_API int dflash_block_attention_noalloc(const dflash_geom *g, int B, int layer, int Tq,
                                              const void *q, const void *q_rope,
                                              const void *kv_pool, const int32_t *block_table,
                                              const int32_t *kv_len, int32_t window,
                                              const float *sinks, float scale, int mask_mode,
                                              int num_segments, void *out, int32_t *dev_status,
                                              dflash_stream_t stream);

/* Size in bytes of the fixed scratch used by dflash_block_attention_noalloc. */
DFLASH_API size_t dflash_block_attention_noalloc_max_scratch_bytes(void);

/* ---------------------------------------------------------------------
 * dflash_test_attention_skip_tile -- for tests of the bounded-wait path only.
 * While set (tile >= 0), every dflash_block_attention launched from the
 * calling host thread leaves key tile `tile` of each CTA's segment unloaded
 * (MLA: the first 64-key half of it): the wait for it runs out (about 2 s),
 * the kernel winds down, ORs
 * DFLASH_DEV_WAIT_TIMEOUT into *dev_status and the context stays usable.
 * tile < 0 turns it off (the default).  Never set it in production.
 * ------------------------------------------------------------------- */
DFLASH_API void dflash_test_attention_skip_tile(int tile);

/* Human-readable name of a dflash_status_code (static string). */
DFLASH_API const char *dflash_status_string(int code);

/* Library ABI version (increments when a signature changes). */
DFLASH_API int dflash_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH_H */
