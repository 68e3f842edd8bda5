// ctx_update.cu -- the per-step context-KV update.
//
// Follows TensorRT-LLM PR #20550 (Description, TLLM_DFLASH_OVERLAP_CONTEXT_
// PROJECTION: "fc + hidden_norm + latent GEMM + RMSNorm/RoPE" on the gen
// tokens, then the accepted-mask write) and PR #13995 ("migrate draft path to
// per-layer cached K/V pool": one GEMM stacked across the drafter layers on
// the newly accepted K+1 rows; "fuse cross-layer k_norm and avoid mask-mul
// alloc": one RMSNorm over [N, L, nkv, hd] with stacked per-layer weights and
// a shared eps; "match RoPE between context and query": one cos/sin
// convention).
//
// Launch chain on the caller's stream:
//   prep      ctx_len snapshot (+ fp32 -> bf16 of the hidden rows)
//   gemm      Y1 = X W_fc^T            (weights streamed once)
//   norm      hn = bf16(bf16(Y1) * gamma_h / rms)
//   gemm      Y2 = hn W_kv^T           (all layers' K/V rows in one pass)
//   epilogue  k RMSNorm + RoPE (GQA) / latent RMSNorm + RoPE (MLA), masked
//             paged bf16 store, ctx_len advance
#include "dflash_internal.cuh"
#include "gemm_tc.cuh"

namespace dflash {
namespace {

// ----------------------------------------------------------- workspace map
struct CtxWs {
  int32_t *ctx_snap;  // [B]
  int *counters;      // stream-K tile tickets: fc tiles, then K/V tiles
  int n_counters;
  uint16_t *x;        // [Npad, D_in] bf16 (fp32 hidden converted)
  uint16_t *hn;       // [Npad, D]    bf16
  float *y1;          // [N, D]     fc output
  float *y2;          // [N, Wrows] K/V (or latent) projection
  float *part1;       // fc partial tiles
  float *part2;       // K/V partial tiles
  size_t bytes;
};

struct CtxDims {
  int N, Npad, D_in, D, Wrows;
};

CtxDims ctx_dims(const dflash_geom &g, int B) {
  CtxDims d;
  d.N = B * g.block_size;
  d.Npad = static_cast<int>(align_up(static_cast<size_t>(d.N > 0 ? d.N : 1), 16));
  d.D_in = g.d_in;
  d.D = g.d_model;
  d.Wrows = (g.kind == DFLASH_KIND_GQA) ? g.num_layers * 2 * g.nkv * g.head_dim
                                        : g.num_layers * (g.latent_dim + g.rope_dim);
  return d;
}

CtxWs ctx_ws_map(const dflash_geom &g, int B, void *base) {
  const CtxDims d = ctx_dims(g, B);
  char *p = static_cast<char *>(base);
  size_t off = 0;
  CtxWs w;
  w.ctx_snap = reinterpret_cast<int32_t *>(p + off);
  off = align_up(off + sizeof(int32_t) * (B > 0 ? B : 1), 256);
  w.counters = reinterpret_cast<int *>(p + off);
  w.n_counters = gemm_num_tiles(d.D, d.Npad) + gemm_num_tiles(d.Wrows, d.Npad);
  off = align_up(off + sizeof(int) * w.n_counters, 256);
  w.y1 = reinterpret_cast<float *>(p + off);
  off = align_up(off + sizeof(float) * d.Npad * d.D, 256);
  w.y2 = reinterpret_cast<float *>(p + off);
  off = align_up(off + sizeof(float) * static_cast<size_t>(d.Npad) * d.Wrows, 256);
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

// ------------------------------------------------------------------ prep
__global__ void prep_kernel(const float *hidden_f32, uint16_t *x, int n_elems, int row_elems,
                            int n_pad_rows, const int32_t *ctx_len, int32_t *ctx_snap, int B,
                            int *counters, int n_counters) {
  griddep_launch();
  griddep_wait();
  const int tid = blockIdx.x * blockDim.x + threadIdx.x;
  if (tid < B) ctx_snap[tid] = ctx_len[tid];
  for (int k = tid; k < n_counters; k += gridDim.x * blockDim.x) counters[k] = 0;
  if (hidden_f32 == nullptr) return;
  const int total = n_pad_rows * row_elems;
  for (int e = tid; e < total; e += gridDim.x * blockDim.x)
    x[e] = e < n_elems ? f32_to_bf16_rn(hidden_f32[e]) : static_cast<uint16_t>(0);
}

// ----------------------------------------------------- hidden RMSNorm
// One CTA per row: h = bf16(sum of partials), hn = bf16(h * g / rms(h)).
__global__ void __launch_bounds__(1024) hidden_norm_kernel(const float *y, const uint16_t *gamma,
                                                           uint16_t *hn, int D, float eps) {
  __shared__ float red[32];
  extern __shared__ float hbuf[];  // [D]
  griddep_launch();
  griddep_wait();
  const int n = blockIdx.x;
  const float *row = y + static_cast<size_t>(n) * D;
  float ss = 0.f;
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    const float h = bf16_to_f32(f32_to_bf16_rn(row[d]));
    hbuf[d] = h;
    ss += h * h;
  }
  ss = block_sum(ss, red);
  const float inv = rsqrtf(ss / static_cast<float>(D) + eps);
  for (int d = threadIdx.x; d < D; d += blockDim.x)
    hn[static_cast<size_t>(n) * D + d] = f32_to_bf16_rn(hbuf[d] * inv * bf16_to_f32(gamma[d]));
}

// ----------------------------------------------------------- write mask
struct MaskArgs {
  const int32_t *n_acc;
  const int32_t *ctx_snap;
  const int32_t *alloc_limit;
  const int32_t *tbl;
  const uint8_t *valid;
  int T, M, P, NP;
  int32_t *st;
};

// Destination of context row (r, i), or false when the row is not written.
__device__ __forceinline__ bool ctx_row_dest(const MaskArgs &m, int r, int i, int *page, int *slot,
                                             int *pos, bool report) {
  const int n = m.n_acc[r];
  const int c = m.ctx_snap[r];
  const bool live = m.valid ? (m.valid[r] != 0) : true;
  if (!live || n < 1 || n > m.T || c < 0 || i >= n) return false;
  const int p = c + i;
  if (p >= m.alloc_limit[r]) return false;
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

// ------------------------------------------------------ GQA epilogue
// grid (N rows, L*2*nkv heads), block = head_dim threads.
__global__ void epilogue_gqa_kernel(const float *y, int ldy, const MaskArgs m, const RopeFreqs rf,
                                    const uint16_t *gamma_k, uint16_t *pool, int L, int nkv,
                                    int hd, float eps, int32_t *ctx_len, int B) {
  __shared__ float red[32];
  __shared__ float kbuf[kMaxHeadDim];
  griddep_launch();
  griddep_wait();
  const int n = blockIdx.x;
  const int head = blockIdx.y;  // ((l * 2 + kv) * nkv + h)
  const int d = threadIdx.x;
  if (n == 0 && head == 0) {
    // ctx_len advance; every reader of the pre-step value uses the snapshot.
    for (int r = d; r < B; r += blockDim.x) {
      const int nn = m.n_acc[r], c = m.ctx_snap[r];
      const bool live = (m.valid ? (m.valid[r] != 0) : true) && nn >= 1 && nn <= m.T && c >= 0;
      const long long s = static_cast<long long>(c) + nn;
      const int A = m.alloc_limit[r];
      ctx_len[r] = live ? static_cast<int>(s < A ? s : A) : 0;
    }
  }
  const int r = n / m.T, i = n % m.T;
  int page, slot, pos;
  if (!ctx_row_dest(m, r, i, &page, &slot, &pos, head == 0 && d == 0)) return;
  const int l = head / (2 * nkv);
  const int kv = (head / nkv) & 1;
  const int h = head % nkv;
  float v = y[static_cast<size_t>(n) * ldy + head * hd + d];
  if (kv == 0) {
    const float ss = block_sum(v * v, red);
    const float inv = rsqrtf(ss / static_cast<float>(hd) + eps);
    const float kn = v * inv * bf16_to_f32(gamma_k[static_cast<size_t>(l) * hd + d]);
    kbuf[d] = kn;
    __syncthreads();
    const int half = hd >> 1;
    const int j = d < half ? d : d - half;
    float c, s;
    rope_cos_sin(pos, rf.f[j], &c, &s);
    v = d < half ? kn * c - kbuf[d + half] * s : kn * c + kbuf[d - half] * s;
  }
  const size_t dst =
      ((((static_cast<size_t>(l) * m.NP + page) * 2 + kv) * nkv + h) * m.P + slot) * hd + d;
  pool[dst] = f32_to_bf16_rn(v);
}

// ------------------------------------------------------ MLA epilogue
// grid (N rows, L), block = lat + rope threads.
__global__ void epilogue_mla_kernel(const float *y, int ldy, const MaskArgs m, const RopeFreqs rf,
                                    const uint16_t *gamma_kv, uint16_t *pool, int L, int lat,
                                    int rope, float eps, int32_t *ctx_len, int B) {
  __shared__ float red[32];
  __shared__ float rbuf[kMaxHeadDim];
  griddep_launch();
  griddep_wait();
  const int n = blockIdx.x;
  const int l = blockIdx.y;
  const int d = threadIdx.x;
  const int W = lat + rope;
  if (n == 0 && l == 0) {
    for (int r = d; r < B; r += blockDim.x) {
      const int nn = m.n_acc[r], c = m.ctx_snap[r];
      const bool live = (m.valid ? (m.valid[r] != 0) : true) && nn >= 1 && nn <= m.T && c >= 0;
      const long long s = static_cast<long long>(c) + nn;
      const int A = m.alloc_limit[r];
      ctx_len[r] = live ? static_cast<int>(s < A ? s : A) : 0;
    }
  }
  const int r = n / m.T, i = n % m.T;
  int page, slot, pos;
  if (!ctx_row_dest(m, r, i, &page, &slot, &pos, l == 0 && d == 0)) return;
  const float v = y[static_cast<size_t>(n) * ldy + l * W + d];
  const float ss = block_sum(d < lat ? v * v : 0.f, red);
  float outv;
  if (d < lat) {
    const float inv = rsqrtf(ss / static_cast<float>(lat) + eps);
    outv = v * inv * bf16_to_f32(gamma_kv[static_cast<size_t>(l) * lat + d]);
  } else {
    rbuf[d - lat] = v;
  }
  __syncthreads();
  if (d >= lat) {
    const int e = d - lat, half = rope >> 1;
    const int j = e < half ? e : e - half;
    float c, s;
    rope_cos_sin(pos, rf.f[j], &c, &s);
    outv = e < half ? v * c - rbuf[e + half] * s : v * c + rbuf[e - half] * s;
  }
  const size_t dst = ((static_cast<size_t>(l) * m.NP + page) * m.P + slot) * W + d;
  pool[dst] = f32_to_bf16_rn(outv);
}

}  // namespace

size_t ctx_workspace_bytes(const dflash_geom &g, int B) { return ctx_ws_map(g, B, nullptr).bytes; }

cudaError_t launch_ctx_kv_update(const dflash_geom &g, int B, const void *hidden, int hidden_dtype,
                                 const int32_t *n_acc, int32_t *ctx_len, const int32_t *alloc_limit,
                                 const int32_t *tbl, const uint8_t *valid, const dflash_weights &w,
                                 void *pool, void *ws, int32_t *st, cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  const CtxDims d = ctx_dims(g, B);
  const CtxWs W = ctx_ws_map(g, B, ws);
  cudaError_t e;

  // prep: ctx_len snapshot, fp32 hidden -> bf16
  const bool f32 = hidden_dtype == DFLASH_DTYPE_F32;
  {
    const int threads = 256;
    int blocks = f32 ? (d.Npad * d.D_in + threads - 1) / threads : 1;
    if (blocks > 4 * device_sm_count()) blocks = 4 * device_sm_count();
    if (blocks * threads < B) blocks = (B + threads - 1) / threads;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(threads);
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((e = cudaLaunchKernelEx(&cfg, prep_kernel,
                                f32 ? static_cast<const float *>(hidden) : nullptr, W.x,
                                d.N * d.D_in, d.D_in, d.Npad, ctx_len, W.ctx_snap, B, W.counters,
                                W.n_counters)) !=
        cudaSuccess)
      return e;
  }
  const uint16_t *X = f32 ? W.x : static_cast<const uint16_t *>(hidden);

  // fc GEMM
  const int n_fc_tiles = gemm_num_tiles(d.D, d.Npad);
  if ((e = launch_gemm(X, d.N, d.D_in, static_cast<const uint16_t *>(w.w_fc), d.D, W.part1, W.y1,
                       W.counters, /*pdl=*/true, s)) != cudaSuccess)
    return e;

  // hidden RMSNorm
  {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(d.N);
    cfg.blockDim = dim3(1024);
    cfg.dynamicSmemBytes = sizeof(float) * d.D;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((e = ensure_smem_limit(hidden_norm_kernel, 64 * 1024)) != cudaSuccess) return e;
    if ((e = cudaLaunchKernelEx(&cfg, hidden_norm_kernel, static_cast<const float *>(W.y1),
                                static_cast<const uint16_t *>(w.gamma_h), W.hn, d.D,
                                static_cast<float>(g.eps_hidden))) != cudaSuccess)
      return e;
  }

  // stacked K/V (or latent) GEMM over every layer
  if ((e = launch_gemm(W.hn, d.N, d.D, static_cast<const uint16_t *>(w.w_kv), d.Wrows, W.part2,
                       W.y2, W.counters + n_fc_tiles, /*pdl=*/true, s)) != cudaSuccess)
    return e;

  // epilogue
  MaskArgs m;
  m.n_acc = n_acc;
  m.ctx_snap = W.ctx_snap;
  m.alloc_limit = alloc_limit;
  m.tbl = tbl;
  m.valid = valid;
  m.T = g.block_size;
  m.M = g.max_pages;
  m.P = g.page_size;
  m.NP = g.num_pool_pages;
  m.st = st;
  RopeFreqs rf;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.stream = s;
  if (g.kind == DFLASH_KIND_GQA) {
    fill_rope_freqs(&rf, g.head_dim, g.rope_theta);
    cfg.gridDim = dim3(d.N, g.num_layers * 2 * g.nkv);
    cfg.blockDim = dim3(g.head_dim);
    e = cudaLaunchKernelEx(&cfg, epilogue_gqa_kernel, static_cast<const float *>(W.y2), d.Wrows, m, rf,
                           static_cast<const uint16_t *>(w.gamma_k), static_cast<uint16_t *>(pool),
                           g.num_layers, g.nkv, g.head_dim, static_cast<float>(g.eps_k), ctx_len, B);
  } else {
    fill_rope_freqs(&rf, g.rope_dim, g.rope_theta);
    cfg.gridDim = dim3(d.N, g.num_layers);
    cfg.blockDim = dim3(g.latent_dim + g.rope_dim);
    e = cudaLaunchKernelEx(&cfg, epilogue_mla_kernel, static_cast<const float *>(W.y2), d.Wrows, m, rf,
                           static_cast<const uint16_t *>(w.gamma_k), static_cast<uint16_t *>(pool),
                           g.num_layers, g.latent_dim, g.rope_dim, static_cast<float>(g.eps_k),
                           ctx_len, B);
  }
  return e;
}

}  // namespace dflash
