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
// Up to 64 rows the fc GEMM runs as 4-CTA clusters that finish h = bf16(Y1)
// and its per-slice sums of squares themselves (and, in an idle warp, the
// epilogue's row set-up: destination and RoPE cos/sin per row), and the norm
// is an elementwise pass; up to 256 rows the norm is a cluster per row and
// the epilogue a CTA per (row, head); beyond (prefill, large batches) one CTA
// per row of 16-byte loads, with the row destinations resolved once by a row
// set-up kernel, and an epilogue of 16-byte loads and 8-byte stores.
#include <algorithm>

#include "ctx_rows.cuh"
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
  int4 *dst;          // [Npad] row destinations (many-row epilogue)
  float2 *cs;         // [Npad][nf] RoPE cos/sin per row (many-row epilogue)
  uint16_t *h;        // [64][D] bf16(Y1) from the cluster fc GEMM (up to 64 rows)
  float *ssq;         // [D / 32][64] per-slice sums of h^2 (cluster fc GEMM)
  size_t bytes;
};

struct CtxDims {
  int N, Npad, D_in, D, Wrows, nf;
};

CtxDims ctx_dims_rows(const dflash_geom &g, int N) {
  CtxDims d;
  d.N = N;
  d.Npad = static_cast<int>(align_up(static_cast<size_t>(d.N > 0 ? d.N : 1), 16));
  d.D_in = g.d_in;
  d.D = g.d_model;
  d.Wrows = (g.kind == DFLASH_KIND_GQA) ? g.num_layers * 2 * g.nkv * g.head_dim
                                        : g.num_layers * (g.latent_dim + g.rope_dim);
  d.nf = (g.kind == DFLASH_KIND_GQA) ? g.head_dim / 2 : g.rope_dim / 2;
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
  w.dst = reinterpret_cast<int4 *>(p + off);
  off = align_up(off + sizeof(int4) * d.Npad, 256);
  w.cs = reinterpret_cast<float2 *>(p + off);
  off = align_up(off + sizeof(float2) * d.Npad * d.nf, 256);
  const size_t hrows = d.N <= 64 ? 64 : 0;
  w.h = reinterpret_cast<uint16_t *>(p + off);
  off = align_up(off + sizeof(uint16_t) * hrows * d.D, 256);
  w.ssq = reinterpret_cast<float *>(p + off);
  off = align_up(off + sizeof(float) * hrows * (d.D / 32), 256);
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

// hn = bf16(h * gamma_h / rms(h)) when the cluster fc GEMM has already formed
// h = bf16(Y1) and each row's sum of squares in nsl 32-feature slices: CTA
// (x, n) normalises columns 512x .. 512x + 511 of row n, 8 a thread, and adds
// the row's slices in the same order as every other CTA of the row (one rms
// per row).  CTA (0, 0) also snapshots ctx_len for the epilogue.
__global__ void __launch_bounds__(64) hidden_norm_h_kernel(
    const uint16_t *h, const float *ssq, int nsl, int rows, const uint16_t *gamma, uint16_t *hn,
    int D, float eps, const int32_t *ctx_len, int32_t *ctx_snap, int B) {
  __shared__ float red[2];
  griddep_launch();
  const int n = blockIdx.y, tid = threadIdx.x;
  const int c0 = blockIdx.x * 512 + tid * 8;
  const bool in = c0 < D;
  const uint4 gv = in ? *reinterpret_cast<const uint4 *>(gamma + c0) : make_uint4(0, 0, 0, 0);
  griddep_wait();
  if (n == 0 && blockIdx.x == 0)
    for (int r = tid; r < B; r += 64) ctx_snap[r] = ctx_len[r];
  const uint4 hv = in ? *reinterpret_cast<const uint4 *>(h + static_cast<size_t>(n) * D + c0)
                      : make_uint4(0, 0, 0, 0);
  float part = 0.f;
  for (int sl = tid; sl < nsl; sl += 64) part += ssq[static_cast<size_t>(sl) * rows + n];
  part = warp_sum(part);
  if ((tid & 31) == 0) red[tid >> 5] = part;
  __syncthreads();
  const float inv = rsqrtf((red[0] + red[1]) / static_cast<float>(D) + eps);
  if (in) {
    const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float h0 = __uint_as_float(hw[k] << 16), h1 = __uint_as_float(hw[k] & 0xffff0000u);
      const float g0 = __uint_as_float(gw[k] << 16), g1 = __uint_as_float(gw[k] & 0xffff0000u);
      o[k] = static_cast<uint32_t>(f32_to_bf16_rn(h0 * inv * g0)) |
             (static_cast<uint32_t>(f32_to_bf16_rn(h1 * inv * g1)) << 16);
    }
    *reinterpret_cast<uint4 *>(hn + static_cast<size_t>(n) * D + c0) =
        make_uint4(o[0], o[1], o[2], o[3]);
  }
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

// ------------------------------------------- many rows (prefill, large batches)
// Beyond kClusterNormMaxRows rows the norm and the epilogue trade per-row
// parallelism for bytes in flight: thousands of small CTAs, each waiting on a
// few 4-byte loads, leave HBM idle.  Here every thread moves 16-byte vectors
// and issues all its loads before it adds any.

// Y[n, col..col+3] as a float4, the tile's partials added in CTA order (the
// order gemm_out_finish uses).  The second partial's load goes out with the
// first; any further ones follow.
struct Vec4Load {
  float4 a, b;
  int cnt;
};

__device__ __forceinline__ float4 add4(float4 x, float4 y) {
  return make_float4(x.x + y.x, x.y + y.y, x.z + y.z, x.w + y.w);
}

__device__ __forceinline__ const float *vec4_src(const GemmOut &g, int n, int col, unsigned *t) {
  const int nt = n / g.ntile, nr = n - nt * g.ntile;
  *t = static_cast<unsigned>(nt) * g.mtiles + static_cast<unsigned>(col >> 7);
  const size_t stride = static_cast<size_t>(g.ntile) * 128;
  return g.part + static_cast<size_t>(*t) * g.maxc * stride + static_cast<size_t>(nr) * 128 +
         (col & 127);
}

__device__ __forceinline__ void vec4_issue(const GemmOut &g, int n, int col, bool on, Vec4Load &v) {
  unsigned t;
  const float *src = vec4_src(g, n, col, &t);
  const size_t stride = static_cast<size_t>(g.ntile) * 128;
  v.cnt = on ? gemm_tile_parts(g, t) : 0;
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  v.a = v.cnt > 0 ? __ldcg(reinterpret_cast<const float4 *>(src)) : z;
  v.b = v.cnt > 1 ? __ldcg(reinterpret_cast<const float4 *>(src + stride)) : z;
}

__device__ __forceinline__ float4 vec4_finish(const GemmOut &g, int n, int col, const Vec4Load &v) {
  float4 acc = v.a;
  if (v.cnt > 1) acc = add4(acc, v.b);
  if (v.cnt > 2) {
    unsigned t;
    const float *src = vec4_src(g, n, col, &t);
    const size_t stride = static_cast<size_t>(g.ntile) * 128;
    for (int j = 2; j < v.cnt; ++j)
      acc = add4(acc, __ldcg(reinterpret_cast<const float4 *>(src + j * stride)));
  }
  return acc;
}

// The same with only the first partial's load in flight (fewer registers:
// for the K/V GEMM at prefill sizes a second partial is the exception).
struct Vec4Load1 {
  float4 a;
  int cnt;
};

__device__ __forceinline__ void vec4_issue1(const GemmOut &g, int n, int col, bool on, Vec4Load1 &v) {
  unsigned t;
  const float *src = vec4_src(g, n, col, &t);
  v.cnt = on ? gemm_tile_parts(g, t) : 0;
  v.a = v.cnt > 0 ? __ldcg(reinterpret_cast<const float4 *>(src)) : make_float4(0.f, 0.f, 0.f, 0.f);
}

__device__ __forceinline__ float4 vec4_finish1(const GemmOut &g, int n, int col, const Vec4Load1 &v) {
  float4 acc = v.a;
  if (v.cnt > 1) {
    unsigned t;
    const float *src = vec4_src(g, n, col, &t);
    const size_t stride = static_cast<size_t>(g.ntile) * 128;
    for (int j = 1; j < v.cnt; ++j)
      acc = add4(acc, __ldcg(reinterpret_cast<const float4 *>(src + j * stride)));
  }
  return acc;
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
  return static_cast<uint32_t>(f32_to_bf16_rn(lo)) | (static_cast<uint32_t>(f32_to_bf16_rn(hi)) << 16);
}


// Row set-up of the many-row epilogue, the first launch of the chain: one
// warp per GEMM row resolves the row's destination (request by binary search
// of cu_rows, write rule, page lookup) and stores the row's RoPE cos/sin for
// every rotate-half pair (the angle formed in double precision, once per row
// instead of once per head and layer).  It reads only the call's index
// inputs, so the fc GEMM streams its weights meanwhile.
__global__ void __launch_bounds__(256) row_setup_kernel(const RowDest rd, const RopeFreqs rf,
                                                        int N) {
  griddep_launch();
  griddep_wait();
  const int n = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (n >= N) return;  // warp-uniform
  row_setup_warp(rd, rf, n, threadIdx.x & 31);
}

// hn = bf16(bf16(Y1 row) * gamma_h / rms), one CTA of D/32 threads per row:
// thread t holds the 8-column groups t + k*D/32, k < 4, two float4 loads per
// partial.  CTA 0 snapshots ctx_len.
constexpr int kWideNormGroups = 4;

__global__ void __launch_bounds__(256) hidden_norm_wide_kernel(
    const GemmOut y, const uint16_t *gamma, uint16_t *hn, int D, float eps,
    const int32_t *ctx_len, int32_t *ctx_snap, int B) {
  __shared__ float red[32];
  griddep_launch();
  griddep_wait();
  const int n = blockIdx.x, tid = threadIdx.x;
  const int T = D >> 5;
  const bool act = tid < T;
  if (n == 0)
    for (int r = tid; r < B; r += blockDim.x) ctx_snap[r] = ctx_len[r];
  Vec4Load ld[kWideNormGroups][2];
#pragma unroll
  for (int k = 0; k < kWideNormGroups; ++k) {
    const int col = 8 * (tid + k * T);
    vec4_issue(y, n, col, act, ld[k][0]);
    vec4_issue(y, n, col + 4, act, ld[k][1]);
  }
  float h[kWideNormGroups][8];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < kWideNormGroups; ++k) {
    const int col = 8 * (tid + k * T);
    const float4 u0 = vec4_finish(y, n, col, ld[k][0]), u1 = vec4_finish(y, n, col + 4, ld[k][1]);
    const float v[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      h[k][e] = bf16_to_f32(f32_to_bf16_rn(v[e]));
      ss += h[k][e] * h[k][e];
    }
  }
  const float tot = block_sum(ss, red);
  const float inv = rsqrtf(tot / static_cast<float>(D) + eps);
  if (!act) return;
  const bool g16 = (reinterpret_cast<uintptr_t>(gamma) & 15u) == 0;
#pragma unroll
  for (int k = 0; k < kWideNormGroups; ++k) {
    const int col = 8 * (tid + k * T);
    uint16_t gb[8];
    if (g16) {
      const uint4 q = *reinterpret_cast<const uint4 *>(gamma + col);
      const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        gb[2 * e] = static_cast<uint16_t>(wv[e] & 0xffffu);
        gb[2 * e + 1] = static_cast<uint16_t>(wv[e] >> 16);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) gb[e] = gamma[col + e];
    }
    float o[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = h[k][e] * inv * bf16_to_f32(gb[e]);
    uint4 q;
    q.x = pack2_bf16(o[0], o[1]);
    q.y = pack2_bf16(o[2], o[3]);
    q.z = pack2_bf16(o[4], o[5]);
    q.w = pack2_bf16(o[6], o[7]);
    *reinterpret_cast<uint4 *>(hn + static_cast<size_t>(n) * D + col) = q;
  }
}

// GQA epilogue for many rows: a unit is one KV head of one layer of one row,
// K and V, handled by hd/8 lanes; lane j holds columns 4j..4j+3 and
// hd/2 + 4j..+3 of K and of V (four rotate-half pairs of K, whose cos/sin the
// norm stored per row) and issues all four 16-byte loads before it adds any.
// 256 threads = 256 / (hd/8) units per CTA.  The k RMSNorm is a shuffle sum
// over the unit's lanes; each row leaves as two 8-byte stores per lane.
// Needs hd / 8 a power of two <= 32.
__global__ void __launch_bounds__(256, 4) epilogue_gqa_wide_kernel(
    const GemmOut y, const MaskArgs m, const int4 *dst, const float2 *cs,
    const uint16_t *gamma_k, uint16_t *pool, int N, int L, int nkv, int hd, float eps,
    int32_t *ctx_len, int B) {
  griddep_launch();
  griddep_wait();
  if (blockIdx.x == 0) advance_ctx_len(m, ctx_len, B);
  const int lpu = hd >> 3, half = hd >> 1;
  const int H = L * nkv;
  const long long u = static_cast<long long>(blockIdx.x) * (blockDim.x / lpu) + threadIdx.x / lpu;
  const int j = threadIdx.x % lpu;
  if (u >= static_cast<long long>(N) * H) return;  // whole units leave together
  const int n = static_cast<int>(u / H), lh = static_cast<int>(u % H);
  const int l = lh / nkv, h = lh % nkv;
  const int ck = ((l * 2) * nkv + h) * hd + 4 * j, cv = ck + nkv * hd;
  Vec4Load1 kl, kh, vl, vh;
  vec4_issue1(y, n, ck, true, kl);
  vec4_issue1(y, n, ck + half, true, kh);
  vec4_issue1(y, n, cv, true, vl);
  vec4_issue1(y, n, cv + half, true, vh);
  const int4 d = dst[n];
  // cos/sin of pairs 4j..4j+3 (16-byte aligned: hd/2 is a multiple of 4)
  const float4 *t = reinterpret_cast<const float4 *>(cs + static_cast<size_t>(n) * half + 4 * j);
  const float4 c01 = t[0], c23 = t[1];
  const float4 a = vec4_finish1(y, n, ck, kl), b = vec4_finish1(y, n, ck + half, kh);
  const float4 va4 = vec4_finish1(y, n, cv, vl), vb4 = vec4_finish1(y, n, cv + half, vh);
  if (d.x < 0) return;
  const unsigned mask = (lpu == 32 ? 0xffffffffu : ((1u << lpu) - 1u))
                        << ((threadIdx.x & 31) & ~(lpu - 1));
  float ss = a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w + b.x * b.x + b.y * b.y + b.z * b.z +
             b.w * b.w;
  for (int o = lpu >> 1; o > 0; o >>= 1) ss += __shfl_xor_sync(mask, ss, o);
  const float inv = rsqrtf(ss / static_cast<float>(hd) + eps);
  const uint16_t *gk = gamma_k + static_cast<size_t>(l) * hd;
  float ka[4] = {a.x, a.y, a.z, a.w}, kb[4] = {b.x, b.y, b.z, b.w};
  const float cv4[4] = {c01.x, c01.z, c23.x, c23.z}, sv4[4] = {c01.y, c01.w, c23.y, c23.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int c = 4 * j + e;
    const float k0 = ka[e] * inv * bf16_to_f32(gk[c]);
    const float k1 = kb[e] * inv * bf16_to_f32(gk[c + half]);
    ka[e] = k0 * cv4[e] - k1 * sv4[e];
    kb[e] = k1 * cv4[e] + k0 * sv4[e];
  }
  const size_t plane = static_cast<size_t>(nkv) * m.P * hd;  // K -> V of the same page
  uint16_t *krow =
      pool + ((((static_cast<size_t>(l) * m.NP + d.x) * 2) * nkv + h) * m.P + d.y) * hd;
  uint16_t *vrow = krow + plane;
  *reinterpret_cast<uint2 *>(krow + 4 * j) = make_uint2(pack2_bf16(ka[0], ka[1]), pack2_bf16(ka[2], ka[3]));
  *reinterpret_cast<uint2 *>(krow + half + 4 * j) =
      make_uint2(pack2_bf16(kb[0], kb[1]), pack2_bf16(kb[2], kb[3]));
  *reinterpret_cast<uint2 *>(vrow + 4 * j) =
      make_uint2(pack2_bf16(va4.x, va4.y), pack2_bf16(va4.z, va4.w));
  *reinterpret_cast<uint2 *>(vrow + half + 4 * j) =
      make_uint2(pack2_bf16(vb4.x, vb4.y), pack2_bf16(vb4.z, vb4.w));
}

// MLA epilogue for many rows: one warp per (row, layer).  Lane l holds the
// latent groups g = l + 32k (columns 4g..4g+3 and lat/2 + 4g..+3, k < G) and,
// for l < rope/8, the rope group l (rope columns 4l..+3 and rope/2 + 4l..+3):
// rotate-half pairs again.  All loads go out first; the latent RMSNorm is a
// warp sum; every group leaves as two 8-byte stores.  Needs lat % 8 == rope %
// 8 == 0 and lat <= 256 G.
template <int G>
__global__ void __launch_bounds__(256) epilogue_mla_wide_kernel(
    const GemmOut y, const MaskArgs m, const int4 *dst, const float2 *cs,
    const uint16_t *gamma_kv, uint16_t *pool, int N, int L, int lat, int rope, float eps,
    int32_t *ctx_len, int B) {
  griddep_launch();
  griddep_wait();
  if (blockIdx.x == 0) advance_ctx_len(m, ctx_len, B);
  const long long u = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (u >= static_cast<long long>(N) * L) return;  // warp-uniform
  const int n = static_cast<int>(u / L), l = static_cast<int>(u % L);
  const int W = lat + rope, hl = lat >> 1, hr = rope >> 1;
  const int base = l * W;
  Vec4Load1 la[G], lb[G], ra, rb;
#pragma unroll
  for (int k = 0; k < G; ++k) {
    const int g = lane + 32 * k;
    const bool on = g < (lat >> 3);
    vec4_issue1(y, n, base + (on ? 4 * g : 0), on, la[k]);
    vec4_issue1(y, n, base + (on ? hl + 4 * g : 0), on, lb[k]);
  }
  const bool ron = lane < (rope >> 3);
  vec4_issue1(y, n, base + (ron ? lat + 4 * lane : 0), ron, ra);
  vec4_issue1(y, n, base + (ron ? lat + hr + 4 * lane : 0), ron, rb);
  const int4 d = dst[n];
  float4 c01 = make_float4(0.f, 0.f, 0.f, 0.f), c23 = c01;
  if (ron) {  // cos/sin of rope pairs 4*lane..+3 (16-byte aligned: rope/2 is a multiple of 4)
    const float4 *t = reinterpret_cast<const float4 *>(cs + static_cast<size_t>(n) * hr + 4 * lane);
    c01 = t[0];
    c23 = t[1];
  }
  float4 a[G], b[G];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < G; ++k) {
    const int g = lane + 32 * k;
    const bool on = g < (lat >> 3);
    a[k] = vec4_finish1(y, n, base + (on ? 4 * g : 0), la[k]);
    b[k] = vec4_finish1(y, n, base + (on ? hl + 4 * g : 0), lb[k]);
    ss += a[k].x * a[k].x + a[k].y * a[k].y + a[k].z * a[k].z + a[k].w * a[k].w + b[k].x * b[k].x +
          b[k].y * b[k].y + b[k].z * b[k].z + b[k].w * b[k].w;
  }
  float4 ro = vec4_finish1(y, n, base + (ron ? lat + 4 * lane : 0), ra);
  float4 rh = vec4_finish1(y, n, base + (ron ? lat + hr + 4 * lane : 0), rb);
  ss = warp_sum(ss);
  if (d.x < 0) return;  // warp-uniform
  uint16_t *row = pool + ((static_cast<size_t>(l) * m.NP + d.x) * m.P + d.y) * W;
  const float inv = rsqrtf(ss / static_cast<float>(lat) + eps);
  const uint16_t *gk = gamma_kv + static_cast<size_t>(l) * lat;
#pragma unroll
  for (int k = 0; k < G; ++k) {
    const int g = lane + 32 * k;
    if (g < (lat >> 3)) {
      const int c0 = 4 * g, c1 = hl + 4 * g;
      const float4 x = a[k], z = b[k];
      *reinterpret_cast<uint2 *>(row + c0) =
          make_uint2(pack2_bf16(x.x * inv * bf16_to_f32(gk[c0]), x.y * inv * bf16_to_f32(gk[c0 + 1])),
                     pack2_bf16(x.z * inv * bf16_to_f32(gk[c0 + 2]), x.w * inv * bf16_to_f32(gk[c0 + 3])));
      *reinterpret_cast<uint2 *>(row + c1) =
          make_uint2(pack2_bf16(z.x * inv * bf16_to_f32(gk[c1]), z.y * inv * bf16_to_f32(gk[c1 + 1])),
                     pack2_bf16(z.z * inv * bf16_to_f32(gk[c1 + 2]), z.w * inv * bf16_to_f32(gk[c1 + 3])));
    }
  }
  if (ron) {
    float va[4] = {ro.x, ro.y, ro.z, ro.w}, vb[4] = {rh.x, rh.y, rh.z, rh.w};
    const float cv[4] = {c01.x, c01.z, c23.x, c23.z}, sv[4] = {c01.y, c01.w, c23.y, c23.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float x0 = va[e], x1 = vb[e];
      va[e] = x0 * cv[e] - x1 * sv[e];
      vb[e] = x1 * cv[e] + x0 * sv[e];
    }
    *reinterpret_cast<uint2 *>(row + lat + 4 * lane) =
        make_uint2(pack2_bf16(va[0], va[1]), pack2_bf16(va[2], va[3]));
    *reinterpret_cast<uint2 *>(row + lat + hr + 4 * lane) =
        make_uint2(pack2_bf16(vb[0], vb[1]), pack2_bf16(vb[2], vb[3]));
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
                                    int L, int nkv, int hd, float eps, int32_t *ctx_len, int B,
                                    const int4 *dst, const float2 *cs) {
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
  const int l = head / (2 * nkv);
  const int kv = (head / nkv) & 1;
  const int h = head % nkv;
  // a set-up row's destination and cos/sin go out with the Y2 loads
  int4 d = make_int4(-1, 0, 0, 0);
  float2 csv = make_float2(1.f, 0.f);
  if (!kStaged && dst) {
    d = dst[n];
    if (kv == 0 && act) csv = cs[static_cast<size_t>(n) * (hd >> 1) + t];
  }
  // ctx_len advance; every reader of the pre-step value uses the snapshot
  if (!kStaged && n == 0 && head == 0) advance_ctx_len(m, ctx_len, B);
  int r, i;
  if (!row_of(m, n, &r, &i)) return;
  int page = 0, slot = 0, pos;
  if (kStaged) {
    pos = m.ctx_snap[r] + i;
  } else if (dst) {
    if (d.x < 0) return;
    page = d.x;
    slot = d.y;
    pos = d.z;
  } else if (!ctx_row_dest(m, r, i, &page, &slot, &pos, head == 0 && t == 0)) {
    return;
  }
  float v0 = gemm_out_finish(y, ld0), v1 = gemm_out_finish(y, ld1);
  if (kv == 0) {
    const float ss = block_sum(act ? v0 * v0 + v1 * v1 : 0.f, red);
    const float inv = rsqrtf(ss / static_cast<float>(hd) + eps);
    if (act) {
      const float k0 = v0 * inv * bf16_to_f32(gamma_k[static_cast<size_t>(l) * hd + t]);
      const float k1 = v1 * inv * bf16_to_f32(gamma_k[static_cast<size_t>(l) * hd + t + half]);
      float c, s;
      if (!kStaged && dst) {
        c = csv.x;
        s = csv.y;
      } else {
        rope_cos_sin(pos, rf.f[t], &c, &s);
      }
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

// The same epilogue with kEpiHeads heads of one row per CTA (grid (N rows,
// L*2*nkv / kEpiHeads)): a quarter of the CTAs, each head's k-norm sum over
// its own warps (one barrier for all heads), when the head count divides.
constexpr int kEpiHeads = 4;
template <bool kStaged>
__global__ void epilogue_gqa_heads_kernel(const GemmOut y, const MaskArgs m, const RopeFreqs rf,
                                          const uint16_t *gamma_k, uint16_t *pool,
                                          uint16_t *staged, int L, int nkv, int hd, float eps,
                                          int32_t *ctx_len, int B, const int4 *dst,
                                          const float2 *cs) {
  __shared__ float red[kEpiHeads][4];
  __shared__ __align__(16) uint16_t obuf[kEpiHeads][kMaxHeadDim];
  griddep_launch();
  griddep_wait();
  const int n = blockIdx.x;
  const int tph = blockDim.x / kEpiHeads;  // threads per head: a multiple of 32
  const int hs = threadIdx.x / tph, t = threadIdx.x % tph;
  const int head = blockIdx.y * kEpiHeads + hs;  // ((l * 2 + kv) * nkv + h)
  const int half = hd >> 1;
  const bool act = t < half;
  GemmOutLoad ld0, ld1;
  {
    const int c0 = head * hd + (act ? t : 0), c1 = c0 + half;
    const int nt = n / y.ntile, nr = n - nt * y.ntile;
    const unsigned t0 = static_cast<unsigned>(nt) * y.mtiles + (c0 >> 7);
    const unsigned t1 = static_cast<unsigned>(nt) * y.mtiles + (c1 >> 7);
    gemm_out_issue(y, t0, act ? gemm_tile_parts(y, t0) : 0, nr, c0 & 127, ld0);
    gemm_out_issue(y, t1, act ? gemm_tile_parts(y, t1) : 0, nr, c1 & 127, ld1);
  }
  const int l = head / (2 * nkv);
  const int kv = (head / nkv) & 1;
  const int h = head % nkv;
  int4 d = make_int4(-1, 0, 0, 0);
  float2 csv = make_float2(1.f, 0.f);
  if (!kStaged && dst) {
    d = dst[n];
    if (kv == 0 && act) csv = cs[static_cast<size_t>(n) * half + t];
  }
  if (!kStaged && n == 0 && blockIdx.y == 0) advance_ctx_len(m, ctx_len, B);
  int r, i;
  if (!row_of(m, n, &r, &i)) return;  // the whole CTA: one row
  int page = 0, slot = 0, pos;
  if (kStaged) {
    pos = m.ctx_snap[r] + i;
  } else if (dst) {
    if (d.x < 0) return;
    page = d.x;
    slot = d.y;
    pos = d.z;
  } else if (!ctx_row_dest(m, r, i, &page, &slot, &pos, blockIdx.y == 0 && threadIdx.x == 0)) {
    return;
  }
  float v0 = gemm_out_finish(y, ld0), v1 = gemm_out_finish(y, ld1);
  const float part = warp_sum((kv == 0 && act) ? v0 * v0 + v1 * v1 : 0.f);
  if ((t & 31) == 0) red[hs][t >> 5] = part;
  __syncthreads();
  if (kv == 0 && act) {
    float ss = 0.f;
    for (int w = 0; w < (tph >> 5); ++w) ss += red[hs][w];
    const float inv = rsqrtf(ss / static_cast<float>(hd) + eps);
    const float k0 = v0 * inv * bf16_to_f32(gamma_k[static_cast<size_t>(l) * hd + t]);
    const float k1 = v1 * inv * bf16_to_f32(gamma_k[static_cast<size_t>(l) * hd + t + half]);
    float c, sn;
    if (!kStaged && dst) {
      c = csv.x;
      sn = csv.y;
    } else {
      rope_cos_sin(pos, rf.f[t], &c, &sn);
    }
    v0 = k0 * c - k1 * sn;
    v1 = k1 * c + k0 * sn;
  }
  if (act) {
    obuf[hs][t] = f32_to_bf16_rn(v0);
    obuf[hs][t + half] = f32_to_bf16_rn(v1);
  }
  __syncthreads();
  if (t < hd / 8) {  // head_dim % 8 == 0: the row leaves as 16-byte vectors
    uint16_t *row =
        kStaged ? staged + static_cast<size_t>(n) * L * 2 * nkv * hd + head * hd
                : pool + ((((static_cast<size_t>(l) * m.NP + page) * 2 + kv) * nkv + h) * m.P +
                          slot) * hd;
    reinterpret_cast<uint4 *>(row)[t] = reinterpret_cast<const uint4 *>(obuf[hs])[t];
  }
}

// ------------------------------------------------------ MLA epilogue
// grid (N rows, L), block = lat / 2 + rope / 2 threads rounded up to a warp:
// thread t < lat/2 holds latent columns t and t + lat/2; thread lat/2 + j
// holds the rope pair j, j + rope/2.  kStaged as for GQA.
template <bool kStaged>
__global__ void epilogue_mla_kernel(const GemmOut y, const MaskArgs m, const RopeFreqs rf,
                                    const uint16_t *gamma_kv, uint16_t *pool, uint16_t *staged,
                                    int L, int lat, int rope, float eps, int32_t *ctx_len, int B,
                                    const int4 *dst, const float2 *cs) {
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
  // a set-up row's destination and cos/sin go out with the Y2 loads
  int4 d = make_int4(-1, 0, 0, 0);
  float2 csv = make_float2(1.f, 0.f);
  if (!kStaged && dst) {
    d = dst[n];
    if (is_rope) csv = cs[static_cast<size_t>(n) * hr + (t - hl)];
  }
  if (!kStaged && n == 0 && l == 0) advance_ctx_len(m, ctx_len, B);
  int r, i;
  if (!row_of(m, n, &r, &i)) return;
  int page = 0, slot = 0, pos;
  if (kStaged) {
    pos = m.ctx_snap[r] + i;
  } else if (dst) {
    if (d.x < 0) return;
    page = d.x;
    slot = d.y;
    pos = d.z;
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
    if (!kStaged && dst) {
      c = csv.x;
      s = csv.y;
    } else {
      rope_cos_sin(pos, rf.f[t - hl], &c, &s);
    }
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

// The launch chain [row set-up] -> [prep] -> fc GEMM -> hidden norm -> K/V GEMM
// -> epilogue (the row set-up for the many-row epilogue, the prep for fp32
// hidden rows).
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

  // epilogue arguments (the row set-up resolves row destinations with them)
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
  const bool gqa = g.kind == DFLASH_KIND_GQA;
  const int lpu = g.head_dim / 8;
  const bool wide = d.N > kClusterNormMaxRows;
  const bool wide_epi = wide && !split &&
                        (gqa ? (lpu >= 1 && lpu <= 32 && (lpu & (lpu - 1)) == 0 && g.head_dim % 8 == 0)
                             : (g.latent_dim % 8 == 0 && g.rope_dim % 8 == 0));
  RowDest rd;
  rd.dst = wide_epi ? W.dst : nullptr;
  rd.cs = W.cs;
  rd.nf = d.nf;
  rd.m = m;
  rd.m.ctx_snap = ctx_len;
  RopeFreqs rf;
  fill_rope_freqs(&rf, gqa ? g.head_dim : g.rope_dim, g.rope_theta);

  // row set-up of the many-row epilogue (destinations, RoPE cos/sin)
  if (wide_epi) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3((d.N + 7) / 8);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((e = cudaLaunchKernelEx(&cfg, row_setup_kernel, rd, rf, d.N)) != cudaSuccess) return e;
  }

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

  // fc GEMM + hidden RMSNorm.  Up to 64 rows: the fc GEMM as clusters that
  // finish h = bf16(Y1) and its per-slice sums of squares themselves, then a
  // plain elementwise norm.
  GemmOut y1, y2;
  const bool fc_cl = !wide && aligned16(w.gamma_h) && fc_cluster_ok(d.N, d.D_in, d.D);
  // the fused update's row set-up (destination, RoPE cos/sin) runs in idle
  // warps of the cluster fc GEMM; the epilogue then reads it
  const bool fc_setup = fc_cl && !split;
  if (fc_cl) {
    RowDest frd = rd;
    frd.dst = W.dst;
    if ((e = launch_fc_cluster(X, d.N, d.D_in, static_cast<const uint16_t *>(w.w_fc), d.D, W.h,
                               W.ssq, st, s, fc_setup ? &frd : nullptr,
                               fc_setup ? &rf : nullptr)) != cudaSuccess)
      return e;
  } else if ((e = launch_gemm(X, d.N, d.D_in, static_cast<const uint16_t *>(w.w_fc), d.D,
                              W.part1, st, /*pdl=*/true, s, &y1)) != cudaSuccess) {
    return e;
  }

  // hidden RMSNorm: after the cluster fc GEMM a plain elementwise kernel;
  // otherwise a cluster of G CTAs per row for decode-sized row counts, one
  // CTA per row beyond
  if (fc_cl) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3((d.D + 511) / 512, d.N);
    cfg.blockDim = dim3(64);
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((e = cudaLaunchKernelEx(&cfg, hidden_norm_h_kernel, static_cast<const uint16_t *>(W.h),
                                static_cast<const float *>(W.ssq), d.D / 32, fc_cluster_rows(d.N),
                                static_cast<const uint16_t *>(w.gamma_h), W.hn, d.D,
                                static_cast<float>(g.eps_hidden),
                                static_cast<const int32_t *>(ctx_len), snap, B)) != cudaSuccess)
      return e;
  } else if (wide) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(d.N);
    cfg.blockDim = dim3((d.D / 32 + 31) / 32 * 32);
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (d.D % 64 != 0 || d.D > 8192) return cudaErrorInvalidValue;
    if ((e = cudaLaunchKernelEx(&cfg, hidden_norm_wide_kernel, y1,
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
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.stream = s;
  uint16_t *pool16 = static_cast<uint16_t *>(pool);
  if (wide_epi && gqa) {
    const long long units = static_cast<long long>(d.N) * g.num_layers * g.nkv;
    const int upc = 256 / lpu;
    cfg.gridDim = dim3(static_cast<unsigned>((units + upc - 1) / upc));
    cfg.blockDim = dim3(256);
    e = cudaLaunchKernelEx(&cfg, epilogue_gqa_wide_kernel, y2, m,
                           static_cast<const int4 *>(W.dst), static_cast<const float2 *>(W.cs),
                           static_cast<const uint16_t *>(w.gamma_k), pool16, d.N, g.num_layers,
                           g.nkv, g.head_dim, static_cast<float>(g.eps_k), ctx_len, B);
  } else if (wide_epi) {
    const long long units = static_cast<long long>(d.N) * g.num_layers;
    cfg.gridDim = dim3(static_cast<unsigned>((units + 7) / 8));
    cfg.blockDim = dim3(256);
    auto kern = g.latent_dim <= 256   ? epilogue_mla_wide_kernel<1>
                : g.latent_dim <= 512 ? epilogue_mla_wide_kernel<2>
                : g.latent_dim <= 768 ? epilogue_mla_wide_kernel<3>
                                      : epilogue_mla_wide_kernel<4>;
    e = cudaLaunchKernelEx(&cfg, kern, y2, m, static_cast<const int4 *>(W.dst),
                           static_cast<const float2 *>(W.cs),
                           static_cast<const uint16_t *>(w.gamma_k), pool16, d.N, g.num_layers,
                           g.latent_dim, g.rope_dim, static_cast<float>(g.eps_k), ctx_len, B);
  } else if (gqa && (g.num_layers * 2 * g.nkv) % kEpiHeads == 0 && g.head_dim <= 128) {
    fill_rope_freqs(&rf, g.head_dim, g.rope_theta);
    cfg.gridDim = dim3(d.N, g.num_layers * 2 * g.nkv / kEpiHeads);
    cfg.blockDim = dim3(kEpiHeads * std::max(32, (g.head_dim / 2 + 31) / 32 * 32));
    e = cudaLaunchKernelEx(&cfg,
                           split ? epilogue_gqa_heads_kernel<true> : epilogue_gqa_heads_kernel<false>,
                           y2, m, rf, static_cast<const uint16_t *>(w.gamma_k), pool16, staged,
                           g.num_layers, g.nkv, g.head_dim, static_cast<float>(g.eps_k), ctx_len, B,
                           static_cast<const int4 *>(fc_setup ? W.dst : nullptr),
                           static_cast<const float2 *>(fc_setup ? W.cs : nullptr));
  } else if (gqa) {
    fill_rope_freqs(&rf, g.head_dim, g.rope_theta);
    cfg.gridDim = dim3(d.N, g.num_layers * 2 * g.nkv);
    cfg.blockDim = dim3(std::max(32, (g.head_dim / 2 + 31) / 32 * 32));
    e = cudaLaunchKernelEx(&cfg, split ? epilogue_gqa_kernel<true> : epilogue_gqa_kernel<false>, y2,
                           m, rf, static_cast<const uint16_t *>(w.gamma_k), pool16, staged,
                           g.num_layers, g.nkv, g.head_dim, static_cast<float>(g.eps_k), ctx_len, B,
                           static_cast<const int4 *>(fc_setup ? W.dst : nullptr),
                           static_cast<const float2 *>(fc_setup ? W.cs : nullptr));
  } else {
    fill_rope_freqs(&rf, g.rope_dim, g.rope_theta);
    cfg.gridDim = dim3(d.N, g.num_layers);
    cfg.blockDim = dim3((g.latent_dim / 2 + g.rope_dim / 2 + 31) / 32 * 32);
    e = cudaLaunchKernelEx(&cfg, split ? epilogue_mla_kernel<true> : epilogue_mla_kernel<false>, y2,
                           m, rf, static_cast<const uint16_t *>(w.gamma_k), pool16, staged,
                           g.num_layers, g.latent_dim, g.rope_dim, static_cast<float>(g.eps_k),
                           ctx_len, B, static_cast<const int4 *>(fc_setup ? W.dst : nullptr),
                           static_cast<const float2 *>(fc_setup ? W.cs : nullptr));
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
