// attention_tc.cu -- split-KV block attention (GQA) on the 5th-generation
// tensor cores.
//
// Follows vLLM PR #54092 (Purpose item 2, Changes item 2): small uniform query
// blocks (1 bonus + N drafts) run split over KV segments with per-query-token
// partial softmax state and a separate reduce; with a sliding window the
// segments divide only the keys the window can see; sinks join the reduce.
//
// One CTA = (segment s, row tile rt) x KV head x request.  Its 128 MMA rows
// are the query rows (token i, head h) of the KV head's group (G = hq / nkv
// heads x Tq tokens; rows past G*Tq are zero padding).  Per 128-key tile:
//   TMA   K and V pages of the tile -> shared memory ring (`nst` stages)
//   MMA   S = Q K^T     (M=128, N=128, K=hd; Q from TMEM) -> TMEM S (2 buffers)
//   softmax warps: mask, online max with lazy rescale (the reference max only
//         moves when the tile max exceeds it by 2^8, so O in TMEM is rarely
//         rescaled), P = exp2(s - m) -> bf16 -> TMEM
//   MMA   O += P V      (M=128, N=hd, K=128; P from TMEM) -> TMEM O
// and at the end each real row writes (m, l, O) of its segment to the
// workspace for the merge kernel.  Both MMAs take their A operand (Q, P) from
// tensor memory: with A in shared memory the tensor pipe spends most of its
// time re-reading Q, and keeping P out of shared memory also drops a store, a
// proxy fence and 32 KB of shared memory per tile.  The single issuing thread
// is the critical resource here (each tcgen05.mma takes ~70 cycles to issue
// whatever its N, and every commit and barrier wait adds to the same serial
// stream), so tiles are 128 keys wide: per key that halves the QK
// instructions and the waits and commits of a 64-key tile.
//
// Roles (8 warps): warp 2 issues TMA (and, when the call fuses the block
// scatter, first writes the block's own K/V rows of its key range into the
// cache), warp 3 issues QK and owns the TMEM allocation, lane 0 of warp 0
// issues PV, warps 4-7 run the softmax (warp w reads and writes TMEM lanes
// 32*(w%4)..+31, i.e. runs on SM sub-partition w%4), warp 1 only joins the
// final barrier.  When the group has at most 64 query rows (the decode
// case: a 16-token block times a few heads per KV head), those rows are
// loaded twice, as MMA rows r and r + 64: the tensor core then hands all four
// sub-partitions a copy of the scores and each softmax warp takes half of a
// row's 128 key columns, so the exp2 work spreads over all four SFU pipes
// instead of two.  Row r's P then carries its first 64 keys (zeros after) and
// row r + 64's its last 64 (zeros before), so O rows r and r + 64 hold the two
// halves of the row's sum, added in the epilogue.
//
// Every wait is an mbarrier try_wait, which suspends the thread in hardware
// rather than polling shared memory, and is bounded: a timeout raises
// DFLASH_DEV_WAIT_TIMEOUT and the CTA winds down.
#include <cuda.h>

#include <algorithm>

#include "attention_common.cuh"

namespace dflash {

cudaError_t make_tmap_bf16_2d(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols,
                              uint64_t row_stride_elems, uint32_t box_rows, uint32_t box_cols);

namespace {

constexpr int kKT = kAttnTileKeys;  // 128 keys per tile
static_assert(kKT == 128, "TMEM column plan below assumes 128-key tiles");
constexpr int kRows = 128;
constexpr int kThreadsTC = 256;
constexpr int kSmemMax = 227 * 1024;  // dynamic shared memory per CTA
// V is the MMA's B operand stored N(=dim)-contiguous: 128-byte swizzled rows of
// 64 dims, one row per key; next 64-dim chunk at kVChunk bytes, next 8 keys at
// 1024 bytes.
constexpr uint32_t kVChunk = kKT * 128;
// Tensor memory columns (all 512 allocated; head_dim <= 128):
constexpr uint32_t kColS = 0;    // two 128-column fp32 S buffers
constexpr uint32_t kColO = 256;  // O accumulator, head_dim fp32 columns
constexpr uint32_t kColQ = 384;  // Q, head_dim / 2 columns of bf16 pairs
constexpr uint32_t kColP = 448;  // P, 64 columns of bf16 pairs (128 keys)
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxAttnHeadDim = 128;

struct TcParams {
  AttnParams a;
  int GT, RT, box_rows, nst, chunks, split;
  int skip_tile;  // tests only: the producer never issues this tile (-1: off)
  uint32_t stage_bytes, k_bytes, bar_off, x_off;
  uint32_t idesc_qk, idesc_pv, v_lbo, v_sbo;
  float scale_log2;
};

// kSplit: the split layout (a KV head's query rows fit in 64); each
// instantiation carries only its own softmax.  kScatter: the call fuses the
// layer's block scatter (a separate instantiation: any scatter code inside
// the plain kernel, even never run, slowed it by ~10%).
template <bool kSplit, bool kScatter>
__global__ void __launch_bounds__(kThreadsTC, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm, const __grid_constant__ TcParams P) {
  const AttnParams &p = P.a;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  uint8_t *sKV = sm;
  const int nst = P.nst;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + P.bar_off);
  uint64_t *kv_full = bars, *kv_empty = bars + nst, *s_full = bars + 2 * nst;
  uint64_t *p_full = s_full + 2, *o_done = p_full + 1, *drain = o_done + 1, *q_full = drain + 1;
  uint64_t *s_free = q_full + 1, *drain_pv = s_free + 2;
  uint32_t *tslot = reinterpret_cast<uint32_t *>(drain_pv + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tslot + 1);
  volatile int *consumed = reinterpret_cast<volatile int *>(tslot + 2);

  const int s = blockIdx.x / P.RT, rt = blockIdx.x % P.RT;
  const int kvh = blockIdx.y, r = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < nst; ++i) {
      ptx::mbar_init(ptx::smem_u32(&kv_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&kv_empty[i]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&s_full[0]), 1);
    ptx::mbar_init(ptx::smem_u32(&s_full[1]), 1);
    // one arrival per softmax warp at work: all four in the split layout,
    // else those owning at least one real row
    const int real_rows = min(kRows, P.GT - static_cast<int>(blockIdx.x % P.RT) * kRows);
    const uint32_t sm_warps = kSplit ? 4u : static_cast<uint32_t>((real_rows + 31) / 32);
    ptx::mbar_init(ptx::smem_u32(p_full), sm_warps);
    ptx::mbar_init(ptx::smem_u32(&s_free[0]), sm_warps);
    ptx::mbar_init(ptx::smem_u32(&s_free[1]), sm_warps);
    ptx::mbar_init(ptx::smem_u32(o_done), 1);
    ptx::mbar_init(ptx::smem_u32(drain), 1);
    ptx::mbar_init(ptx::smem_u32(drain_pv), 1);
    ptx::mbar_init(ptx::smem_u32(q_full), 4u);  // one arrival per softmax warp
    *abort_flag = 0;
    *consumed = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tm);
  }
  if (warp == 3) {
    ptx::tmem_alloc(ptx::smem_u32(tslot), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tslot;
  griddep_launch();
  if (warp == 2) {
    // While the preceding grid finishes, pull this segment's first ring-full
    // of K/V into L2.  kv_len and the table may still be changing, so they
    // are read with relaxed loads and used for nothing but this hint: L2 is
    // the point of coherence, so a prefetched line never hides a later write
    // from the copies below, and a wrong guess only costs bandwidth.
    int kl = ptx::ld_relaxed_s32(p.kv_len + r);
    const long long cap = static_cast<long long>(p.M) * p.P;
    kl = kl < 0 ? 0 : (kl > cap ? static_cast<int>(cap) : kl);
    const SegRange g = segment_range_for(p, kl, s);
    const int boxes = kKT / P.box_rows;
    const int nbox = boxes * 2 * P.chunks;
    const int npre = min(g.t1 - g.t0, P.nst) * nbox;
    for (int j = lane; j < npre; j += 32) {
      const int tt = j / nbox, jb = j % nbox;
      const int b = jb / (2 * P.chunks), kv = (jb / P.chunks) & 1, c = jb % P.chunks;
      const int key0 = (g.t0 + tt) * kKT + b * P.box_rows;
      const int lp = key0 / p.P;
      if (lp < p.M && key0 < g.kv_len) {
        const int page = ptx::ld_relaxed_s32(p.tbl + static_cast<int64_t>(r) * p.M + lp);
        if (page >= 0 && page < p.NP) {
          const long long row0 =
              ((((static_cast<long long>(p.layer) * p.NP + page) * 2 + kv) * p.nkv + kvh) * p.P) +
              key0 % p.P;
          ptx::tma_prefetch_2d(&tm, c * 64, static_cast<int32_t>(row0));
        }
      }
    }
  }
  // Everything above overlaps the previous kernel's tail; inputs are read
  // only after it has completed.
  griddep_wait();
  const SegRange sr = segment_range(p, r, s);
  const int ntiles = sr.t1 - sr.t0;
  const uint32_t tm_s = tmem + kColS;
  const uint32_t tm_o = tmem + kColO;
  const uint32_t tm_q = tmem + kColQ;
  const uint32_t tm_p = tmem + kColP;

  // Q rows of this tile -> TMEM (softmax warp w fills its own lane quarter),
  // in parallel with the producer's first loads; the MMA issuer waits on
  // q_full.  In the split layout lanes 64-127 repeat rows 0-63, and each warp
  // zeroes the half of its P columns that it never writes.
  if (warp >= 4 && ntiles > 0) {
    const int q4 = warp & 3;
    const int row = kSplit ? 32 * (q4 & 1) + lane : 32 * q4 + lane;
    const int R = rt * kRows + row;
    const bool real = R < P.GT;
    const int i = real ? R / p.G : 0;
    const int h = kvh * p.G + (real ? R % p.G : 0);
    const uint4 *src = reinterpret_cast<const uint4 *>(
        p.q + ((static_cast<size_t>(r) * p.Tq + i) * p.hq + h) * p.dq);
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    uint4 v[kMaxAttnHeadDim / 8];
#pragma unroll
    for (int u = 0; u < kMaxAttnHeadDim / 8; ++u)
      v[u] = (real && u < p.dq / 8) ? src[u] : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int c = 0; c < kMaxAttnHeadDim / 32; ++c) {
      if (c < p.dq / 32) {
        uint32_t w16[16];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          w16[4 * u] = v[4 * c + u].x;
          w16[4 * u + 1] = v[4 * c + u].y;
          w16[4 * u + 2] = v[4 * c + u].z;
          w16[4 * u + 3] = v[4 * c + u].w;
        }
        ptx::tmem_st16(tm_q + lane_off + 16 * c, w16);
      }
    }
    if (kSplit) {
      uint32_t z[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) z[e] = 0u;
      const uint32_t zc = tm_p + lane_off + (q4 < 2 ? 32 : 0);
      ptx::tmem_st16(zc, z);
      ptx::tmem_st16(zc + 16, z);
    }
    ptx::tmem_wait_st();
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(q_full));
  }

  const int boxes = kKT / P.box_rows;

  if ((ntiles > 0 || kScatter) && warp == 2) {
    // ------------------------------------------------ TMA producer (warp 2)
    // Fused block scatter: the producer warp first writes the block rows of
    // this CTA's key range (their tiles are the segment's last, so only that
    // CTA's copies wait for it); the __syncwarp before the first copy orders
    // every lane's stores and proxy fence before it.  No warp barrier of its
    // own: one placed ahead of the role branches slowed the kernel by ~10%
    // even where it did nothing.
    if constexpr (kScatter)
      block_scatter_rows(block_scatter_args(p, sr), r, kvh, sr, s == 0 && rt == 0, lane);
    // The page ids of the segment are fetched warp-wide, one batch of 32
    // (tile, box) lookups ahead, so no table read sits between two TMA issues.
    const int tiles_per_batch = 32 / boxes;
    // With one row tile per segment every K/V line is read exactly once:
    // loading it evict-first keeps the stream from displacing what is reused
    // (measured: 5 x (scatter + attention) of the 32K Qwen3-8B-shaped step,
    // 197.6 -> 185.6 us).  Several row tiles re-read the segment, so they keep
    // the normal policy.
    const uint64_t pol = P.RT == 1 ? ptx::policy_evict_first() : ptx::policy_evict_normal();
    auto fetch_page = [&](int t_batch) -> int {
      const int tt = t_batch + lane / boxes, b = lane % boxes;
      int page = 0;
      if (tt < ntiles) {
        const int key0 = (sr.t0 + tt) * kKT + b * P.box_rows;
        const int lp = key0 / p.P;
        if (lp < p.M && key0 < sr.kv_len) {
          page = p.tbl[static_cast<int64_t>(r) * p.M + lp];
          if (page < 0 || page >= p.NP) {
            raise_status(p.st, DFLASH_DEV_BAD_PAGE);
            page = 0;
          }
        }
      }
      return page;
    };
    int cur = fetch_page(0);
    int nxt = fetch_page(tiles_per_batch);
    int issued = 0;
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int tb = t % tiles_per_batch;
      if (tb == 0 && t > 0) {
        cur = nxt;
        nxt = fetch_page(t + tiles_per_batch);
      }
      const int st = t % nst;
      bool got = true;
      if (lane == 0 && t >= nst)
        got = ptx::mbar_wait(ptx::smem_u32(&kv_empty[st]),
                             static_cast<uint32_t>(((t / nst) & 1) ^ 1), abort_flag);
      if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) {
        ok = false;
        break;
      }
      const bool skip = t == P.skip_tile;
      if (lane == 0 && !skip)
        ptx::mbar_arrive_expect_tx(ptx::smem_u32(&kv_full[st]), P.stage_bytes);
      __syncwarp();
      // The tile's boxes (page x K/V x 64-dim chunk) are issued by different
      // lanes: copies issued by one thread complete one after another, so
      // the number of issuing threads bounds the load rate of a CTA.
      const int kbase = (sr.t0 + t) * kKT;
      uint8_t *stage = sKV + st * P.stage_bytes;
      const int nbox = boxes * 2 * P.chunks;
      for (int j0 = 0; j0 < nbox; j0 += 32) {
        const int j = j0 + lane;
        const int b = (j < nbox) ? j / (2 * P.chunks) : 0;
        const int page = __shfl_sync(0xffffffffu, cur, tb * boxes + b);
        if (j < nbox && !skip) {
          const int kv = (j / P.chunks) & 1, c = j % P.chunks;
          const int key0 = kbase + b * P.box_rows;
          const long long row0 =
              ((((static_cast<long long>(p.layer) * p.NP + page) * 2 + kv) * p.nkv + kvh) * p.P) +
              key0 % p.P;
          const uint32_t dst =
              ptx::smem_u32(stage + kv * P.k_bytes + c * kVChunk + b * P.box_rows * 128);
          ptx::tma_load_2d_hint(dst, &tm, c * 64, static_cast<int32_t>(row0),
                                ptx::smem_u32(&kv_full[st]), pol);
        }
      }
      ++issued;
    }
    if (!ok && lane == 0) {
      for (int t = *consumed; t < issued; ++t) {
        volatile int dummy = 0;
        ptx::mbar_wait(ptx::smem_u32(&kv_full[t % nst]), static_cast<uint32_t>((t / nst) & 1),
                       &dummy);
      }
    }
  } else if (ntiles > 0 && warp == 3) {
    if (lane == 0) {
      // ------------------------------------------------ QK issuer (warp 3)
      // S_t = Q K_t^T into S buffer t & 1 once tile t has landed and the
      // softmax has read S_{t-2} from that buffer.  A thread issues a
      // tcgen05.mma only every ~70 cycles, so QK and PV have an issuing
      // thread each: PV of tile t never waits behind QK of tile t+1.
      const uint64_t dk0 = ptx::desc_kmajor_sw128(ptx::smem_u32(sKV), 0);
      bool ok = ptx::mbar_wait(ptx::smem_u32(q_full), 0u, abort_flag);
      for (int t = 0; ok && t < ntiles; ++t) {
        const int st = t % nst;
        ok = ptx::mbar_wait(ptx::smem_u32(&kv_full[st]), static_cast<uint32_t>((t / nst) & 1),
                            abort_flag);
        if (ok && t >= 2)
          ok = ptx::mbar_wait(ptx::smem_u32(&s_free[t & 1]),
                              static_cast<uint32_t>(((t >> 1) & 1) ^ 1), abort_flag);
        if (!ok) break;
        ptx::tc_fence_after();
        *consumed = t + 1;
        const uint64_t kb = dk0 + ((st * P.stage_bytes) >> 4);
        for (int ks = 0; ks < P.chunks * 4; ++ks) {
          const int c = ks >> 2, j = ks & 3;
          ptx::mma_bf16_ts(tm_s + (t & 1) * kKT, tm_q + ks * 8, kb + ((c * kVChunk + j * 32) >> 4),
                           P.idesc_qk, ks > 0 ? 1u : 0u);
        }
        ptx::mma_commit(ptx::smem_u32(&s_full[t & 1]));
      }
      if (!ok) {
        ptx::mma_commit(ptx::smem_u32(drain));
        volatile int dummy = 0;
        ptx::mbar_wait(ptx::smem_u32(drain), 0u, &dummy);
      }
    }
  } else if (ntiles > 0 && warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ PV issuer (warp 0)
      // O += P_t V_t once the softmax has written P_t; its completion frees
      // the ring stage (QK of the tile completed before its softmax began).
      const uint64_t dv0 = ptx::smem_desc(ptx::smem_u32(sKV) + P.k_bytes, P.v_lbo, P.v_sbo,
                                          ptx::kSwizzle128B);
      bool ok = true;
      for (int t = 0; ok && t < ntiles; ++t) {
        ok = ptx::mbar_wait(ptx::smem_u32(p_full), static_cast<uint32_t>(t & 1), abort_flag);
        if (!ok) break;
        ptx::tc_fence_after();
        const int st = t % nst;
        const uint64_t vb = dv0 + ((st * P.stage_bytes) >> 4);
#pragma unroll
        for (int ks = 0; ks < kKT / 16; ++ks)
          ptx::mma_bf16_ts(tm_o, tm_p + ks * 8, vb + ((ks * 2048) >> 4), P.idesc_pv,
                           (t > 0 || ks > 0) ? 1u : 0u);
        ptx::mma_commit(ptx::smem_u32(o_done));
        ptx::mma_commit(ptx::smem_u32(&kv_empty[st]));
      }
      if (!ok) {
        ptx::mma_commit(ptx::smem_u32(drain_pv));
        volatile int dummy = 0;
        ptx::mbar_wait(ptx::smem_u32(drain_pv), 0u, &dummy);
      }
    }
  } else if (warp >= 4 && kSplit) {
    // ------------------------------------------------ softmax, split layout
    // Warp pair (q4, q4 ^ 2) shares query rows 32*(q4&1)..+31: warp q4 < 2
    // takes key columns 0-63 from TMEM lanes of rows 0-63, warp q4 >= 2 takes
    // columns 64-127 from the duplicate rows 64-127.  Row maxima are exchanged
    // through shared memory behind a pair barrier (double-buffered by tile
    // parity); every abort decision is made pair-uniform at that barrier, so
    // both partners take identical rescale decisions and their O halves stay
    // on one scale.
    const int q4 = warp & 3;
    const int half = q4 >> 1;
    const int rrow = 32 * (q4 & 1) + lane;
    const bool real = rrow < P.GT;
    const int i = real ? rrow / p.G : 0;
    const int h = kvh * p.G + (real ? rrow % p.G : 0);
    int lo = 0, hi = -1;
    if (real) row_key_range(p, sr.kv_len, i, &lo, &hi);
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t pair_bar = 2u + static_cast<uint32_t>(q4 & 1);
    float *xmax = reinterpret_cast<float *>(sm + P.x_off);  // [2 parity][2 half][64 rows]
    float *xl = xmax + 256;                                 // [64 rows]
    float m_ref = -INFINITY, l = 0.f;
    bool bad = false;
    for (int t = 0; t < ntiles; ++t) {
      const bool got = __all_sync(0xffffffffu,
                                  ptx::mbar_wait(ptx::smem_u32(&s_full[t & 1]),
                                                 static_cast<uint32_t>((t >> 1) & 1), abort_flag));
      float sv[64];
      if (got) {
        ptx::tc_fence_after();
        ptx::tmem_ld64f_sync(tm_s + lane_off + (t & 1) * kKT + 64 * half, sv);
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&s_free[t & 1]));
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c) sv[c] = -INFINITY;
      }
      const int kbase = (sr.t0 + t) * kKT + 64 * half;
      if (!(lo <= kbase && hi >= kbase + 63)) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (kbase + c < lo || kbase + c > hi) sv[c] = -INFINITY;
      }
      float mx[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) mx[c] = fmaxf(sv[c], sv[c + 32]);
#pragma unroll
      for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
        for (int c = 0; c < w; ++c) mx[c] = fmaxf(mx[c], mx[c + w]);
      xmax[((t & 1) * 2 + half) * 64 + rrow] = mx[0];
      if (ptx::bar_or(pair_bar, 64, bad || !got)) {
        bad = true;
        break;
      }
      const float tmax = fmaxf(mx[0], xmax[((t & 1) * 2 + (half ^ 1)) * 64 + rrow]) * P.scale_log2;
      float corr = 1.f;
      bool need = false;
      if (m_ref == -INFINITY) {
        m_ref = tmax;
      } else if (tmax > m_ref + 8.f) {
        corr = ptx::ex2(m_ref - tmax);
        m_ref = tmax;
        need = true;
      }
      uint32_t pk[32];
      float sum = 0.f;
      if (m_ref != -INFINITY) {
        const float nm = -m_ref;
#pragma unroll
        for (int c = 0; c < 64; ++c) sv[c] = ptx::ex2(fmaf(sv[c], P.scale_log2, nm));
#pragma unroll
        for (int c = 0; c < 32; ++c) pk[c] = ptx::pack_bf16x2(sv[2 * c], sv[2 * c + 1]);
#pragma unroll
        for (int c = 0; c < 32; ++c) mx[c] = sv[c] + sv[c + 32];
#pragma unroll
        for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
          for (int c = 0; c < w; ++c) mx[c] += mx[c + w];
        sum = mx[0];
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) pk[c] = 0u;
      }
      l = l * corr + sum;
      // PV of the previous tile must be done before O is rescaled and before
      // the single P buffer is overwritten.
      if (t > 0) {
        const bool got_o = __all_sync(0xffffffffu,
                                      ptx::mbar_wait(ptx::smem_u32(o_done),
                                                     static_cast<uint32_t>((t - 1) & 1), abort_flag));
        if (!got_o) {
          bad = true;  // the next pair barrier (or the epilogue's) carries it
          continue;
        }
        ptx::tc_fence_after();
        if (__any_sync(0xffffffffu, need)) {
          for (int c = 0; c < p.dv; c += 16) {
            uint32_t ov[16];
            ptx::tmem_ld16_sync(tm_o + lane_off + c, ov);
#pragma unroll
            for (int e = 0; e < 16; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * corr);
            ptx::tmem_st16(tm_o + lane_off + c, ov);
          }
        }
      }
      {
        uint32_t p0[16], p1[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          p0[c] = pk[c];
          p1[c] = pk[16 + c];
        }
        ptx::tmem_st16(tm_p + lane_off + 32 * half, p0);
        ptx::tmem_st16(tm_p + lane_off + 32 * half + 16, p1);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(p_full));
    }
    // epilogue: the half-1 warp hands its partial row sums and its O half to
    // the half-0 warp (through the idle KV ring), which writes (m, l, O) of
    // rows 0-63
    bool okf = !bad && ntiles > 0;
    if (okf) {
      okf = __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(o_done),
                                                   static_cast<uint32_t>((ntiles - 1) & 1),
                                                   abort_flag));
      ptx::tc_fence_after();
    }
    float *xo = reinterpret_cast<float *>(sKV);  // [head_dim][64 rows]
    if (half == 1) {
      xl[rrow] = l;
      if (okf) {
        for (int c = 0; c < p.dv; c += 16) {
          uint32_t ov[16];
          ptx::tmem_ld16_sync(tm_o + lane_off + c, ov);
#pragma unroll
          for (int e = 0; e < 16; ++e) xo[(c + e) * 64 + rrow] = __uint_as_float(ov[e]);
        }
      }
    }
    const bool pair_bad = ptx::bar_or(pair_bar, 64, !okf && ntiles > 0);
    if (half == 0) {
      const bool any = real && !pair_bad && ntiles > 0 && m_ref != -INFINITY;
      const size_t wsi = ((static_cast<size_t>(r) * p.Tq + i) * p.hq + h) * p.S + s;
      if (real) {
        p.ws_m[wsi] = any ? m_ref * 0.69314718055994530942f : -INFINITY;
        p.ws_l[wsi] = any ? l + xl[rrow] : 0.f;
      }
      if (__any_sync(0xffffffffu, any)) {
        float4 *dst = reinterpret_cast<float4 *>(p.ws_o + wsi * p.dv);
        for (int c = 0; c < p.dv; c += 16) {
          uint32_t ov[16];
          ptx::tmem_ld16_sync(tm_o + lane_off + c, ov);
          if (any) {
            float o[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = __uint_as_float(ov[e]) + xo[(c + e) * 64 + rrow];
#pragma unroll
            for (int e = 0; e < 16; e += 4)
              dst[(c + e) / 4] = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
          }
        }
      }
    }
  } else if (warp >= 4 && !kSplit) {
    // ------------------------------------------------ softmax / epilogue
    const int q4 = warp & 3;
    const int row = 32 * q4 + lane;
    const int R = rt * kRows + row;
    const bool real = R < P.GT;
    // warps whose 32 rows are all padding sit the tile loop out (warp-uniform)
    const bool warp_active = rt * kRows + 32 * q4 < P.GT;
    const int i = real ? R / p.G : 0;
    const int h = kvh * p.G + (real ? R % p.G : 0);
    int lo = 0, hi = -1;
    if (real) row_key_range(p, sr.kv_len, i, &lo, &hi);
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int t = 0; t < ntiles && warp_active; ++t) {
      const bool got_s = ptx::mbar_wait(ptx::smem_u32(&s_full[t & 1]),
                                        static_cast<uint32_t>((t >> 1) & 1), abort_flag);
      if (!__all_sync(0xffffffffu, got_s)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const int kbase = (sr.t0 + t) * kKT;
      const bool partial = !(lo <= kbase && hi >= kbase + kKT - 1);  // row sees part of the tile
      // pass 1: tile maximum of the raw scores over both 64-column halves
      float raw_max = -INFINITY;
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        float sv[64];
        ptx::tmem_ld64f_sync(tm_s + lane_off + (t & 1) * kKT + 64 * hh, sv);
        if (partial) {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (kbase + 64 * hh + c < lo || kbase + 64 * hh + c > hi) sv[c] = -INFINITY;
        }
        float mx[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) mx[c] = fmaxf(sv[c], sv[c + 32]);
#pragma unroll
        for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
          for (int c = 0; c < w; ++c) mx[c] = fmaxf(mx[c], mx[c + w]);
        raw_max = fmaxf(raw_max, mx[0]);
      }
      const float tmax = raw_max * P.scale_log2;
      float corr = 1.f;
      bool need = false;
      if (m_ref == -INFINITY) {
        m_ref = tmax;
      } else if (tmax > m_ref + 8.f) {
        corr = ptx::ex2(m_ref - tmax);
        m_ref = tmax;
        need = true;
      }
      // PV of the previous tile must be done before O is rescaled and before
      // the single P buffer is overwritten.
      if (t > 0) {
        const bool got_o = ptx::mbar_wait(ptx::smem_u32(o_done),
                                          static_cast<uint32_t>((t - 1) & 1), abort_flag);
        if (!__all_sync(0xffffffffu, got_o)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        if (__any_sync(0xffffffffu, need)) {
          for (int c = 0; c < p.dv; c += 16) {
            uint32_t ov[16];
            ptx::tmem_ld16_sync(tm_o + lane_off + c, ov);
#pragma unroll
            for (int e = 0; e < 16; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * corr);
            ptx::tmem_st16(tm_o + lane_off + c, ov);
          }
        }
      }
      // pass 2: P = exp2(s - m) per half, straight into TMEM
      float sum = 0.f;
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        float sv[64];
        ptx::tmem_ld64f_sync(tm_s + lane_off + (t & 1) * kKT + 64 * hh, sv);
        if (partial) {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (kbase + 64 * hh + c < lo || kbase + 64 * hh + c > hi) sv[c] = -INFINITY;
        }
        uint32_t p0[16], p1[16];
        if (m_ref != -INFINITY) {
          const float nm = -m_ref;
#pragma unroll
          for (int c = 0; c < 64; ++c) sv[c] = ptx::ex2(fmaf(sv[c], P.scale_log2, nm));
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            p0[c] = ptx::pack_bf16x2(sv[2 * c], sv[2 * c + 1]);
            p1[c] = ptx::pack_bf16x2(sv[32 + 2 * c], sv[32 + 2 * c + 1]);
          }
          float mx[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) mx[c] = sv[c] + sv[c + 32];
#pragma unroll
          for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
            for (int c = 0; c < w; ++c) mx[c] += mx[c + w];
          sum += mx[0];
        } else {
#pragma unroll
          for (int c = 0; c < 16; ++c) p0[c] = p1[c] = 0u;
        }
        ptx::tmem_st16(tm_p + lane_off + 32 * hh, p0);
        ptx::tmem_st16(tm_p + lane_off + 32 * hh + 16, p1);
      }
      l = l * corr + sum;
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        ptx::mbar_arrive(ptx::smem_u32(&s_free[t & 1]));
        ptx::mbar_arrive(ptx::smem_u32(p_full));
      }
    }
    // epilogue: (m, l, O) of this segment
    if (ntiles > 0 && ok && warp_active) {
      const bool got_o = ptx::mbar_wait(ptx::smem_u32(o_done),
                                        static_cast<uint32_t>((ntiles - 1) & 1), abort_flag);
      ok = __all_sync(0xffffffffu, got_o);
      ptx::tc_fence_after();
    }
    const bool any = real && ok && ntiles > 0 && m_ref != -INFINITY;
    const size_t wsi = ((static_cast<size_t>(r) * p.Tq + i) * p.hq + h) * p.S + s;
    if (real) {
      p.ws_m[wsi] = any ? m_ref * 0.69314718055994530942f : -INFINITY;
      p.ws_l[wsi] = any ? l : 0.f;
    }
    // TMEM loads are warp-collective: the whole warp loads when any lane needs it.
    if (__any_sync(0xffffffffu, any)) {
      float4 *dst = reinterpret_cast<float4 *>(p.ws_o + wsi * p.dv);
      for (int c = 0; c < p.dv; c += 16) {
        uint32_t ov[16];
        ptx::tmem_ld16_sync(tm_o + lane_off + c, ov);
        if (any) {
#pragma unroll
          for (int e = 0; e < 16; e += 4)
            dst[(c + e) / 4] = make_float4(__uint_as_float(ov[e]), __uint_as_float(ov[e + 1]),
                                           __uint_as_float(ov[e + 2]), __uint_as_float(ov[e + 3]));
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) raise_status(p.st, DFLASH_DEV_WAIT_TIMEOUT);
  if (warp == 3) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

thread_local int t_skip_tile = -1;

}  // namespace

void attention_test_skip_tile(int tile) { t_skip_tile = tile; }
int attention_test_skip_tile_value() { return t_skip_tile; }

cudaError_t launch_attn_tc(const AttnParams &a, const dflash_geom &g, cudaStream_t s) {
  TcParams P;
  P.a = a;
  P.skip_tile = t_skip_tile;
  const int hd = g.head_dim;  // 64 or 128 (validated by the caller)
  P.chunks = hd / 64;
  P.GT = a.Tq * a.G;
  P.RT = (P.GT + kRows - 1) / kRows;
  P.box_rows = a.P < kKT ? a.P : kKT;
  // Split layout when a KV head's query rows fit in half the MMA rows.
  P.split = P.GT <= 64 ? 1 : 0;
  P.k_bytes = P.chunks * kVChunk;
  P.stage_bytes = 2 * P.k_bytes;
  const uint32_t x_bytes = 320 * 4;  // split-layout row maxima and row sums
  const uint32_t bar_bytes = 8 * 8 * 2 + 10 * 8 + 16;
  P.nst = std::max(2, std::min<int>(8, static_cast<int>((kSmemMax - 1024 - bar_bytes - x_bytes) /
                                                          P.stage_bytes)));
  P.bar_off = P.nst * P.stage_bytes;
  P.x_off = (P.bar_off + (2 * P.nst + 10) * 8 + 16 + 15) & ~15u;
  const uint32_t smem = 1024 + P.x_off + x_bytes;
  P.idesc_qk = ptx::idesc_bf16_f32(kRows, kKT, false);
  P.idesc_pv = ptx::idesc_bf16_f32(kRows, hd, true);
  P.v_lbo = kVChunk;
  P.v_sbo = 1024;
  P.scale_log2 = a.scale * 1.4426950408889634f;  // scale > 0 (validated by the caller)

  CUtensorMap tm;
  const uint64_t rows = static_cast<uint64_t>(g.num_layers) * g.num_pool_pages * 2 * g.nkv *
                        static_cast<uint64_t>(g.page_size);
  cudaError_t e = make_tmap_bf16_2d(&tm, a.pool, rows, hd, hd, P.box_rows, 64);
  if (e != cudaSuccess) return e;
  if ((e = ensure_smem_limit<attn_tc_kernel<true, false>>(kSmemMax)) != cudaSuccess) return e;
  if ((e = ensure_smem_limit<attn_tc_kernel<false, false>>(kSmemMax)) != cudaSuccess) return e;
  if ((e = ensure_smem_limit<attn_tc_kernel<true, true>>(kSmemMax)) != cudaSuccess) return e;
  if ((e = ensure_smem_limit<attn_tc_kernel<false, true>>(kSmemMax)) != cudaSuccess) return e;
  const bool scat = a.blk_k != nullptr;
  auto kern = P.split ? (scat ? attn_tc_kernel<true, true> : attn_tc_kernel<true, false>)
                      : (scat ? attn_tc_kernel<false, true> : attn_tc_kernel<false, false>);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(a.S * P.RT, a.nkv, a.B);
  cfg.blockDim = dim3(kThreadsTC);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tm, P);
}

}  // namespace dflash
