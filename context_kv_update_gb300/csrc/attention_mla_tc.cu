// attention_mla_tc.cu -- split-KV block attention over the single shared MLA
// latent, on the 5th-generation tensor cores.
//
// Follows vLLM PR #54092 (Purpose item 2, Changes item 2) for the split-KV
// form (per-segment partial softmax state over the visible keys, a separate
// reduce), applied to the absorbed-latent drafter attention: every query row
// (token i, head h) scores one 512 + 64 wide latent row per key,
//   s_j = scale * (<q_lat, c_j> + <q_rope, r_j>),  values c_j (512 wide).
//
// With 512-wide values a 128-row output tile alone would fill all of TMEM,
// and the 576-wide queries of 128 rows would not fit next to it.  So a CTA
// takes 64 query rows and keeps keys, not rows, in TMEM lanes:
//   S^T[128 keys x 64 rows] = K[128 x 576] . Q^T      (A = K from smem, K-major;
//                                                      B = Q from smem, K-major)
//   O^T[512 dims x 64 rows] += V^T[512 x 128] . P^T   (A = the same latent rows
//                                                      read MN-major; B = P^T)
// in four 128-dim blocks.  The MMAs of a tile are issued by two threads (one
// thread issues a tcgen05.mma only every ~70 cycles, about twice what an
// N = 64 MMA takes to execute): each runs QK over part of the chunks into its
// own S^T partial, which the softmax adds, and two of the four PV blocks.
// TMEM: two S^T buffers of 2 x 64 columns + 4 x 64 O^T columns.  Shared
// memory: Q (9 chunks of 64 rows x 64 dims, 72 KB) and one
// 128-key tile as 9 chunks of 64 dims (8 latent + 1 rope, 144 KB); the rope
// chunk's slot then holds P^T (it is free once QK has read it).
//
// The softmax warps hold one key per thread and 64 row scores.  They keep a
// per-row reference maximum m_ref in shared memory and only rebuild it (an
// exact cross-lane maximum, O^T and the row-sum partials rescaled) when some
// score of the tile exceeds m_ref by more than 2^8 -- on the first tile and
// rarely after.  P = exp2(s - m_ref) goes to shared memory as the PV operand;
// each thread accumulates its key's share of the row sums, reduced across
// the 128 keys once at the end.
//
// A tile is loaded chunk by chunk: chunks 2b, 2b+1 of tile t+1 are issued as
// soon as PV block b of tile t has released their slots (the rope chunk once
// the whole PV is done), and QK of tile t+1 starts on chunk 0 while the
// others are still landing.  The boxes of a slot group (2 chunks x 2 pages
// of 64 keys) are issued by different lanes at once: a TMA issue does not
// return before the copy engine takes it, so boxes issued one after another
// (by one lane, or one lane per loop step) refill a tile ~2x slower.  Every mbarrier wait is a
// bounded try_wait; a timeout raises DFLASH_DEV_WAIT_TIMEOUT.
#include <cuda.h>

#include <algorithm>

#include "attention_common.cuh"

namespace dflash {

cudaError_t make_tmap_bf16_2d(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols,
                              uint64_t row_stride_elems, uint32_t box_rows, uint32_t box_cols);

namespace {

constexpr int kKT = kAttnTileKeys;  // 128 keys per tile (MMA M of QK)
static_assert(kKT == 128, "keys fill the 128 TMEM lanes");
constexpr int kRowsN = 64;          // query rows per CTA (MMA N)
constexpr int kThreads = 256;
constexpr int kLat = 512;
constexpr int kWidth = 576;                 // latent + rope
constexpr int kChunks = kWidth / 64;        // 9 dim chunks: 0-7 latent, 8 rope
constexpr int kRopeSlot = kChunks - 1;
constexpr uint32_t kChunkBytes = kKT * 128;      // 128 keys x 64 dims
constexpr uint32_t kQChunkBytes = kRowsN * 128;  // 64 rows x 64 dims
constexpr uint32_t kSlotOff = kChunks * kQChunkBytes;
constexpr uint32_t kBarOff = kSlotOff + kChunks * kChunkBytes;
constexpr int kNumBars = 20;
constexpr uint32_t kXOff = (kBarOff + kNumBars * 8 + 8 + 15) & ~15u;
constexpr uint32_t kXBytes = (2 * 64 + 64 * 4 + 64 * 4) * 4 + 64 * 8;  // m_ref[2][64], xm, xl, roff
constexpr uint32_t kSmemBytes = 1024 + kXOff + kXBytes;
static_assert(kSmemBytes <= 227 * 1024, "shared memory plan");
constexpr uint32_t kColS = 0;    // two S^T buffers of 2 x 64 columns (one partial per issuer)
constexpr uint32_t kColO = 256;  // O^T: 4 blocks x 64 columns
constexpr uint32_t kTmemCols = 512;
constexpr float kLn2 = 0.69314718055994530942f;

struct MlaParams {
  AttnParams a;
  int GT, RT, box_rows;
  uint32_t idesc_qk, idesc_pv;
  float scale_log2;
};

__device__ __forceinline__ uint32_t sw128_off(int row, int unit16) {
  return static_cast<uint32_t>(row * 128 + ((unit16 ^ (row & 7)) << 4));
}

// Reduce 64 per-lane values across the warp, one row per value: after five
// exchange steps (32 + 16 + 8 + 4 + 2 shuffles instead of 5 per row) lane L
// holds the results of rows 2L and 2L + 1 in v[0], v[1] (at the step that
// exchanges lane bit o, the lane with that bit set keeps the upper half).
// MAX selects fmaxf, else addition.
template <bool MAX>
__device__ __forceinline__ void warp_transpose_reduce64(float (&v)[64], int lane) {
#pragma unroll
  for (int st = 0; st < 5; ++st) {
    const int o = 16 >> st;      // lane bit exchanged at this step
    const int half = 32 >> st;   // values kept per lane after the step
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int j = 0; j < half; ++j) {
      const float send = upper ? v[j] : v[j + half];
      const float keep = upper ? v[j + half] : v[j];
      const float recv = __shfl_xor_sync(0xffffffffu, send, o);
      v[j] = MAX ? fmaxf(keep, recv) : keep + recv;
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_mla_tc_kernel(const __grid_constant__ CUtensorMap tm, const MlaParams P) {
  const AttnParams &p = P.a;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  uint8_t *sQ = sm;
  uint8_t *sSlot = sm + kSlotOff;
  uint8_t *sPT = sSlot + kRopeSlot * kChunkBytes;  // P^T shares the rope chunk's slot
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kBarOff);
  uint64_t *ch_full = bars;           // [9]  chunk slot filled
  uint64_t *blk_empty = bars + 9;     // [4]  PV block b done with slots 2b, 2b+1
  uint64_t *s_full = bars + 13;       // [2]  S^T buffer written
  uint64_t *p_full = bars + 15;       //      P^T written (4 softmax warps)
  uint64_t *o_done = bars + 16;       //      PV of the tile complete (2 issuers)
  uint64_t *q_full = bars + 17;       //      Q in shared memory (2 warps)
  uint64_t *drain = bars + 18;        // [2]  per-issuer wind-down
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + kNumBars);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tslot + 1);
  float *m_ref = reinterpret_cast<float *>(sm + kXOff);  // [2][64], log2 units
  float *xm = m_ref + 128;                              // [64 rows][4 warps]
  float *xl = xm + 256;                                 // [64 rows][4 warps]
  long long *roff = reinterpret_cast<long long *>(xl + 256);  // [64 rows] workspace row

  const int s = blockIdx.x / P.RT, rg = blockIdx.x % P.RT;
  const int r = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R0 = rg * kRowsN;

  if (threadIdx.x == 0) {
    for (int c = 0; c < kChunks; ++c) ptx::mbar_init(ptx::smem_u32(&ch_full[c]), 1);
    for (int b = 0; b < 4; ++b) ptx::mbar_init(ptx::smem_u32(&blk_empty[b]), 1);
    ptx::mbar_init(ptx::smem_u32(&s_full[0]), 2);
    ptx::mbar_init(ptx::smem_u32(&s_full[1]), 2);
    ptx::mbar_init(ptx::smem_u32(p_full), 4);
    ptx::mbar_init(ptx::smem_u32(o_done), 2);
    ptx::mbar_init(ptx::smem_u32(q_full), 2);
    ptx::mbar_init(ptx::smem_u32(&drain[0]), 1);
    ptx::mbar_init(ptx::smem_u32(&drain[1]), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tm);
  }
  if (threadIdx.x >= 128 && threadIdx.x < 192) {
    m_ref[threadIdx.x - 128] = -INFINITY;
    m_ref[64 + threadIdx.x - 128] = -INFINITY;
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
  griddep_wait();
  const SegRange sr = segment_range(p, r, s);
  const int ntiles = sr.t1 - sr.t0;
  const uint32_t tm_s = tmem + kColS;
  const uint32_t tm_o = tmem + kColO;

  if (warp < 2 && ntiles > 0) {
    // ------------------------------------------------ Q -> smem (warps 0-1)
    // one row per thread: 64 latent + 8 rope 16-byte units, K-major SW128
    const int rho = threadIdx.x;
    const int R = R0 + rho;
    const bool real = R < P.GT;
    const int i = real ? R / p.hq : 0, h = real ? R % p.hq : 0;
    const size_t qi = (static_cast<size_t>(r) * p.Tq + i) * p.hq + h;
    const uint4 *ql = reinterpret_cast<const uint4 *>(p.q + qi * kLat);
    const uint4 *qr = reinterpret_cast<const uint4 *>(p.q_rope + qi * (kWidth - kLat));
#pragma unroll 8
    for (int u = 0; u < kChunks * 8; ++u) {
      const uint4 v = !real ? make_uint4(0, 0, 0, 0) : (u < 64 ? ql[u] : qr[u - 64]);
      *reinterpret_cast<uint4 *>(sQ + (u >> 3) * kQChunkBytes + sw128_off(rho, u & 7)) = v;
    }
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(q_full));
  } else if (ntiles > 0 && warp == 2) {
    // ------------------------------------------------ TMA producer (warp 2)
    const int boxes = kKT / P.box_rows;
    const int tiles_per_batch = 32 / boxes;
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
    int last_fill[kChunks];
#pragma unroll
    for (int c = 0; c < kChunks; ++c) last_fill[c] = -1;
    bool ok = true;
    for (int t = 0; t < ntiles && ok; ++t) {
      const int tb = t % tiles_per_batch;
      if (tb == 0 && t > 0) {
        cur = nxt;
        nxt = fetch_page(t + tiles_per_batch);
      }
      const int kbase = (sr.t0 + t) * kKT;
      // groups of slots released together: chunks {0,1}, {2,3}, {4,5},
      // {6,7} by PV blocks 0-3 of the previous tile, the rope chunk by its end
      for (int grp = 0; grp < 5 && ok; ++grp) {
        const int c_lo = 2 * grp, c_hi = grp < 4 ? 2 * grp + 2 : kChunks;
        bool got = true;
        if (lane == 0 && t > 0) {
          uint64_t *bar = grp < 4 ? &blk_empty[grp] : o_done;
          got = ptx::mbar_wait(ptx::smem_u32(bar), static_cast<uint32_t>((t - 1) & 1), abort_flag);
        }
        if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) {
          ok = false;
          break;
        }
        if (lane == 0)
          for (int c = c_lo; c < c_hi; ++c)
            ptx::mbar_arrive_expect_tx(ptx::smem_u32(&ch_full[c]), kChunkBytes);
        __syncwarp();
        // the group's boxes (chunk x page box) are issued by different lanes
        // at once: a lane's TMA issue does not return before the copy engine
        // takes it, so boxes issued one after another by one lane serialise
        const int nb = (c_hi - c_lo) * boxes;
        for (int j0 = 0; j0 < nb; j0 += 32) {
          const int jj = j0 + lane;
          const int j = c_lo * boxes + (jj < nb ? jj : 0);
          const int c = j / boxes, b = j % boxes;
          const int page = __shfl_sync(0xffffffffu, cur, tb * boxes + b);
          if (jj < nb) {
            const int key0 = kbase + b * P.box_rows;
            const long long row0 =
                (static_cast<long long>(p.layer) * p.NP + page) * p.P + key0 % p.P;
            ptx::tma_load_2d(ptx::smem_u32(sSlot + c * kChunkBytes + b * P.box_rows * 128), &tm,
                             c * 64, static_cast<int32_t>(row0), ptx::smem_u32(&ch_full[c]));
          }
        }
        for (int c = c_lo; c < c_hi; ++c) last_fill[c] = t;
      }
    }
    if (!ok && lane == 0) {
      // let the copies in flight land before the CTA exits
      for (int c = 0; c < kChunks; ++c) {
        if (last_fill[c] < 0) continue;
        volatile int dummy = 0;
        ptx::mbar_wait(ptx::smem_u32(&ch_full[c]), static_cast<uint32_t>(last_fill[c] & 1), &dummy);
      }
    }
  }
  if (ntiles > 0 && lane == 0 && (warp == 3 || warp == 0)) {
    // ------------------------------------------------ MMA issuers
    // One thread issues a tcgen05.mma only every ~70 cycles, and these N = 64
    // MMAs execute in about half that, so the work of a tile is split over
    // two issuing threads (warp 3 and warp 0, after its Q rows): issuer 0
    // runs QK over latent chunks 0-4 into one S^T partial and PV blocks 0-1;
    // issuer 1 QK over chunks 5-8 (rope) into a second partial and PV blocks
    // 2-3.  The softmax adds the two partials.  Descriptors are formed once
    // and advanced by adding the byte offset (>> 4) to the address field.
    const int role = warp == 3 ? 0 : 1;
    const int c_lo = role == 0 ? 0 : 5, c_hi = role == 0 ? 5 : kChunks;
    const int b_lo = 2 * role;
    const uint64_t dq0 = ptx::desc_kmajor_sw128(ptx::smem_u32(sQ), 0);
    const uint64_t dk0 = ptx::desc_kmajor_sw128(ptx::smem_u32(sSlot), 0);
    const uint64_t dv0 = ptx::smem_desc(ptx::smem_u32(sSlot), kChunkBytes, 1024, ptx::kSwizzle128B);
    const uint64_t dp0 = ptx::smem_desc(ptx::smem_u32(sPT), kChunkBytes, 1024, ptx::kSwizzle128B);
    bool ok = ptx::mbar_wait(ptx::smem_u32(q_full), 0u, abort_flag);
    for (int t = 0; ok && t < ntiles; ++t) {
      const uint32_t ph = static_cast<uint32_t>(t & 1);
      const uint32_t d_s = tm_s + (t & 1) * (2 * kRowsN) + role * kRowsN;
      // S^T partial = K_t Q^T over this issuer's chunks, each as it lands
      for (int c = c_lo; c < c_hi && ok; ++c) {
        ok = ptx::mbar_wait(ptx::smem_u32(&ch_full[c]), ph, abort_flag);
        if (!ok) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int j = 0; j < 4; ++j)
          ptx::mma_bf16(d_s, dk0 + ((c * kChunkBytes + j * 32) >> 4),
                        dq0 + ((c * kQChunkBytes + j * 32) >> 4), P.idesc_qk,
                        (c > c_lo || j > 0) ? 1u : 0u);
      }
      if (!ok) break;
      ptx::mma_commit(ptx::smem_u32(&s_full[t & 1]));
      // O^T += V^T P^T for this issuer's two 128-dim blocks
      ok = ptx::mbar_wait(ptx::smem_u32(p_full), ph, abort_flag);
      if (!ok) break;
      ptx::tc_fence_after();
#pragma unroll
      for (int bb = 0; bb < 2; ++bb) {
        const int b = b_lo + bb;
#pragma unroll
        for (int ks = 0; ks < kKT / 16; ++ks)
          ptx::mma_bf16(tm_o + b * kRowsN, dv0 + ((2 * b * kChunkBytes + ks * 2048) >> 4),
                        dp0 + ((ks * 2048) >> 4), P.idesc_pv, (t > 0 || ks > 0) ? 1u : 0u);
        ptx::mma_commit(ptx::smem_u32(&blk_empty[b]));
      }
      ptx::mma_commit(ptx::smem_u32(o_done));
    }
    if (!ok) {
      ptx::mma_commit(ptx::smem_u32(&drain[role]));
      volatile int dummy = 0;
      ptx::mbar_wait(ptx::smem_u32(&drain[role]), 0u, &dummy);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------ softmax (warps 4-7)
    const int q4 = warp & 3;
    const int key = 32 * q4 + lane;  // TMEM lane = key within the tile
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    // visible key range of a query token
    auto lo_of = [&](int i) {
      if (p.window <= 0) return 0;
      const int w0 = sr.kv_len - p.Tq + i - p.window + 1;
      return w0 > 0 ? w0 : 0;
    };
    auto hi_of = [&](int i) {
      return p.mask_mode == DFLASH_MASK_CAUSAL_TAIL ? sr.kv_len - p.Tq + i : sr.kv_len - 1;
    };
    const int R_last = min(R0 + kRowsN, P.GT) - 1;
    const int i_first = R0 / p.hq, i_last = max(R_last, R0) / p.hq;
    const int lo_max = lo_of(i_last), hi_min = hi_of(i_first);
    int cur = 0;  // m_ref buffer in use
    float lp[kRowsN];
#pragma unroll
    for (int c = 0; c < kRowsN; ++c) lp[c] = 0.f;
    bool bad = false;
    for (int t = 0; t < ntiles; ++t) {
      const bool got = __all_sync(0xffffffffu,
                                  ptx::mbar_wait(ptx::smem_u32(&s_full[t & 1]),
                                                 static_cast<uint32_t>((t >> 1) & 1), abort_flag));
      float sv[kRowsN];
      if (got) {
        ptx::tc_fence_after();
        const uint32_t sa = tm_s + lane_off + (t & 1) * (2 * kRowsN);
        ptx::tmem_ld64f_sync(sa, sv);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float s2[32];
          ptx::tmem_ld32f_sync(sa + kRowsN + 32 * h, s2);
#pragma unroll
          for (int c = 0; c < 32; ++c) sv[32 * h + c] += s2[c];
        }
      } else {
#pragma unroll
        for (int c = 0; c < kRowsN; ++c) sv[c] = -INFINITY;
      }
      const int tile0 = (sr.t0 + t) * kKT;
      const int kpos = tile0 + key;
      if (!(tile0 >= lo_max && tile0 + kKT - 1 <= hi_min)) {
        // a tile some row sees only in part (or past kv_len): mask per row
#pragma unroll
        for (int c = 0; c < kRowsN; ++c) {
          const int R = R0 + c;
          const int i = R / p.hq;
          if (R > R_last || kpos < lo_of(i) || kpos > hi_of(i)) sv[c] = -INFINITY;
        }
      }
      const float *mr = m_ref + 64 * cur;
      bool need = false;
#pragma unroll
      for (int c4 = 0; c4 < kRowsN / 4; ++c4) {
        const float4 m4 = *reinterpret_cast<const float4 *>(mr + 4 * c4);
        need |= sv[4 * c4] * P.scale_log2 > m4.x + 8.f;
        need |= sv[4 * c4 + 1] * P.scale_log2 > m4.y + 8.f;
        need |= sv[4 * c4 + 2] * P.scale_log2 > m4.z + 8.f;
        need |= sv[4 * c4 + 3] * P.scale_log2 > m4.w + 8.f;
      }
      if (ptx::bar_or(2, 128, need || !got)) {
        // ---- rebuild m_ref: exact tile maxima, rescale O^T and the row sums
        if (ptx::bar_or(3, 128, !got)) {
          bad = true;
          break;
        }
        bool got_o = true;
        if (t > 0)
          got_o = ptx::mbar_wait(ptx::smem_u32(o_done), static_cast<uint32_t>((t - 1) & 1),
                                 abort_flag);
        {
          float mx[kRowsN];
#pragma unroll
          for (int c = 0; c < kRowsN; ++c) mx[c] = sv[c];
          warp_transpose_reduce64<true>(mx, lane);
          const int row0 = 2 * lane;
          xm[row0 * 4 + q4] = mx[0];
          xm[(row0 + 1) * 4 + q4] = mx[1];
        }
        if (ptx::bar_or(2, 128, !got_o)) {
          bad = true;
          break;
        }
        ptx::tc_fence_after();
        float *mn = m_ref + 64 * (cur ^ 1);
        if (q4 < 2) {  // one row per thread
          const int c = 32 * q4 + lane;
          const float4 w4 = *reinterpret_cast<const float4 *>(xm + c * 4);
          const float tmax = fmaxf(fmaxf(w4.x, w4.y), fmaxf(w4.z, w4.w)) * P.scale_log2;
          const float old = mr[c];
          mn[c] = (old == -INFINITY || tmax > old + 8.f) ? tmax : old;
        }
        ptx::bar_sync(2, 128);
#pragma unroll
        for (int c = 0; c < kRowsN; ++c) {
          const float old = mr[c], nw = mn[c];
          lp[c] *= (old == -INFINITY || old == nw) ? 1.f : ptx::ex2(old - nw);
        }
        if (t > 0) {
          for (int b = 0; b < 4; ++b) {
            for (int c0 = 0; c0 < kRowsN; c0 += 16) {
              uint32_t ov[16];
              ptx::tmem_ld16_sync(tm_o + lane_off + b * kRowsN + c0, ov);
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const float old = mr[c0 + e], nw = mn[c0 + e];
                const float corr = (old == -INFINITY || old == nw) ? 1.f : ptx::ex2(old - nw);
                ov[e] = __float_as_uint(__uint_as_float(ov[e]) * corr);
              }
              ptx::tmem_st16(tm_o + lane_off + b * kRowsN + c0, ov);
            }
          }
          ptx::tmem_wait_st();
        }
        cur ^= 1;
      }
      // P = exp2(s - m_ref) -> P^T row `key` (64 rows = 8 units of 8), row sums
      const float *m2 = m_ref + 64 * cur;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        uint32_t pk[4];
        const float4 ma = *reinterpret_cast<const float4 *>(m2 + 8 * u);
        const float4 mb = *reinterpret_cast<const float4 *>(m2 + 8 * u + 4);
        const float mm[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = 8 * u + 2 * e;
          const float p0 =
              sv[c] == -INFINITY ? 0.f : ptx::ex2(fmaf(sv[c], P.scale_log2, -mm[2 * e]));
          const float p1 = sv[c + 1] == -INFINITY
                               ? 0.f
                               : ptx::ex2(fmaf(sv[c + 1], P.scale_log2, -mm[2 * e + 1]));
          lp[c] += p0;
          lp[c + 1] += p1;
          pk[e] = ptx::pack_bf16x2(p0, p1);
        }
        *reinterpret_cast<uint4 *>(sPT + sw128_off(key, u)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(p_full));
    }
    // ---- epilogue: row sums over the 128 keys, then (m, l, O) per real row
    bool okf = !bad && ntiles > 0;
    if (okf) {
      okf = __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(o_done),
                                                   static_cast<uint32_t>((ntiles - 1) & 1),
                                                   abort_flag));
      ptx::tc_fence_after();
    }
    warp_transpose_reduce64<false>(lp, lane);
    {
      const int row0 = 2 * lane;
      xl[row0 * 4 + q4] = lp[0];
      xl[(row0 + 1) * 4 + q4] = lp[1];
    }
    // per-row workspace offsets, computed once
    if (q4 < 2) {
      const int c = 32 * q4 + lane;
      const int R = R0 + c;
      long long off = -1;
      if (R < P.GT) {
        const int i = R / p.hq, h = R % p.hq;
        off = static_cast<long long>(((static_cast<size_t>(r) * p.Tq + i) * p.hq + h) * p.S + s);
      }
      roff[c] = off;
    }
    const bool any_bad = ptx::bar_or(2, 128, !okf && ntiles > 0);
    const float *mf = m_ref + 64 * cur;
    if (q4 < 2) {
      const int c = 32 * q4 + lane;
      const long long wsi = roff[c];
      if (wsi >= 0) {
        const bool any = !any_bad && ntiles > 0 && mf[c] != -INFINITY;
        const float4 l4 = *reinterpret_cast<const float4 *>(xl + c * 4);
        p.ws_m[wsi] = any ? mf[c] * kLn2 : -INFINITY;
        p.ws_l[wsi] = any ? (l4.x + l4.y) + (l4.z + l4.w) : 0.f;
      }
    }
    if (!any_bad && ntiles > 0) {
      // O^T (dims in lanes) -> O rows in the idle tile slots [64 rows][512]
      // (bank-conflict-free: a warp writes 32 consecutive dims of one row),
      // then every row leaves as coalesced 16-byte stores
      float *stage = reinterpret_cast<float *>(sSlot);
      for (int b = 0; b < 4; ++b) {
        const int d = b * 128 + 32 * q4 + lane;
        for (int c0 = 0; c0 < kRowsN; c0 += 16) {
          uint32_t ov[16];
          ptx::tmem_ld16_sync(tm_o + lane_off + b * kRowsN + c0, ov);
#pragma unroll
          for (int e = 0; e < 16; ++e) stage[(c0 + e) * kLat + d] = __uint_as_float(ov[e]);
        }
      }
      ptx::bar_sync(2, 128);
      const int tid = threadIdx.x - 128;
#pragma unroll 4
      for (int q = tid; q < kRowsN * kLat / 4; q += 128) {
        const int c = q / (kLat / 4), c4 = q % (kLat / 4);
        const long long wsi = roff[c];
        if (wsi >= 0 && mf[c] != -INFINITY)
          reinterpret_cast<float4 *>(p.ws_o + wsi * kLat)[c4] =
              reinterpret_cast<const float4 *>(stage)[q];
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

}  // namespace

int mla_rows_per_cta() { return kRowsN; }

cudaError_t launch_attn_mla_tc(const AttnParams &a, const dflash_geom &g, cudaStream_t s) {
  MlaParams P;
  P.a = a;
  P.GT = a.Tq * a.hq;
  P.RT = (P.GT + kRowsN - 1) / kRowsN;
  P.box_rows = a.P < kKT ? a.P : kKT;
  P.idesc_qk = ptx::idesc_bf16_f32(kKT, kRowsN, false, false);
  P.idesc_pv = ptx::idesc_bf16_f32(128, kRowsN, true, true);
  P.scale_log2 = a.scale * 1.4426950408889634f;
  CUtensorMap tm;
  const uint64_t rows = static_cast<uint64_t>(g.num_layers) * g.num_pool_pages *
                        static_cast<uint64_t>(g.page_size);
  cudaError_t e = make_tmap_bf16_2d(&tm, a.pool, rows, kWidth, kWidth, P.box_rows, 64);
  if (e != cudaSuccess) return e;
  if ((e = ensure_smem_limit(attn_mla_tc_kernel, 227 * 1024)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(a.S * P.RT, 1, a.B);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_mla_tc_kernel, tm, P);
}

}  // namespace dflash
