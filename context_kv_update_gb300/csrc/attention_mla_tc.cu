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
// takes 64 query rows and keeps keys, not rows, in TMEM lanes.  Keys come in
// half-tiles of 64 (two per 128-key segment tile), double-buffered in shared
// memory, so the copies of half-tile h+1 land while h is scored and applied:
//   S^T[64 keys x 64 rows] = K[64 x 576] . Q^T        (M = 64: TMEM lanes
//                                                      32q..32q+15 hold keys
//                                                      16q..16q+15)
//   O^T[512 dims x 64 rows] += V^T[512 x 64] . P^T    (four 128-dim blocks;
//                                                      A = the same latent rows
//                                                      read MN-major)
// QK of a half-tile is issued by two threads (one thread issues a
// tcgen05.mma only every ~70 cycles), each over half of the K-steps into its
// own S^T partial, which the softmax adds; QK of h+1 starts as soon as h+1
// has landed, so scoring the next half-tile overlaps the softmax of this one.
// PV is issued by the softmax warps themselves: once all four have written
// their P^T rows, each warp's lane 0 applies P^T to its own 128-dim block of
// O^T, with no hand-off to another thread.
// TMEM: two S^T buffers of 2 x 64 columns + 4 x 64 O^T columns.  Shared
// memory: Q (9 chunks of 64 rows x 64 dims, 72 KB), two half-tile buffers of
// 9 chunks of 64 keys x 64 dims (72 KB each), P^T (8 KB).
//
// The softmax warps read one key per lane from lanes 0-15 of each warp (the
// lanes the M = 64 result occupies); lane l keeps the key's rows 0-31 and
// hands rows 32-63 to lane l + 16, so every lane scores 32 rows.  They keep a
// per-row reference maximum m_ref in shared memory and only rebuild it (an
// exact cross-lane maximum, O^T and the row-sum partials rescaled) when some
// score of the half-tile exceeds m_ref by more than 2^8 -- on the first one
// and rarely after.  P = exp2(s - m_ref) goes to shared memory as the PV operand
// once the previous PV has read it; each thread accumulates its key's share
// of the row sums, reduced across the keys once at the end.
//
// When the call fuses the block scatter, the producer warp first writes the
// block's own latent rows of its key range into the cache (a separate
// instantiation, so the plain kernel carries none of that code).
//
// The copies of a half-tile (9 chunks x its pages) are issued by different
// lanes at once: a TMA issue does not return before the copy engine takes
// it, so boxes issued one after another refill a buffer ~2x slower.  Every
// mbarrier wait is a bounded try_wait; a timeout raises
// DFLASH_DEV_WAIT_TIMEOUT and every role winds down.
#include <cuda.h>

#include <algorithm>

#include "attention_common.cuh"

namespace dflash {

cudaError_t make_tmap_bf16_2d(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols,
                              uint64_t row_stride_elems, uint32_t box_rows, uint32_t box_cols);

namespace {

constexpr int kKT = kAttnTileKeys;  // 128 keys per segment tile
static_assert(kKT == 128, "a segment tile is two half-tiles");
constexpr int kHK = 64;             // keys per half-tile (MMA M of QK)
constexpr int kRowsN = 64;          // query rows per CTA (MMA N)
constexpr int kThreads = 256;
constexpr int kLat = 512;
constexpr int kWidth = 576;                 // latent + rope
constexpr int kChunks = kWidth / 64;        // 9 dim chunks: 0-7 latent, 8 rope
constexpr uint32_t kChunkBytes = kHK * 128;      // 64 keys x 64 dims
constexpr uint32_t kQChunkBytes = kRowsN * 128;  // 64 rows x 64 dims
constexpr uint32_t kBufBytes = kChunks * kChunkBytes;  // one half-tile
constexpr uint32_t kBufOff = kChunks * kQChunkBytes;
constexpr uint32_t kPTOff = kBufOff + 2 * kBufBytes;
constexpr uint32_t kBarOff = kPTOff + kHK * 128;  // P^T: 64 keys x 64 rows bf16
constexpr int kNumBars = 14;
constexpr uint32_t kXOff = (kBarOff + kNumBars * 8 + 8 + 15) & ~15u;
constexpr uint32_t kXBytes = (2 * 64 + 64 * 4) * 4;  // m_ref[2][64], xm[64][4]
constexpr uint32_t kSmemBytes = 1024 + kXOff + kXBytes;
static_assert(kSmemBytes <= 227 * 1024, "shared memory plan");
static_assert(64 * 4 * 4 + 64 * 8 <= kHK * 128, "xl and roff fit the idle P^T region");
static_assert(kRowsN * kLat * 4 <= 2 * kBufBytes, "the O rows fit the idle buffers");
constexpr uint32_t kColS = 0;    // two S^T buffers of 2 x 64 columns (one partial per issuer)
constexpr uint32_t kColO = 256;  // O^T: 4 blocks x 64 columns
constexpr uint32_t kTmemCols = 512;
constexpr float kLn2 = 0.69314718055994530942f;

struct MlaParams {
  AttnParams a;
  int GT, RT, box_rows;
  int skip_h;  // tests only: the producer never issues this half-tile (-1: off)
  uint32_t idesc_qk, idesc_pv;
  float scale_log2;
};

__device__ __forceinline__ uint32_t sw128_off(int row, int unit16) {
  return static_cast<uint32_t>(row * 128 + ((unit16 ^ (row & 7)) << 4));
}

// Reduce 32 per-lane values over each 16-lane half of the warp, one row per
// value: after four exchange steps (16 + 8 + 4 + 2 shuffles instead of 4 per
// row) lane L holds the results of rows 2(L mod 16) and 2(L mod 16) + 1 of its
// half in v[0], v[1] (at the step that exchanges lane bit o, the lane with
// that bit set keeps the upper half).  MAX selects fmaxf, else addition.
template <bool MAX>
__device__ __forceinline__ void half_warp_transpose_reduce32(float (&v)[32], int lane) {
#pragma unroll
  for (int st = 0; st < 4; ++st) {
    const int o = 8 >> st;       // lane bit exchanged at this step
    const int half = 16 >> st;   // values kept per lane after the step
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

template <bool kScatter>
__global__ void __launch_bounds__(kThreads, 1)
    attn_mla_tc_kernel(const __grid_constant__ CUtensorMap tm, const __grid_constant__ MlaParams P) {
  const AttnParams &p = P.a;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  uint8_t *sQ = sm;
  uint8_t *sBuf = sm + kBufOff;
  uint8_t *sPT = sm + kPTOff;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kBarOff);
  uint64_t *full = bars;          // [2] half-tile buffer filled
  uint64_t *empty = bars + 2;     // [2] buffer read by the four PV blocks
  uint64_t *s_full = bars + 4;    // [2] S^T buffer written (2 issuers)
  uint64_t *o_done = bars + 6;    //     PV of the half-tile complete (4 softmax warps)
  uint64_t *q_full = bars + 7;    //     Q in shared memory (6 warps)
  uint64_t *drain = bars + 8;     // [2] per-issuer wind-down
  uint64_t *drain_sm = bars + 10; // [4] per-softmax-warp wind-down
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + kNumBars);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tslot + 1);
  float *m_ref = reinterpret_cast<float *>(sm + kXOff);  // [2][64], log2 units
  float *xm = m_ref + 128;                              // [64 rows][4 warps]
  // epilogue only, in the idle P^T region
  float *xl = reinterpret_cast<float *>(sPT);                          // [64 rows][4 warps]
  long long *roff = reinterpret_cast<long long *>(sPT + 64 * 4 * 4);   // [64 rows]

  const int s = blockIdx.x / P.RT, rg = blockIdx.x % P.RT;
  const int r = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R0 = rg * kRowsN;

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(ptx::smem_u32(&full[b]), 1);
      ptx::mbar_init(ptx::smem_u32(&empty[b]), 4);
      ptx::mbar_init(ptx::smem_u32(&s_full[b]), 2);
      ptx::mbar_init(ptx::smem_u32(&drain[b]), 1);
    }
    for (int w = 0; w < 4; ++w) ptx::mbar_init(ptx::smem_u32(&drain_sm[w]), 1);
    ptx::mbar_init(ptx::smem_u32(o_done), 4);
    ptx::mbar_init(ptx::smem_u32(q_full), 6);
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
  // half-tiles: two per tile, less the last tile's second half when it lies
  // wholly past kv_len
  const int nh = ntiles <= 0 ? 0
                             : 2 * ntiles - ((sr.t1 - 1) * kKT + kHK >= sr.kv_len ? 1 : 0);
  auto kbase_of = [&](int h) { return (sr.t0 + (h >> 1)) * kKT + (h & 1) * kHK; };
  const uint32_t tm_s = tmem + kColS;
  const uint32_t tm_o = tmem + kColO;

  // ------------------------------------------------ Q -> smem, K-major SW128
  // The CTA's 64 query rows (token i, head h) = rows R0 .. R0 + 63 of the
  // request's [Tq * hq] rows are contiguous in q and in q_rope.  Warps 4-7
  // copy the latent part (64 x 64 16-byte units) and warps 0-1 the rope part
  // (64 x 8 units), each lane a strided run of units, all loads of a batch in
  // flight before the first store (a row per thread with a load-store pair
  // per unit costs one memory round trip per unit).
  if (nh > 0 && (warp >= 4 || warp < 2)) {
    const size_t q0 = static_cast<size_t>(r) * p.Tq * p.hq + R0;
    if (warp >= 4) {
      const int tid = threadIdx.x - 128;
      const uint4 *ql = reinterpret_cast<const uint4 *>(p.q + q0 * kLat);
      uint4 v[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const int g = tid + 128 * k;
        v[k] = R0 + (g >> 6) < P.GT ? ql[g] : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const int g = tid + 128 * k, row = g >> 6, u = g & 63;
        *reinterpret_cast<uint4 *>(sQ + (u >> 3) * kQChunkBytes + sw128_off(row, u & 7)) = v[k];
      }
    } else {
      const int tid = threadIdx.x;
      const uint4 *qr = reinterpret_cast<const uint4 *>(p.q_rope + q0 * (kWidth - kLat));
      uint4 v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int g = tid + 64 * k;
        v[k] = R0 + (g >> 3) < P.GT ? qr[g] : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int g = tid + 64 * k;
        *reinterpret_cast<uint4 *>(sQ + 8 * kQChunkBytes + sw128_off(g >> 3, g & 7)) = v[k];
      }
    }
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(q_full));
  }
  if ((nh > 0 || kScatter) && warp == 2) {
    // ------------------------------------------------ TMA producer (warp 2)
    // Fused block scatter: the producer warp first writes the block's latent
    // rows of this CTA's key range (every row group of the segment writes the
    // same bytes); the __syncwarp before the first copy orders every lane's
    // stores and proxy fence before it.
    if constexpr (kScatter)
      block_scatter_rows(block_scatter_args(p, sr), r, 0, sr, s == 0 && rg == 0, lane);
    // half-tile h goes to buffer h & 1 once both issuers' PV of h - 2 has
    // read it; its boxes (chunk x page box) are issued by different lanes
    const int bph = kHK / P.box_rows;        // boxes per chunk of a half-tile
    const int halves_per_batch = 32 / bph;   // page lookups fetched warp-wide
    auto fetch_page = [&](int h_batch) -> int {
      const int hh = h_batch + lane / bph, bx = lane % bph;
      int page = 0;
      if (hh < nh) {
        const int key0 = kbase_of(hh) + bx * P.box_rows;
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
    int nxt = fetch_page(halves_per_batch);
    int last_fill[2] = {-1, -1};
    bool ok = true;
    for (int h = 0; h < nh; ++h) {
      const int hb = h % halves_per_batch;
      if (hb == 0 && h > 0) {
        cur = nxt;
        nxt = fetch_page(h + halves_per_batch);
      }
      const int b = h & 1;
      bool got = true;
      if (lane == 0 && h >= 2)
        got = ptx::mbar_wait(ptx::smem_u32(&empty[b]), static_cast<uint32_t>(((h >> 1) - 1) & 1),
                             abort_flag);
      if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) {
        ok = false;
        break;
      }
      const bool skip = h == P.skip_h;
      if (lane == 0 && !skip) ptx::mbar_arrive_expect_tx(ptx::smem_u32(&full[b]), kBufBytes);
      __syncwarp();
      const int kbase = kbase_of(h);
      uint8_t *buf = sBuf + b * kBufBytes;
      const int nb = kChunks * bph;
      for (int j0 = 0; j0 < nb; j0 += 32) {
        const int jj = j0 + lane;
        const int c = (jj < nb ? jj : 0) / bph, bx = (jj < nb ? jj : 0) % bph;
        const int page = __shfl_sync(0xffffffffu, cur, hb * bph + bx);
        if (jj < nb && !skip) {
          const int key0 = kbase + bx * P.box_rows;
          const long long row0 = (static_cast<long long>(p.layer) * p.NP + page) * p.P + key0 % p.P;
          ptx::tma_load_2d(ptx::smem_u32(buf + c * kChunkBytes + bx * P.box_rows * 128), &tm,
                           c * 64, static_cast<int32_t>(row0), ptx::smem_u32(&full[b]));
        }
      }
      if (!skip) last_fill[b] = h;
    }
    if (!ok && lane == 0) {
      // let the copies in flight land before the CTA exits
      for (int b = 0; b < 2; ++b) {
        if (last_fill[b] < 0) continue;
        volatile int dummy = 0;
        ptx::mbar_wait(ptx::smem_u32(&full[b]), static_cast<uint32_t>((last_fill[b] >> 1) & 1),
                       &dummy);
      }
    }
  }
  if (nh > 0 && lane == 0 && (warp == 3 || warp == 0)) {
    // ------------------------------------------------ QK issuers
    // QK(h) = S^T of half-tile h once it has landed.  Issuer 0 (warp 3) runs
    // the first 18 of QK's 36 K-steps into one S^T partial, issuer 1 (warp 0,
    // after its Q rows) the other 18 into a second partial; the softmax adds
    // the two.  The S^T buffer QK(h) writes is free then: the copies of h
    // were issued only after PV(h - 2), which the softmax issues after it has
    // read S^T(h - 2).  Descriptors are formed once and advanced by adding
    // the byte offset (>> 4) to the address field.
    const int role = warp == 3 ? 0 : 1;
    constexpr int kQkSteps = kChunks * 4;
    const int ks_lo = role * (kQkSteps / 2), ks_hi = ks_lo + kQkSteps / 2;
    const uint64_t dq0 = ptx::desc_kmajor_sw128(ptx::smem_u32(sQ), 0);
    const uint64_t dk0 = ptx::desc_kmajor_sw128(ptx::smem_u32(sBuf), 0);
    bool ok = ptx::mbar_wait(ptx::smem_u32(q_full), 0u, abort_flag);
    for (int h = 0; ok && h < nh; ++h) {
      const int b = h & 1;
      ok = ptx::mbar_wait(ptx::smem_u32(&full[b]), static_cast<uint32_t>((h >> 1) & 1), abort_flag);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t d_s = tm_s + static_cast<uint32_t>((b * 2 + role) * kRowsN);
      const uint32_t boff = b * kBufBytes;
      for (int ks = ks_lo; ks < ks_hi; ++ks) {
        const int c = ks >> 2, j = ks & 3;
        ptx::mma_bf16(d_s, dk0 + ((boff + c * kChunkBytes + j * 32) >> 4),
                      dq0 + ((c * kQChunkBytes + j * 32) >> 4), P.idesc_qk,
                      ks > ks_lo ? 1u : 0u);
      }
      ptx::mma_commit(ptx::smem_u32(&s_full[b]));
    }
    if (!ok) {
      ptx::mma_commit(ptx::smem_u32(&drain[role]));
      volatile int dummy = 0;
      ptx::mbar_wait(ptx::smem_u32(&drain[role]), 0u, &dummy);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------ softmax (warps 4-7)
    // The M = 64 result puts key 16*q4 + l of the half-tile in TMEM lane
    // 32*q4 + l (l < 16); lanes 16-31 of each warp carry no key.  Lane l keeps
    // rows 0-31 of key 16*q4 + l and hands rows 32-63 to lane l + 16, so every
    // lane scores 32 rows of one key.
    const int q4 = warp & 3;
    const int hf = lane >> 4;               // this lane's rows: 32*hf .. 32*hf + 31
    const int key = 16 * q4 + (lane & 15);  // the half-tile key they belong to
    constexpr int kR = kRowsN / 2;
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    // PV: this warp's lane 0 applies P^T to O^T block q4 (dims 128*q4 ..
    // +127; A = the half-tile's latent rows read MN-major, B = P^T)
    const uint64_t dv0 = ptx::smem_desc(ptx::smem_u32(sBuf), kChunkBytes, 1024, ptx::kSwizzle128B);
    const uint64_t dp0 = ptx::smem_desc(ptx::smem_u32(sPT), kChunkBytes, 1024, ptx::kSwizzle128B);
    bool pv_issued = false;
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
    float lp[kR];
#pragma unroll
    for (int c = 0; c < kR; ++c) lp[c] = 0.f;
    bool bad = false;
    for (int h = 0; h < nh; ++h) {
      const bool got = __all_sync(0xffffffffu,
                                  ptx::mbar_wait(ptx::smem_u32(&s_full[h & 1]),
                                                 static_cast<uint32_t>((h >> 1) & 1), abort_flag));
      float sv[kR];
      if (got) {
        ptx::tc_fence_after();
        const uint32_t sa = tm_s + lane_off + (h & 1) * (2 * kRowsN);
        float sf[kRowsN];
        {
          float s2[32];
          ptx::tmem_ld64_ld32f_sync(sa, sa + kRowsN, sf, s2);
#pragma unroll
          for (int c = 0; c < 32; ++c) sf[c] += s2[c];
          ptx::tmem_ld32f_sync(sa + kRowsN + 32, s2);
#pragma unroll
          for (int c = 0; c < 32; ++c) sf[32 + c] += s2[c];
        }
#pragma unroll
        for (int c = 0; c < kR; ++c) {
          const float up = __shfl_sync(0xffffffffu, sf[kR + c], lane & 15);
          sv[c] = hf ? up : sf[c];
        }
      } else {
#pragma unroll
        for (int c = 0; c < kR; ++c) sv[c] = -INFINITY;
      }
      const int tile0 = kbase_of(h);
      const int kpos = tile0 + key;
      if (!(tile0 >= lo_max && tile0 + kHK - 1 <= hi_min)) {
        // a half-tile some row sees only in part (or past kv_len): mask per row
#pragma unroll
        for (int c = 0; c < kR; ++c) {
          const int R = R0 + kR * hf + c;
          const int i = R / p.hq;
          if (R > R_last || kpos < lo_of(i) || kpos > hi_of(i)) sv[c] = -INFINITY;
        }
      }
      const float *mr = m_ref + 64 * cur;  // all 64 rows
      const float *mrh = mr + kR * hf;    // this lane's rows
      bool need = false;
#pragma unroll
      for (int c4 = 0; c4 < kR / 4; ++c4) {
        const float4 m4 = *reinterpret_cast<const float4 *>(mrh + 4 * c4);
        need |= sv[4 * c4] * P.scale_log2 > m4.x + 8.f;
        need |= sv[4 * c4 + 1] * P.scale_log2 > m4.y + 8.f;
        need |= sv[4 * c4 + 2] * P.scale_log2 > m4.z + 8.f;
        need |= sv[4 * c4 + 3] * P.scale_log2 > m4.w + 8.f;
      }
      // PV of the previous half-tile must be done before O^T is rescaled and
      // before the single P^T buffer is rewritten: the rebuild waits for it
      // first, the common path only before it stores P
      bool o_seen = h == 0;
      if (ptx::bar_or(2, 128, need || !got || bad)) {
        if (ptx::bar_or(3, 128, !got || bad)) {
          bad = true;
          break;
        }
        const bool got_o =
            o_seen || __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(o_done),
                                                             static_cast<uint32_t>((h - 1) & 1),
                                                             abort_flag));
        if (ptx::bar_or(3, 128, !got_o)) {
          bad = true;
          break;
        }
        o_seen = true;
        // ---- rebuild m_ref: exact half-tile maxima, rescale O^T and the row sums
        ptx::tc_fence_after();
        {
          float mx[kR];
#pragma unroll
          for (int c = 0; c < kR; ++c) mx[c] = sv[c];
          half_warp_transpose_reduce32<true>(mx, lane);
          const int row0 = kR * hf + 2 * (lane & 15);
          xm[row0 * 4 + q4] = mx[0];
          xm[(row0 + 1) * 4 + q4] = mx[1];
        }
        ptx::bar_sync(2, 128);
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
        for (int c = 0; c < kR; ++c) {
          const float old = mr[kR * hf + c], nw = mn[kR * hf + c];
          lp[c] *= (old == -INFINITY || old == nw) ? 1.f : ptx::ex2(old - nw);
        }
        if (h > 0) {
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
      // P = exp2(s - m_ref) in place (row sums as it goes), then -> units
      // 4*hf .. 4*hf+3 of P^T row `key` (64 rows = 8 units of 8) once the
      // previous PV is done
      {
        const float *m2 = m_ref + 64 * cur + kR * hf;
#pragma unroll
        for (int c4 = 0; c4 < kR / 4; ++c4) {
          const float4 m4 = *reinterpret_cast<const float4 *>(m2 + 4 * c4);
          const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = 4 * c4 + e;
            sv[c] = sv[c] == -INFINITY ? 0.f : ptx::ex2(fmaf(sv[c], P.scale_log2, -mm[e]));
            lp[c] += sv[c];
          }
        }
      }
      const bool got_o =
          o_seen || __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(o_done),
                                                           static_cast<uint32_t>((h - 1) & 1),
                                                           abort_flag));
      if (got_o) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            pk[e] = ptx::pack_bf16x2(sv[8 * u + 2 * e], sv[8 * u + 2 * e + 1]);
          *reinterpret_cast<uint4 *>(sPT + sw128_off(key, 4 * hf + u)) =
              make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        ptx::fence_proxy_async_smem();
      }
      ptx::tc_fence_before();
      // every warp's P^T rows are in place (or all four wind down together)
      if (ptx::bar_or(3, 128, !got_o)) {
        bad = true;
        break;
      }
      if (lane == 0) {
        ptx::tc_fence_after();
        const uint32_t boff = (h & 1) * kBufBytes;
#pragma unroll
        for (int ks = 0; ks < kHK / 16; ++ks)
          ptx::mma_bf16(tm_o + q4 * kRowsN, dv0 + ((boff + 2 * q4 * kChunkBytes + ks * 2048) >> 4),
                        dp0 + ((ks * 2048) >> 4), P.idesc_pv, (h > 0 || ks > 0) ? 1u : 0u);
        ptx::mma_commit(ptx::smem_u32(&empty[h & 1]));
        ptx::mma_commit(ptx::smem_u32(o_done));
      }
      __syncwarp();
      pv_issued = true;
    }
    // ---- epilogue: row sums over the keys, then (m, l, O) per real row
    bool okf = !bad && nh > 0;
    if (okf) {
      okf = __all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_u32(o_done),
                                                   static_cast<uint32_t>((nh - 1) & 1),
                                                   abort_flag));
      ptx::tc_fence_after();
    }
    if (!okf && pv_issued && lane == 0) {
      // winding down: this warp's PV MMAs finish before TMEM is released
      ptx::mma_commit(ptx::smem_u32(&drain_sm[q4]));
      volatile int dummy = 0;
      ptx::mbar_wait(ptx::smem_u32(&drain_sm[q4]), 0u, &dummy);
    }
    __syncwarp();
    const bool any_bad = ptx::bar_or(2, 128, !okf && nh > 0);
    // the P^T region is idle from here (the last PV is done, or the CTA is
    // winding down and writes no partial)
    half_warp_transpose_reduce32<false>(lp, lane);
    if (!any_bad) {
      const int row0 = kR * hf + 2 * (lane & 15);
      xl[row0 * 4 + q4] = lp[0];
      xl[(row0 + 1) * 4 + q4] = lp[1];
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
    }
    ptx::bar_sync(2, 128);
    const float *mf = m_ref + 64 * cur;
    if (q4 < 2) {
      const int c = 32 * q4 + lane;
      const int R = R0 + c;
      if (R < P.GT) {
        const int i = R / p.hq, h = R % p.hq;
        const long long wsi =
            static_cast<long long>(((static_cast<size_t>(r) * p.Tq + i) * p.hq + h) * p.S + s);
        const bool any = !any_bad && nh > 0 && mf[c] != -INFINITY;
        float l = 0.f;
        if (any) {
          const float4 l4 = *reinterpret_cast<const float4 *>(xl + c * 4);
          l = (l4.x + l4.y) + (l4.z + l4.w);
        }
        p.ws_m[wsi] = any ? mf[c] * kLn2 : -INFINITY;
        p.ws_l[wsi] = l;
      }
    }
    if (!any_bad && nh > 0) {
      // O^T (dims in lanes) -> O rows in the idle half-tile buffers [64 rows][512]
      // (bank-conflict-free: a warp writes 32 consecutive dims of one row);
      // then each of 64 threads sends one 2 KB row to the workspace with a
      // bulk copy (the copy engine writes whole lines; per-thread 16-byte
      // stores of all 152 CTAs at once ran at ~3.7 TB/s)
      float *stage = reinterpret_cast<float *>(sBuf);
      for (int b = 0; b < 4; ++b) {
        const int d = b * 128 + 32 * q4 + lane;
        float ov[kRowsN];
        ptx::tmem_ld64f_sync(tm_o + lane_off + b * kRowsN, ov);
#pragma unroll
        for (int c = 0; c < kRowsN; ++c) stage[c * kLat + d] = ov[c];
      }
      ptx::fence_proxy_async_smem();
      ptx::bar_sync(2, 128);
      if (q4 < 2) {
        const int c = 32 * q4 + lane;
        const long long wsi = roff[c];
        if (wsi >= 0 && mf[c] != -INFINITY) {
          ptx::bulk_store_s2g(p.ws_o + wsi * kLat, ptx::smem_u32(stage + c * kLat), kLat * 4);
          ptx::bulk_commit_wait_all();
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

}  // namespace

int mla_rows_per_cta() { return kRowsN; }

cudaError_t launch_attn_mla_tc(const AttnParams &a, const dflash_geom &g, cudaStream_t s) {
  MlaParams P;
  P.a = a;
  P.GT = a.Tq * a.hq;
  P.RT = (P.GT + kRowsN - 1) / kRowsN;
  P.box_rows = a.P < kHK ? a.P : kHK;
  const int skip_tile = attention_test_skip_tile_value();
  P.skip_h = skip_tile >= 0 ? 2 * skip_tile : -1;
  P.idesc_qk = ptx::idesc_bf16_f32(kHK, kRowsN, false, false);
  P.idesc_pv = ptx::idesc_bf16_f32(128, kRowsN, true, true);
  P.scale_log2 = a.scale * 1.4426950408889634f;
  CUtensorMap tm;
  const uint64_t rows = static_cast<uint64_t>(g.num_layers) * g.num_pool_pages *
                        static_cast<uint64_t>(g.page_size);
  cudaError_t e = make_tmap_bf16_2d(&tm, a.pool, rows, kWidth, kWidth, P.box_rows, 64);
  if (e != cudaSuccess) return e;
  if ((e = ensure_smem_limit<attn_mla_tc_kernel<false>>(227 * 1024)) != cudaSuccess) return e;
  if ((e = ensure_smem_limit<attn_mla_tc_kernel<true>>(227 * 1024)) != cudaSuccess) return e;
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
  return a.blk_k != nullptr ? cudaLaunchKernelEx(&cfg, attn_mla_tc_kernel<true>, tm, P)
                            : cudaLaunchKernelEx(&cfg, attn_mla_tc_kernel<false>, tm, P);
}

}  // namespace dflash
