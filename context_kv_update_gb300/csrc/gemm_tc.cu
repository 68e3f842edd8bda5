// gemm_tc.cu -- stream-K tcgen05 GEMM for the weight-bound context projection
// (fc, then the K/V or latent projection stacked over every drafter layer,
// TensorRT-LLM PR #13995 "migrate draft path to per-layer cached K/V pool").
//
// CTA = 6 warps: warp 0 issues TMA loads (one elected lane), warp 1 issues
// tcgen05.mma (one lane), warps 2-5 drain the TMEM accumulator (warp w reads
// TMEM lanes 32*(w%4)..+31) and write fp32 partial tiles.  A ring of `stages`
// shared-memory slots, each one 128x64 weight tile + one NTILEx64 activation
// tile, is guarded by full/empty mbarriers; two TMEM accumulators by
// acc_full / acc_empty, so the next tile's MMAs overlap the last one's drain.
// Every wait is bounded (ptx::mbar_wait) so a broken pipeline winds the
// kernel down instead of hanging it.
#include "gemm_tc.cuh"

#include <algorithm>
#include <mutex>

namespace dflash {
namespace {

constexpr int kThreads = 192;
constexpr int kMaxSmem = 227 * 1024;
// Ring depth cap.  The weight tiles of the first ring slots (up to 6) are
// copied before the dependency wait, and the rest of the ring refills as the
// MMAs drain it.
constexpr int kMaxStages = 12;

struct GemmParams {
  int K, ntile, mtiles, kblocks, maxc, stages;
  long long units;
  float *part;  // [tiles][maxc][ntile][128]
  uint32_t idesc;
  uint32_t tmem_cols;
  int acc_cols;  // TMEM columns per accumulator buffer
  int pdl_wait;
  int32_t *status;
};

__host__ __device__ inline uint32_t a_tile_bytes() { return 128u * 64u * 2u; }
__host__ __device__ inline uint32_t b_tile_bytes(int ntile) { return static_cast<uint32_t>(ntile) * 128u; }

__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const int S = p.stages;
  const uint32_t abytes = a_tile_bytes(), bbytes = b_tile_bytes(p.ntile);
  uint8_t *sA = smem;
  uint8_t *sB = sA + S * abytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sB + S * bbytes);
  // two accumulator buffers: the MMA fills one while the epilogue drains the other
  uint64_t *full = bars, *empty = bars + S, *acc_full = bars + 2 * S, *acc_empty = bars + 2 * S + 2;
  uint64_t *drain = bars + 2 * S + 4;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * S + 5);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *consumed = reinterpret_cast<int *>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(ptx::smem_u32(&full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(ptx::smem_u32(&acc_full[b]), 1);
      ptx::mbar_init(ptx::smem_u32(&acc_empty[b]), 4);
    }
    ptx::mbar_init(ptx::smem_u32(drain), 1);
    *abort_flag = 0;
    *consumed = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tmW);
    ptx::prefetch_tmap(&tmX);
  }
  if (warp == 2) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), p.tmem_cols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // The next kernel of the chain only prefetches what does not depend on this
  // one and then waits for this grid to complete, so it may launch now.
  griddep_launch();

  const long long C = gridDim.x, c = blockIdx.x, U = p.units, KB = p.kblocks;
  const long long u_lo = c * U / C, u_hi = (c + 1) * U / C;
  const long long t_first = u_lo / KB, t_last = (u_hi - 1) / KB;

  if (warp == 0) {
    // ---------------- TMA producer (warp 0)
    // (t, kb, m, nt) and (stage, phase) advance incrementally: no divisions
    // in the loop.  Lane 0 waits for free slots and arms the barriers; the
    // two copies of unit i are issued by lanes 2(i%16) and 2(i%16)+1, since
    // copies issued by one thread complete one after another.
    const uint64_t pol_w = ptx::policy_evict_first();
    struct Cursor {
      long long t;
      int kb, m, nt;
    };
    const Cursor start{t_first, static_cast<int>(u_lo - t_first * KB),
                       static_cast<int>(t_first % p.mtiles), static_cast<int>(t_first / p.mtiles)};
    auto advance = [&](Cursor &q) {
      if (++q.kb == p.kblocks) {
        q.kb = 0;
        ++q.t;
        if (++q.m == p.mtiles) {
          q.m = 0;
          ++q.nt;
        }
      }
    };
    const int total = static_cast<int>(u_hi - u_lo);
    // at most kPreWait slots before the dependency wait: a deeper burst slows
    // the preceding kernels' memory traffic more than it saves (decode step:
    // 6 slots 190.0 us, the whole 12-slot ring 190.55 us, A/B on one box)
    constexpr int kPreWait = 6;
    const int pre = std::min(std::min(S, kPreWait), total);
    bool ok = true;
    // Prologue: weight tiles of the first ring slots do not depend on the
    // previous kernel, so they are in flight before the dependency wait.
    Cursor q = start;
    if (lane == 0)
      for (int i = 0; i < pre; ++i)
        ptx::mbar_arrive_expect_tx(ptx::smem_u32(&full[i]), abytes + bbytes);
    __syncwarp();
    for (int i = 0; i < pre; ++i, advance(q))
      if (lane == 2 * (i & 15))
        ptx::tma_load_2d_hint(ptx::smem_u32(sA + i * abytes), &tmW, q.kb * 64, q.m * 128,
                              ptx::smem_u32(&full[i]), pol_w);
    if (p.pdl_wait) griddep_wait();
    q = start;
    for (int i = 0; i < pre; ++i, advance(q))
      if (lane == 2 * (i & 15) + 1)
        ptx::tma_load_2d(ptx::smem_u32(sB + i * bbytes), &tmX, q.kb * 64, q.nt * p.ntile,
                         ptx::smem_u32(&full[i]));
    int issued = pre;
    int st = pre % S;
    uint32_t ph = (pre / S) & 1;
    for (int i = pre; i < total; ++i, advance(q)) {
      bool got = true;
      if (lane == 0) got = ptx::mbar_spin(ptx::smem_u32(&empty[st]), ph ^ 1u, abort_flag);
      if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) {
        ok = false;
        break;
      }
      if (lane == 0) ptx::mbar_arrive_expect_tx(ptx::smem_u32(&full[st]), abytes + bbytes);
      __syncwarp();
      if (lane == 2 * (i & 15))
        ptx::tma_load_2d_hint(ptx::smem_u32(sA + st * abytes), &tmW, q.kb * 64, q.m * 128,
                              ptx::smem_u32(&full[st]), pol_w);
      if (lane == 2 * (i & 15) + 1)
        ptx::tma_load_2d(ptx::smem_u32(sB + st * bbytes), &tmX, q.kb * 64, q.nt * p.ntile,
                         ptx::smem_u32(&full[st]));
      ++issued;
      if (++st == S) {
        st = 0;
        ph ^= 1u;
      }
    }
    if (!ok && lane == 0) {
      // wind down: let the copies already issued land before the CTA exits
      for (int it = *reinterpret_cast<volatile int *>(consumed); it < issued; ++it) {
        volatile int dummy = 0;
        ptx::mbar_wait(ptx::smem_u32(&full[it % S]), static_cast<uint32_t>((it / S) & 1), &dummy);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      int it = 0, s = 0;
      uint32_t ph = 0;
      int tile_i = 0;
      bool ok = true;
      for (long long t = t_first; t <= t_last && ok; ++t, ++tile_i) {
        const long long ua = std::max(u_lo, t * KB), ub = std::min(u_hi, (t + 1) * KB);
        const int ab = tile_i & 1;
        const uint32_t acc = tmem + static_cast<uint32_t>(ab * p.acc_cols);
        if (!ptx::mbar_spin(ptx::smem_u32(&acc_empty[ab]),
                            static_cast<uint32_t>((tile_i >> 1) & 1) ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        for (long long u = ua; u < ub; ++u, ++it) {
          if (!ptx::mbar_spin(ptx::smem_u32(&full[s]), ph, abort_flag)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t a_base = ptx::smem_u32(sA + s * abytes);
          const uint32_t b_base = ptx::smem_u32(sB + s * bbytes);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            ptx::mma_bf16(acc, ptx::desc_kmajor_sw128(a_base, k), ptx::desc_kmajor_sw128(b_base, k),
                          p.idesc, (u > ua || k > 0) ? 1u : 0u);
          }
          ptx::mma_commit(ptx::smem_u32(&empty[s]));
          *reinterpret_cast<volatile int *>(consumed) = it + 1;
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit(ptx::smem_u32(&acc_full[ab]));
      }
      if (!ok) {
        // make sure no MMA is still reading shared memory / writing TMEM
        ptx::mma_commit(ptx::smem_u32(drain));
        volatile int dummy = 0;
        ptx::mbar_wait(ptx::smem_u32(drain), 0u, &dummy);
      }
    }
  } else {
    // ---------------- epilogue: TMEM -> this CTA's partial of each tile
    // Tile t's partial j = c - c0(t) holds this CTA's K range of the tile;
    // the reader adds the partials in CTA order.
    const int q = warp & 3;
    const int row = q * 32 + lane;
    int tile_i = 0;
    for (long long t = t_first; t <= t_last; ++t, ++tile_i) {
      const int ab = tile_i & 1;
      const uint32_t acc = tmem + static_cast<uint32_t>(ab * p.acc_cols);
      const bool got = ptx::mbar_wait(ptx::smem_u32(&acc_full[ab]),
                                      static_cast<uint32_t>((tile_i >> 1) & 1), abort_flag);
      if (ptx::bar_or(1, 128, !got)) break;  // the 4 epilogue warps leave together
      ptx::tc_fence_after();
      const long long c0 = ((t * KB + 1) * C - 1) / U;
      // c - c0 < maxc by the schedule's bound; checked so that a wrong bound
      // can never write outside the partial buffer
      const bool in = c - c0 < p.maxc;
      float *dst = p.part + ((t * p.maxc + (c - c0)) * p.ntile) * 128 + row;
      for (int n0 = 0; n0 < p.ntile; n0 += 16) {
        uint32_t r[16];
        ptx::tmem_ld16_sync(acc + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(n0),
                            r);
        if (in) {
#pragma unroll
          for (int j = 0; j < 16; ++j) dst[static_cast<size_t>(n0 + j) * 128] = __uint_as_float(r[j]);
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&acc_empty[ab]));
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) raise_status(p.status, DFLASH_DEV_WAIT_TIMEOUT);
  if (warp == 2) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, p.tmem_cols);
  }
}

// ------------------------------------------------------------ fc as cluster split-K
// Y = X W^T for decode row counts (up to 64 rows), each 128-feature output
// tile computed by a cluster of kFcCluster CTAs that split its K range; the
// CTAs add their accumulators through distributed shared memory (rank order,
// deterministic) and CTA k of the cluster finishes features 32k .. 32k + 31:
// it writes h = bf16(Y) and, per row, the sum of h^2 over those 32 features.
// Each CTA pushes every quarter of its accumulator straight into the shared
// memory of the quarter's owner, so one cluster barrier separates the pushes
// from the local sums and no CTA reads another's memory afterwards.
// No partial tiles leave the cluster, so the consumer (the hidden RMSNorm)
// reads one bf16 value per element instead of adding fp32 partials.
constexpr int kFcCluster = 4;

struct FcParams {
  int ntile;   // rows (Npad: 16 .. 64, a multiple of 16)
  int kb_per;  // 64-deep K blocks per CTA
  int stages;
  int M;       // output features (row stride of h)
  uint32_t idesc, tmem_cols;
  uint16_t *h;  // [ntile][M] bf16
  float *ssq;   // [M / 128 * kFcCluster][ntile]
  int32_t *status;
  int setup_rows;  // rows whose set-up warp 2 of CTA n runs (0: none)
  RowDest rd;
  RopeFreqs rf;
};

__global__ void __launch_bounds__(kThreads, 1)
    fc_cluster_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                      const FcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const int S = p.stages;
  const uint32_t abytes = a_tile_bytes(), bbytes = b_tile_bytes(p.ntile);
  uint8_t *sA = smem;
  uint8_t *sB = sA + S * abytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sB + S * bbytes);
  uint64_t *full = bars, *empty = bars + S, *acc_full = bars + 2 * S, *drain = bars + 2 * S + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * S + 2);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *consumed = reinterpret_cast<int *>(tmem_slot + 2);
  // this CTA's 32 features of the tile as pushed by every CTA of the cluster:
  // [kFcCluster source ranks][ntile rows][32] fp32, outside the ring
  float *red_in = reinterpret_cast<float *>(
      smem + ((reinterpret_cast<uintptr_t>(tmem_slot + 4) - reinterpret_cast<uintptr_t>(smem) + 15) &
              ~static_cast<uintptr_t>(15)));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = blockIdx.x / kFcCluster, rank = blockIdx.x % kFcCluster;
  const int kb0 = rank * p.kb_per;
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      ptx::mbar_init(ptx::smem_u32(&full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&empty[i]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(acc_full), 1);
    ptx::mbar_init(ptx::smem_u32(drain), 1);
    *abort_flag = 0;
    *consumed = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tmW);
    ptx::prefetch_tmap(&tmX);
  }
  if (warp == 2) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), p.tmem_cols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_launch();

  if (warp == 0) {
    // ---------------- TMA producer: the weight tiles of the first kFcPreWait
    // ring slots before the dependency wait, the activations after it.  All
    // 128 CTAs start together at the head of the step; a deep burst of weight
    // requests there delays the preceding small kernel's own memory traffic
    // and with it the release (3 slots: step 190.6 -> 189.2 us against 12).
    constexpr int kFcPreWait = 3;
    const uint64_t pol_w = ptx::policy_evict_first();
    const int total = p.kb_per, pre = total < kFcPreWait ? total : (S < kFcPreWait ? S : kFcPreWait);
    if (lane == 0)
      for (int i = 0; i < pre; ++i)
        ptx::mbar_arrive_expect_tx(ptx::smem_u32(&full[i]), abytes + bbytes);
    __syncwarp();
    for (int i = 0; i < pre; ++i)
      if (lane == 2 * (i & 15))
        ptx::tma_load_2d_hint(ptx::smem_u32(sA + i * abytes), &tmW, (kb0 + i) * 64, mt * 128,
                              ptx::smem_u32(&full[i]), pol_w);
    griddep_wait();
    for (int i = 0; i < pre; ++i)
      if (lane == 2 * (i & 15) + 1)
        ptx::tma_load_2d(ptx::smem_u32(sB + i * bbytes), &tmX, (kb0 + i) * 64, 0,
                         ptx::smem_u32(&full[i]));
    bool ok = true;
    int issued = pre;
    for (int i = pre; i < total; ++i) {
      const int st = i % S;
      const uint32_t ph = static_cast<uint32_t>((i / S) & 1);
      bool got = true;
      if (lane == 0) got = ptx::mbar_spin(ptx::smem_u32(&empty[st]), ph ^ 1u, abort_flag);
      if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) {
        ok = false;
        break;
      }
      if (lane == 0) ptx::mbar_arrive_expect_tx(ptx::smem_u32(&full[st]), abytes + bbytes);
      __syncwarp();
      if (lane == 2 * (i & 15))
        ptx::tma_load_2d_hint(ptx::smem_u32(sA + st * abytes), &tmW, (kb0 + i) * 64, mt * 128,
                              ptx::smem_u32(&full[st]), pol_w);
      if (lane == 2 * (i & 15) + 1)
        ptx::tma_load_2d(ptx::smem_u32(sB + st * bbytes), &tmX, (kb0 + i) * 64, 0,
                         ptx::smem_u32(&full[st]));
      ++issued;
    }
    if (!ok && lane == 0) {
      // wind down: let the copies already issued land before the CTA exits
      for (int it = *reinterpret_cast<volatile int *>(consumed); it < issued; ++it) {
        volatile int dummy = 0;
        ptx::mbar_wait(ptx::smem_u32(&full[it % S]), static_cast<uint32_t>((it / S) & 1), &dummy);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer: the CTA's K range into one accumulator
      bool ok = true;
      for (int i = 0; i < p.kb_per && ok; ++i) {
        const int st = i % S;
        ok = ptx::mbar_spin(ptx::smem_u32(&full[st]), static_cast<uint32_t>((i / S) & 1),
                            abort_flag);
        if (!ok) break;
        ptx::tc_fence_after();
        const uint32_t a_base = ptx::smem_u32(sA + st * abytes);
        const uint32_t b_base = ptx::smem_u32(sB + st * bbytes);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          ptx::mma_bf16(tmem, ptx::desc_kmajor_sw128(a_base, k), ptx::desc_kmajor_sw128(b_base, k),
                        p.idesc, (i > 0 || k > 0) ? 1u : 0u);
        ptx::mma_commit(ptx::smem_u32(&empty[st]));
        *reinterpret_cast<volatile int *>(consumed) = i + 1;
      }
      ptx::mma_commit(ptx::smem_u32(ok ? acc_full : drain));
      if (!ok) {
        volatile int dummy = 0;
        ptx::mbar_wait(ptx::smem_u32(drain), 0u, &dummy);
      }
    }
  } else {
    // ---------------- the epilogue's row set-up, while the weights stream
    if (warp == 2 && static_cast<int>(blockIdx.x) < p.setup_rows) {
      griddep_wait();  // it reads the call's index inputs
      row_setup_warp(p.rd, p.rf, blockIdx.x, lane);
    }
    // ---------------- accumulator quarter q (TMEM lanes, i.e. features,
    // 32q .. +31) -> red_in[rank][row][feature - 32q] of cluster CTA q
    // (consecutive lanes write consecutive words)
    const int q = warp & 3;
    const bool got = ptx::mbar_wait(ptx::smem_u32(acc_full), 0u, abort_flag);
    if (__all_sync(0xffffffffu, got)) {
      ptx::tc_fence_after();
      for (int n0 = 0; n0 < p.ntile; n0 += 16) {
        uint32_t r[16];
        ptx::tmem_ld16_sync(tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(n0),
                            r);
#pragma unroll
        for (int j = 0; j < 16; ++j)
          ptx::st_dsmem_f32(red_in + (rank * p.ntile + n0 + j) * 32 + lane, static_cast<uint32_t>(q),
                            __uint_as_float(r[j]));
      }
    }
  }
  ptx::tc_fence_before();
  // every quarter is in its owner's shared memory (an aborted CTA pushes
  // nothing and leaves garbage; its status flag reports the timeout)
  ptx::cluster_sync();
  if (warp >= 2) {
    // ---------------- features 32*rank .. +31 of the tile, added over the
    // cluster in rank order: tpr threads a row, fpt features each
    const int t = threadIdx.x - 64;
    const int tpr = 128 / p.ntile, fpt = 32 / tpr;
    const int n = t / tpr, part = t % tpr;
    const int f0 = 32 * rank + part * fpt;
    float ss = 0.f;
    for (int j0 = 0; j0 < fpt; j0 += 4) {
      float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int c = 0; c < kFcCluster; ++c) {
        const float4 v =
            *reinterpret_cast<const float4 *>(red_in + (c * p.ntile + n) * 32 + part * fpt + j0);
        y.x += v.x;
        y.y += v.y;
        y.z += v.z;
        y.w += v.w;
      }
      const uint32_t lo = ptx::pack_bf16x2(y.x, y.y), hi = ptx::pack_bf16x2(y.z, y.w);
      const float hx = __uint_as_float(lo << 16), hy = __uint_as_float(lo & 0xffff0000u);
      const float hz = __uint_as_float(hi << 16), hw = __uint_as_float(hi & 0xffff0000u);
      ss += (hx * hx + hy * hy) + (hz * hz + hw * hw);
      *reinterpret_cast<uint2 *>(p.h + static_cast<size_t>(n) * p.M + mt * 128 + f0 + j0) =
          make_uint2(lo, hi);
    }
    for (int o = 1; o < tpr; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (part == 0) p.ssq[(mt * kFcCluster + rank) * p.ntile + n] = ss;
  }
  if (*abort_flag && threadIdx.x == 0) raise_status(p.status, DFLASH_DEV_WAIT_TIMEOUT);
  if (warp == 2) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, p.tmem_cols);
  }
}

// ------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct Schedule {
  int ntile, nt, mtiles, kblocks, ctas, maxc, stages;
  long long units;
};

Schedule make_schedule(int M, int K, int Npad) {
  Schedule s;
  s.ntile = Npad <= 256 ? Npad : 256;
  s.nt = (Npad + s.ntile - 1) / s.ntile;
  s.mtiles = (M + 127) / 128;
  s.kblocks = (K + 63) / 64;
  s.units = static_cast<long long>(s.nt) * s.mtiles * s.kblocks;
  // one CTA per SM
  s.ctas = static_cast<int>(std::min<long long>(s.units, device_sm_count()));
  // CTAs sharing one tile: every CTA holds at least q = floor(units / ctas)
  // units, so at most floor(kblocks / q) lie inside the tile's kblocks units,
  // plus one overlapping each end
  const long long q = s.units / s.ctas;
  s.maxc = static_cast<int>(std::min<long long>({s.ctas, s.kblocks, s.kblocks / q + 2}));
  const int stage_bytes = static_cast<int>(a_tile_bytes() + b_tile_bytes(s.ntile));
  s.stages = std::min(kMaxStages, (kMaxSmem - 2048) / stage_bytes);
  return s;
}

}  // namespace

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D bf16 tensor map over a row-major [rows, cols] matrix with a
// box of box_rows x 64 columns and 128-byte swizzle.
cudaError_t make_tmap_bf16_2d(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols,
                              uint64_t row_stride_elems, uint32_t box_rows, uint32_t box_cols) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_stride_elems * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

size_t gemm_partial_bytes(int M, int K, int Npad) {
  const Schedule s = make_schedule(M, K, Npad);
  return static_cast<size_t>(s.nt) * s.mtiles * s.maxc * s.ntile * 128 * sizeof(float);
}

cudaError_t launch_gemm(const uint16_t *X, int N, int K, const uint16_t *W, int M, float *part,
                        int32_t *status, bool pdl, cudaStream_t st, GemmOut *out) {
  const int Npad = static_cast<int>(align_up(static_cast<size_t>(N), 16));
  const Schedule s = make_schedule(M, K, Npad);
  if (s.units * s.ctas >= (1ll << 32)) return cudaErrorInvalidValue;
  CUtensorMap tmW, tmX;
  cudaError_t e;
  if ((e = make_tmap_bf16_2d(&tmW, W, M, K, K, 128, 64)) != cudaSuccess) return e;
  if ((e = make_tmap_bf16_2d(&tmX, X, N, K, K, s.ntile, 64)) != cudaSuccess) return e;

  GemmParams p;
  p.K = K;
  p.ntile = s.ntile;
  p.mtiles = s.mtiles;
  p.kblocks = s.kblocks;
  p.maxc = s.maxc;
  p.stages = s.stages;
  p.units = s.units;
  p.part = part;
  p.idesc = ptx::idesc_bf16_f32(128, s.ntile);
  uint32_t cols = 32;
  while (cols < static_cast<uint32_t>(s.ntile)) cols <<= 1;
  p.acc_cols = static_cast<int>(cols);
  p.tmem_cols = 2 * cols;
  p.pdl_wait = 1;
  p.status = status;

  const size_t smem = 1024 + static_cast<size_t>(s.stages) * (a_tile_bytes() + b_tile_bytes(s.ntile)) +
                      (2 * s.stages + 5) * 8 + 32;
  if ((e = ensure_smem_limit<gemm_tc_kernel>(kMaxSmem)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(s.ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  out->part = part;
  out->units = static_cast<unsigned>(s.units);
  out->ctas = s.ctas;
  out->kblocks = s.kblocks;
  out->mtiles = s.mtiles;
  out->maxc = s.maxc;
  out->ntile = s.ntile;
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel, tmW, tmX, p);
}


namespace {
// Clusters of kFcCluster fc CTAs (one per SM at this shared memory) that fit
// at once on the current device, cached per device and ring depth.
int fc_max_active_clusters(size_t smem) {
  static std::mutex mu;
  static int cache[64][16];  // [device][stages]: count + 1, 0 = not asked yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int key = static_cast<int>(smem / (16 * 1024)) & 15;
  std::lock_guard<std::mutex> lock(mu);
  int &slot = cache[dev][key];
  if (slot > 0) return slot - 1;
  int n = 0;
  if (ensure_smem_limit<fc_cluster_kernel>(kMaxSmem) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(kFcCluster);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kFcCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, fc_cluster_kernel, &cfg) != cudaSuccess) n = 0;
  }
  (void)cudaGetLastError();  // a refused query leaves no sticky error behind
  slot = n + 1;
  return n;
}

struct FcShape {
  int ntile, kb_per, stages, mtiles;
  size_t smem;
};
FcShape fc_shape(int N, int K, int M) {
  FcShape f;
  f.ntile = N <= 16 ? 16 : (N <= 32 ? 32 : 64);  // divides 128: whole rows per reducing thread group
  f.mtiles = M / 128;
  f.kb_per = K / 64 / kFcCluster;
  const int stage_bytes = static_cast<int>(a_tile_bytes() + b_tile_bytes(f.ntile));
  const int red_bytes = kFcCluster * f.ntile * 32 * 4;  // the pushed quarters
  f.stages = std::min({kMaxStages, f.kb_per, (kMaxSmem - 2048 - red_bytes) / stage_bytes});
  f.smem = 1024 + static_cast<size_t>(f.stages) * stage_bytes + (2 * f.stages + 2) * 8 + 32 +
           red_bytes;
  return f;
}
}  // namespace

bool fc_cluster_ok(int N, int K, int M) {
  if (N < 1 || N > 64 || M % 128 != 0 || K % (64 * kFcCluster) != 0) return false;
  const FcShape f = fc_shape(N, K, M);
  return f.stages >= 2 && f.smem <= static_cast<size_t>(kMaxSmem) &&
         fc_max_active_clusters(f.smem) >= f.mtiles;
}

int fc_cluster_rows(int N) { return fc_shape(N, 256, 128).ntile; }

cudaError_t launch_fc_cluster(const uint16_t *X, int N, int K, const uint16_t *W, int M,
                              uint16_t *h, float *ssq, int32_t *status, cudaStream_t st,
                              const RowDest *rd, const RopeFreqs *rf) {
  const FcShape f = fc_shape(N, K, M);
  CUtensorMap tmW, tmX;
  cudaError_t e;
  if ((e = make_tmap_bf16_2d(&tmW, W, M, K, K, 128, 64)) != cudaSuccess) return e;
  if ((e = make_tmap_bf16_2d(&tmX, X, N, K, K, f.ntile, 64)) != cudaSuccess) return e;
  FcParams p;
  p.ntile = f.ntile;
  p.kb_per = f.kb_per;
  p.stages = f.stages;
  p.M = M;
  p.idesc = ptx::idesc_bf16_f32(128, f.ntile);
  p.tmem_cols = f.ntile <= 32 ? 32u : 64u;
  p.h = h;
  p.ssq = ssq;
  p.status = status;
  p.setup_rows = 0;
  if (rd && rf && rd->dst && N <= f.mtiles * kFcCluster) {
    p.setup_rows = N;
    p.rd = *rd;
    p.rf = *rf;
  }
  if ((e = ensure_smem_limit<fc_cluster_kernel>(kMaxSmem)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  cfg.gridDim = dim3(f.mtiles * kFcCluster);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = f.smem;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kFcCluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, fc_cluster_kernel, tmW, tmX, p);
}

}  // namespace dflash
