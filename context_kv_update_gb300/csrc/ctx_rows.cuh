// ctx_rows.cuh -- which pool row a context-update row goes to: the write
// rule, the allocation clamp and the page lookup of the accepted rows, and
// the per-row set-up (destination and RoPE cos/sin) the epilogues can read
// instead of resolving it per head.
#pragma once

#include "dflash_internal.cuh"

namespace dflash {

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

// Destination of each GEMM row, resolved once per row before the epilogue
// (by the row set-up kernel, or by an idle warp of the cluster fc GEMM):
// {page, slot, position, 0}, page -1 when the row is not stored.
struct RowDest {
  int4 *dst;     // [N] or nullptr (the epilogue resolves rows itself)
  float2 *cs;    // [N][nf] cos/sin of the row's RoPE angles
  int nf;        // rotate-half pairs per row (GQA hd/2, MLA rope/2)
  MaskArgs m;    // ctx_snap = the live ctx_len (nothing advances it before the epilogue)
};

// One warp resolves GEMM row n: lane 0 the destination ({page, slot,
// position, 0}, page -1 when the row is not stored; a page outside the pool
// is flagged once), every lane a share of the row's RoPE cos/sin pairs (the
// angle formed in double precision once per row).
__device__ __forceinline__ void row_setup_warp(const RowDest &rd, const RopeFreqs &rf, int n,
                                               int lane) {
  int pos = -1;
  if (lane == 0) {
    int r, i, page = 0, slot = 0, p = 0;
    const bool w = row_of(rd.m, n, &r, &i) && ctx_row_dest(rd.m, r, i, &page, &slot, &p, true);
    rd.dst[n] = make_int4(w ? page : -1, slot, p, 0);
    pos = w ? p : -1;
  }
  pos = __shfl_sync(0xffffffffu, pos, 0);
  if (pos < 0) return;
  for (int f = lane; f < rd.nf; f += 32) {
    float c, sn;
    rope_cos_sin(pos, rf.f[f], &c, &sn);
    rd.cs[static_cast<size_t>(n) * rd.nf + f] = make_float2(c, sn);
  }
}

}  // namespace dflash
