// bookkeeping.cu -- the per-step drafter bookkeeping in one launch.
//
// Follows TensorRT-LLM PR #20550 (Description, TLLM_DFLASH_FUSED_PROLOGUE:
// the page counts and decoded table of _refresh_ctx_block_tables; the
// generation prologue's bonus token, query / context positions and embedding
// ids; the context-KV store's mask of rejected rows, clamp to the request's
// allocation and page lookup; the clamped ctx_len advance with dummy slots
// reset and the advertised context length) and its follow-up commit
// "spec_tail_kernels.py" (block-table decode from clamped, divided offsets;
// destination pages / offsets / write mask; seq_lens; DraftBlockPlacement
// for the block's own positions).
//
// One CTA per request: the table row is decoded by all threads with a block
// reduction for the page count; the per-row outputs are one thread per row.
#include "dflash_internal.cuh"

namespace dflash {
namespace {

struct BkArgs {
  const int32_t *off;
  int64_t off_stride;
  int32_t off_div;
  const int32_t *acc;
  int64_t acc_stride;
  const int32_t *n_acc;
  const int32_t *ctx_pre;
  const uint8_t *valid;
  int32_t max_ctx;
  int32_t mask_id;
  int32_t T, M, P;
  dflash_step_outputs o;
  int32_t *st;
};

// Two memory round trips on the dependent path: the table row and the
// request's scalars load together; then the bonus token and every row's page
// lookup.  Each thread derives the request's scalars itself from shared
// memory, so no second barrier sits between them and the row outputs.
__global__ void __launch_bounds__(128) bookkeeping_kernel(const BkArgs a) {
  __shared__ int s_cnt[4];
  __shared__ int s_in[3];  // n, c, live
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int r = blockIdx.x;
  const int32_t *orow = a.off + static_cast<int64_t>(r) * a.off_stride;
  int n_in = 0, c_in = 0, live_in = 1;
  if (threadIdx.x == 0) {  // issued now, used after the table loads
    n_in = a.n_acc[r];
    c_in = a.ctx_pre[r];
    live_in = a.valid ? (a.valid[r] != 0) : 1;
  }

  // 1. block-table decode: count of non-negative offsets, clamp and divide.
  int cnt = 0;
  for (int j = threadIdx.x; j < a.M; j += blockDim.x) {
    const int v = orow[j];
    cnt += (v >= 0);
    a.o.block_table[static_cast<int64_t>(r) * a.M + j] = (v > 0 ? v : 0) / a.off_div;
  }
  cnt = warp_sum_int(cnt);
  if ((threadIdx.x & 31) == 0) s_cnt[threadIdx.x >> 5] = cnt;
  if (threadIdx.x == 0) {
    s_in[0] = n_in;
    s_in[1] = c_in;
    s_in[2] = live_in;
  }
  __syncthreads();

  // 2. per-request scalars (every thread; thread 0 writes them out).
  int np = 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) np += s_cnt[w];
  const int n = s_in[0], c = s_in[1];
  const bool live = s_in[2] != 0;
  bool okb = live;
  unsigned bits = 0;
  if (live && (n < 1 || n > a.T)) { okb = false; bits |= DFLASH_DEV_BAD_NACCEPTED; }
  if (live && c < 0) { okb = false; bits |= DFLASH_DEV_BAD_CTX_LEN; }
  if (!okb) np = 0;
  const long long cap = static_cast<long long>(np) * a.P;
  const int A = okb ? static_cast<int>(cap < a.max_ctx ? cap : a.max_ctx) : 0;
  int cn = 0;
  if (okb) {
    const long long sum = static_cast<long long>(c) + n;
    cn = static_cast<int>(sum < A ? sum : A);
    if (c > A) bits |= DFLASH_DEV_CTX_OUTRUN;
  }
  const int ok = okb ? 1 : 0;
  // the bonus token's load goes out with the rows' page lookups; everything
  // that uses it is stored last
  int b = a.mask_id;
  if (threadIdx.x == 0 && ok) b = a.acc[static_cast<int64_t>(r) * a.acc_stride + (n - 1)];

  // 3. per-row outputs (row 0's bonus token: thread 0, which loaded it).
  for (int i = threadIdx.x; i < a.T; i += blockDim.x) {
    const int64_t k = static_cast<int64_t>(r) * a.T + i;

    // context row i at c + i
    const int p = ok ? c + i : 0;
    a.o.ctx_pos[k] = p;
    int w = 0, page = -1, slot = -1;
    if (ok && i < n && p < A) {
      const int lp = p / a.P;
      if (lp < a.M) {
        const int v = orow[lp];
        if (v >= 0) { w = 1; page = v / a.off_div; slot = p % a.P; }
      }
    }
    a.o.ctx_wmask[k] = static_cast<uint8_t>(w);
    a.o.ctx_dst_page[k] = page;
    a.o.ctx_dst_slot[k] = slot;

    // block row i at c' + i
    const int q = ok ? cn + i : 0;
    a.o.q_pos[k] = q;
    int bw = 0, bpage = -1, bslot = -1;
    if (ok && static_cast<long long>(q) < cap) {
      const int lp = q / a.P;
      if (lp < a.M) {
        const int v = orow[lp];
        if (v >= 0) { bw = 1; bpage = v / a.off_div; bslot = q % a.P; }
      }
    }
    a.o.blk_mask[k] = static_cast<uint8_t>(bw);
    a.o.blk_page[k] = bpage;
    a.o.blk_slot[k] = bslot;
    a.o.emb_ids[k] = (i == 0) ? b : a.mask_id;
  }
  if (threadIdx.x == 0) {
    a.o.bonus[r] = b;
    a.o.n_pages[r] = np;
    a.o.alloc_limit[r] = A;
    a.o.ctx_len_new[r] = cn;
    a.o.seq_lens[r] = ok ? cn + a.T : 0;
    if (bits) raise_status(a.st, bits);
  }
}

}  // namespace

cudaError_t launch_bookkeeping(const dflash_geom &g, int B, const int32_t *off, int64_t off_stride,
                               int32_t off_div, const int32_t *acc, int64_t acc_stride,
                               const int32_t *n_acc, const int32_t *ctx_pre, const uint8_t *valid,
                               int32_t max_ctx, int32_t mask_id, const dflash_step_outputs &o,
                               int32_t *st, cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  BkArgs a;
  a.off = off;
  a.off_stride = off_stride;
  a.off_div = off_div;
  a.acc = acc;
  a.acc_stride = acc_stride;
  a.n_acc = n_acc;
  a.ctx_pre = ctx_pre;
  a.valid = valid;
  a.max_ctx = max_ctx;
  a.mask_id = mask_id;
  a.T = g.block_size;
  a.M = g.max_pages;
  a.P = g.page_size;
  a.o = o;
  a.st = st;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(B);
  cfg.blockDim = dim3(128);
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, bookkeeping_kernel, a);
}

}  // namespace dflash
