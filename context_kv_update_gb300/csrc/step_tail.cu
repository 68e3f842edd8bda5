// step_tail.cu -- the steps either side of the drafter's hot path.
//
// Before it: strict acceptance of a uniform-width draft in one launch
// [TensorRT-LLM PR #20550, follow-up commit "spec_tail_kernels.py"].  Request
// r drafted K tokens; the target produced K + 1 tokens at the same positions.
// Drafts are accepted while they equal the target's token, and the target's
// token at the first disagreement (or after the last draft) is the bonus, so
// n_accepted = 1 + (leading matches) and accepted[r, n - 1] is the bonus the
// bookkeeping reads.
//
// After it: the noise block's input rows are one embedding lookup over the
// block's ids [bonus, mask_id, ...] [TensorRT-LLM PR #13995, "fuse
// query-input build in pure Torch + fused embedding lookup"].
#include "dflash_internal.cuh"
#include "sm100_ptx.cuh"

namespace dflash {
namespace {

// One warp per request; positions in chunks of 32: the first mismatch is the
// lowest set bit of the chunk's mismatch ballot.
__global__ void __launch_bounds__(256) strict_accept_kernel(int B, int K, const int32_t *draft,
                                                             int64_t draft_stride,
                                                             const int32_t *target,
                                                             int64_t target_stride,
                                                             int32_t *n_acc, int32_t *accepted) {
  ptx::griddep_launch();
  ptx::griddep_wait();
  const int r = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= B) return;
  const int32_t *d = draft + static_cast<int64_t>(r) * draft_stride;
  const int32_t *t = target + static_cast<int64_t>(r) * target_stride;
  int m = K;  // leading matches
  for (int c = 0; c < K; c += 32) {
    const int i = c + lane;
    const bool mismatch = i < K && d[i] != t[i];
    const unsigned bal = __ballot_sync(0xffffffffu, mismatch);
    if (bal) {
      m = c + __ffs(bal) - 1;
      break;
    }
  }
  int32_t *a = accepted + static_cast<int64_t>(r) * (K + 1);
  for (int i = lane; i <= K; i += 32) a[i] = i <= m ? t[i] : -1;
  if (lane == 0) n_acc[r] = m + 1;
}

// One CTA per output row; 16-byte copies.  An id outside [0, vocab) gives a
// zero row and flags DFLASH_DEV_BAD_TOKEN.
__global__ void __launch_bounds__(256) embedding_gather_kernel(const int32_t *ids,
                                                                const uint4 *table, int vocab,
                                                                int units, uint4 *out,
                                                                int32_t *st) {
  ptx::griddep_launch();
  ptx::griddep_wait();
  const int k = blockIdx.x;
  const int id = ids[k];
  const bool ok = id >= 0 && id < vocab;
  if (!ok && threadIdx.x == 0) raise_status(st, DFLASH_DEV_BAD_TOKEN);
  const uint4 *src = table + static_cast<int64_t>(ok ? id : 0) * units;
  uint4 *dst = out + static_cast<int64_t>(k) * units;
  for (int u = threadIdx.x; u < units; u += blockDim.x)
    dst[u] = ok ? __ldg(src + u) : make_uint4(0, 0, 0, 0);
}

cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, cudaStream_t s, cudaLaunchAttribute *attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

}  // namespace

cudaError_t launch_strict_accept(int B, int K, const int32_t *draft, int64_t draft_stride,
                                 const int32_t *target, int64_t target_stride, int32_t *n_acc,
                                 int32_t *accepted, cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = pdl_config(dim3((B + 7) / 8), dim3(256), s, attr);
  return cudaLaunchKernelEx(&cfg, strict_accept_kernel, B, K, draft, draft_stride, target,
                            target_stride, n_acc, accepted);
}

cudaError_t launch_embedding_gather(int n, const int32_t *ids, const void *table, int vocab,
                                    int dim, void *out, int32_t *st, cudaStream_t s) {
  const int units = dim / 8;
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg =
      pdl_config(dim3(n), dim3(units < 256 ? ((units + 31) / 32) * 32 : 256), s, attr);
  return cudaLaunchKernelEx(&cfg, embedding_gather_kernel, ids, static_cast<const uint4 *>(table),
                            vocab, units, static_cast<uint4 *>(out), st);
}

}  // namespace dflash
