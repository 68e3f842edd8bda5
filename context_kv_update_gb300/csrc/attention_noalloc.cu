// attention_noalloc.cu -- dflash_block_attention_noalloc: the block attention
// with its split-KV scratch taken from a fixed array inside this library
// instead of a caller buffer.
//
// Who needs it: callers that cannot allocate device memory at the point where
// they run the attention -- a plugin whose host framework owns all device
// memory and offers it no allocator, or a latency-critical loop that must
// never block in the allocator.  Such a caller still owns q, the pool, the
// tables and the output; only the scratch comes from here.
//
// The scratch is one file-scope __device__ array of kNoAllocScratchBytes.  It
// exists on every GPU that loads this library, for the life of the process.
// Every call shares it and it keeps the last call's contents; nothing in it
// needs clearing between calls (each call writes every partial it later
// reads).  Calls whose GPU work overlaps (on different streams, for example)
// race on it and must be serialised by the caller.
#include <mutex>

#include "attention_common.cuh"

namespace dflash {
namespace {

constexpr size_t kNoAllocScratchBytes = 32u << 20;  // 32 MiB

__device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array, resolved once per device with that
// device current.  In host code the array's name is only a host-side handle,
// so the address must come from cudaGetSymbolAddress.
constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

int cuda_status(cudaError_t e) { return e == cudaSuccess ? DFLASH_OK : DFLASH_ERR_CUDA; }

cudaError_t scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace dflash

using namespace dflash;

extern "C" size_t dflash_block_attention_noalloc_max_scratch_bytes(void) {
  return kNoAllocScratchBytes;
}

extern "C" int dflash_block_attention_noalloc(const dflash_geom *g, int B, int layer, int Tq,
                                              const void *q, const void *q_rope,
                                              const void *kv_pool, const int32_t *block_table,
                                              const int32_t *kv_len, int32_t window,
                                              const float *sinks, float scale, int mask_mode,
                                              int num_segments, void *out, int32_t *dev_status,
                                              dflash_stream_t stream) {
  // the argument checks of dflash_block_attention, then the size limit, then
  // the buffer pointers
  if (const int st =
          attention_args_status(g, B, layer, Tq, q_rope, window, &scale, mask_mode, num_segments))
    return st;
  if (B == 0) return DFLASH_OK;
  const int S = num_segments > 0 ? num_segments : attention_num_segments(*g, B, Tq);
  if (attention_workspace_bytes(*g, B, Tq, S) > kNoAllocScratchBytes)
    return DFLASH_ERR_WORKSPACE_TOO_SMALL;
  if (const int st = attention_ptrs_status(B, q, q_rope, kv_pool, block_table, kv_len, out))
    return st;
  void *scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return DFLASH_ERR_CUDA;
  return cuda_status(launch_block_attention(*g, B, layer, Tq, q, q_rope, kv_pool, block_table,
                                            kv_len, window, sinks, scale, mask_mode, S, scratch,
                                            out, dev_status,
                                            reinterpret_cast<cudaStream_t>(stream)));
}
