// dflash_internal.cuh -- declarations shared by the library's translation units
// (host launchers and small device helpers).  Not part of the public ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dflash.h"

namespace dflash {

// ------------------------------------------------------------ constants
constexpr int kMaxHeadDim = 256;
constexpr int kAttnTileKeys = 128;  // keys per attention tile
constexpr int kGemmTileM = 128;     // weight rows per GEMM tile
constexpr int kGemmTileK = 64;      // reduction depth per pipeline stage (128 B of bf16)
constexpr int kMaxPrefillRows = 65535;  // rows of one prefill store (the norm's grid height)

// ------------------------------------------------------------ status
__device__ __forceinline__ void raise_status(int32_t *st, unsigned bits) {
  if (st) atomicOr(reinterpret_cast<int *>(st), static_cast<int>(bits));
}

// ------------------------------------------------------------ bf16
__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}
__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// ------------------------------------------------------------ reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ int warp_sum_int(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Block-wide sum; `scratch` holds >= 32 floats; every thread gets the result.
__device__ __forceinline__ float block_sum(float v, float *scratch) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) scratch[wid] = v;
  __syncthreads();
  float t = (lane < nw) ? scratch[lane] : 0.f;
  t = warp_sum(t);
  return t;
}

// ------------------------------------------------------------ RoPE
// Rotate-half RoPE frequencies f_j = theta^(-2j/d), j < d/2, computed on the
// host in double precision and passed by value.
struct RopeFreqs {
  double f[kMaxHeadDim / 2];
};

// cos/sin of pos * f, the angle formed and reduced modulo 2*pi in double
// precision, then evaluated in fp32 on the reduced argument.
__device__ __forceinline__ void rope_cos_sin(int pos, double f, float *c, float *s) {
  const double two_pi = 6.283185307179586476925286766559;
  double a = static_cast<double>(pos) * f;
  double k = rint(a * (1.0 / two_pi));
  double red = fma(-k, two_pi, a);
  sincosf(static_cast<float>(red), s, c);
}

// ------------------------------------------------------------ host helpers
int device_sm_count();

// Raise a kernel's dynamic shared-memory limit once per device (before any
// graph capture the first eager call does it; later calls only read a flag).
// The kernel is a template argument so that every kernel -- also two
// instantiations of one kernel template, which share a type -- has its own
// flag.
template <auto Kernel>
cudaError_t ensure_smem_limit(int bytes) {
  static bool done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return e;
}
void fill_rope_freqs(RopeFreqs *rf, int dim, double theta);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ------------------------------------------------------------ launchers
cudaError_t launch_bookkeeping(const dflash_geom &g, int B, const int32_t *off, int64_t off_stride,
                               int32_t off_div, const int32_t *acc, int64_t acc_stride,
                               const int32_t *n_acc, const int32_t *ctx_pre, const uint8_t *valid,
                               int32_t max_ctx, int32_t mask_id, const dflash_step_outputs &o,
                               int32_t *st, cudaStream_t s);

size_t ctx_workspace_bytes(const dflash_geom &g, int B);
cudaError_t launch_ctx_kv_update(const dflash_geom &g, int B, const void *hidden, int hidden_dtype,
                                 const int32_t *n_acc, int32_t *ctx_len, const int32_t *alloc_limit,
                                 const int32_t *tbl, const uint8_t *valid, const dflash_weights &w,
                                 void *pool, void *ws, int32_t *st, cudaStream_t s);
// prefill store: every row of each request (rows cu_rows[r]..cu_rows[r+1]-1)
size_t ctx_prefill_workspace_bytes(const dflash_geom &g, int B, int rows);
cudaError_t launch_ctx_kv_prefill(const dflash_geom &g, int B, int rows, const void *hidden,
                                  int hidden_dtype, const int32_t *cu_rows, int32_t *ctx_len,
                                  const int32_t *alloc_limit, const int32_t *tbl,
                                  const uint8_t *valid, const dflash_weights &w, void *pool,
                                  void *ws, int32_t *st, cudaStream_t s);
// split update: projection into a staged buffer, then the masked store
size_t ctx_staged_bytes(const dflash_geom &g, int B);
cudaError_t launch_ctx_kv_project(const dflash_geom &g, int B, const void *hidden, int hidden_dtype,
                                  const int32_t *ctx_len, const dflash_weights &w, void *staged,
                                  void *ws, int32_t *st, cudaStream_t s);
cudaError_t launch_ctx_kv_commit(const dflash_geom &g, int B, const void *staged,
                                 const int32_t *n_acc, int32_t *ctx_len, const int32_t *alloc_limit,
                                 const int32_t *tbl, const uint8_t *valid, void *pool, int32_t *st,
                                 cudaStream_t s);

// query rows: RMSNorm (gamma non-null) + RoPE at pos[row], [rows][hq][dim]
cudaError_t launch_q_norm_rope(const dflash_geom &g, int rows, const void *q_in,
                               const void *gamma, const int32_t *pos, void *q_out,
                               cudaStream_t s);

cudaError_t launch_block_scatter(const dflash_geom &g, int B, int layer, const void *blk_k,
                                 const void *blk_v, const int32_t *page, const int32_t *slot,
                                 const uint8_t *mask, void *pool, int32_t *st, cudaStream_t s);

// weight packing (stacked per-layer K/V or latent projections and norm gains)
size_t packed_kv_bytes(const dflash_geom &g);
size_t packed_gamma_bytes(const dflash_geom &g);
int max_pack_layers();
cudaError_t launch_pack_weights(const dflash_geom &g, const dflash_layer_weights *layers,
                                void *w_kv, void *gamma, cudaStream_t s);

// either side of the path: strict acceptance, the noise-block embedding lookup
cudaError_t launch_strict_accept(int B, int K, const int32_t *draft, int64_t draft_stride,
                                 const int32_t *target, int64_t target_stride, int32_t *n_acc,
                                 int32_t *accepted, cudaStream_t s);
cudaError_t launch_embedding_gather(int n, const int32_t *ids, const void *table, int vocab,
                                    int dim, void *out, int32_t *st, cudaStream_t s);

int attention_num_segments(const dflash_geom &g, int B, int Tq);
void attention_test_skip_tile(int tile);
int attention_test_skip_tile_value();  // the calling thread's setting (-1: off)
float default_attention_scale(const dflash_geom &g);
int attention_args_status(const dflash_geom *g, int B, int layer, int Tq, const void *q_rope,
                          int32_t window, float *scale, int mask_mode, int num_segments);
int attention_ptrs_status(int B, const void *q, const void *q_rope, const void *kv_pool,
                          const int32_t *block_table, const int32_t *kv_len, const void *out);
size_t attention_workspace_bytes(const dflash_geom &g, int B, int Tq, int S);
cudaError_t launch_block_attention(const dflash_geom &g, int B, int layer, int Tq, const void *q,
                                   const void *q_rope, const void *pool, const int32_t *tbl,
                                   const int32_t *kv_len, int32_t window, const float *sinks,
                                   float scale, int mask_mode, int S, void *ws, void *out,
                                   int32_t *st, cudaStream_t s);
// The same with the layer's block scatter fused in (blk_k null: none);
// Tq == g.block_size.
cudaError_t launch_block_scatter_attention(const dflash_geom &g, int B, int layer, int Tq,
                                           const void *blk_k, const void *blk_v,
                                           const int32_t *blk_page, const int32_t *blk_slot,
                                           const uint8_t *blk_mask, const void *q,
                                           const void *q_rope, const void *pool,
                                           const int32_t *tbl, const int32_t *kv_len,
                                           int32_t window, const float *sinks, float scale,
                                           int mask_mode, int S, void *ws, void *out, int32_t *st,
                                           cudaStream_t s);
int block_scatter_args_status(const dflash_geom &g, const void *blk_k, const void *blk_v,
                              const int32_t *blk_page, const int32_t *blk_slot,
                              const uint8_t *blk_mask, const void *kv_pool);

}  // namespace dflash
