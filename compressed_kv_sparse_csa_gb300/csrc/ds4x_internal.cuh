// Internal declarations shared by the CUDA translation units of libds4x.
// Not part of the ABI; see include/ds4x.h for the public contract.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "ds4x.h"

namespace ds4x {

// ---------------------------------------------------------------------------
// Workspace header: the first 256 bytes of every workspace.
// ---------------------------------------------------------------------------
struct WsHeader {
  int32_t status;        // DS4X_OK / DS4X_EDEVICE / DS4X_ETIMEOUT (sticky)
  uint32_t ticket;       // arrival counter of the fused scorer (self-resetting)
  uint32_t fallback;     // number of scorer calls that took the slow merge
  uint32_t wait_extra;   // arrivals the scorer's exchange waits for beyond its CTAs (0; a
                         // nonzero value makes the bounded wait run out: the time-out test)
  uint32_t pad[60];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");
constexpr size_t kWsHeaderBytes = 256;

// ---------------------------------------------------------------------------
// Sortable 64-bit (score, index) keys: larger key == earlier in the top-k.
// High word: the score's bits mapped to an unsigned total order (-0 first
// canonicalised to +0).  Low word: ~index, so the lower index wins a tie.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t float_to_ordered(float s) {
  uint32_t u = __float_as_uint(s == 0.0f ? 0.0f : s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float ordered_to_float(uint32_t o) {
  uint32_t u = (o & 0x80000000u) ? (o & 0x7fffffffu) : ~o;
  return __uint_as_float(u);
}
__device__ __forceinline__ uint64_t make_key(float s, uint32_t idx) {
  return (uint64_t(float_to_ordered(s)) << 32) | uint64_t(~idx);
}
__device__ __forceinline__ int32_t key_index(uint64_t key) {
  return int32_t(~uint32_t(key & 0xffffffffu));
}
__device__ __forceinline__ float key_score(uint64_t key) {
  return ordered_to_float(uint32_t(key >> 32));
}

// ---------------------------------------------------------------------------
// Block-scale helpers shared by the cache writer and the scorer's query split.
// ---------------------------------------------------------------------------
// Least integer e with amax <= emax * 2^e, where emax = g * 2^G (0.5 <= g < 1):
// with amax = f * 2^F, e = F - G when f <= g, else F - G + 1.
__device__ __forceinline__ int block_exponent(float amax, float g, int G) {
  if (amax == 0.0f) return 0;
  int F;
  const float f = frexpf(amax, &F);
  const int e = F - G + (f > g ? 1 : 0);
  return max(-127, min(127, e));
}

// 2^-e as a float, for e in [-127, 126] (every exponent a finite block can have).
__device__ __forceinline__ float pow2_neg(int e) {
  return __uint_as_float(uint32_t(127 - e) << 23);
}

// Two floats -> two E4M3 codes: `lo` in bits 0-7, `hi` in bits 8-15.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Raises a kernel's dynamic shared-memory limit, once per device.
template <typename Kernel>
cudaError_t set_max_smem_once(Kernel *kernel, int bytes, std::atomic<uint64_t> &done_mask) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = uint64_t(1) << (dev & 63);
  if (done_mask.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done_mask.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Launches kernel<<<grid, block, smem, stream>>>(args...) with programmatic
// stream serialisation: its CTAs may be scheduled while the previous kernel
// in the stream finishes; the kernel waits for it (griddepcontrol.wait)
// before it touches memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t stream,
                       Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ---------------------------------------------------------------------------
// Launchers (host).  Each returns a cudaError_t from cudaGetLastError().
// ---------------------------------------------------------------------------
cudaError_t launch_cache_append(uint8_t *kv_rows, uint8_t *idx_rows, int64_t pos,
                                const float *kv_in, const float *idx_in, int64_t n,
                                cudaStream_t stream);

// Two-stage scorer: full key array, then a single-CTA radix select.
size_t score_two_stage_ws_bytes(int64_t n_rows);
cudaError_t launch_score_two_stage(const uint8_t *idx_rows, int64_t n_rows,
                                   const uint16_t *q, const float *w, int32_t k,
                                   int32_t *out_idx, float *out_score, void *ws,
                                   cudaStream_t stream);

// Fused tensor-core scorer with per-CTA top-512 and a last-CTA merge, over
// one session (rows / n_rows) or a batch (device arrays rows_arr / n_arr of
// n_sess sessions; session s reads q + s * 64 * 128, w + s * 64 and writes
// out_idx + s k, out_score + s k).
struct ScoreBatch {
  const uint8_t *rows;
  int64_t n_rows;
  const uint8_t *const *rows_arr;
  const int64_t *n_arr;
  int32_t n_sess;
  const uint16_t *q;
  const float *w;
  int32_t k;
  int32_t *out_idx;
  float *out_score;
};
// tiles_hint: the one session's tile count, or 0 for a batch (all SMs).
cudaError_t launch_score_batch(const ScoreBatch &sb, int64_t tiles_hint, void *ws, cudaStream_t stream);
size_t score_fused_ws_bytes();
int score_fused_max_ctas();
cudaError_t launch_score_fused(const uint8_t *idx_rows, int64_t n_rows, const uint16_t *q,
                               const float *w, int32_t k, int32_t *out_idx, float *out_score, void *ws,
                               cudaStream_t stream);

// Sparse attention over a batch of (cache, selected rows, query) items; item
// b reads kv_arr[b] / n_arr[b] when those device arrays are given, else the
// one shared cache, and idx + b k, q + b * 64 * 512, out + b * 64 * 512,
// lse + b * 64.
struct AttnBatch {
  const uint8_t *kv;
  int64_t n_rows;
  const uint8_t *const *kv_arr;
  const int64_t *n_arr;
  const int32_t *idx;
  int32_t k;
  float scale;
  const uint16_t *q;
  uint16_t *out;
  float *lse;
  bool q_shared;   // every item reads the one query at q (the window path's two row sets)
  float *out_f32;  // item b's normalised fp32 output at out_f32 + b * 64 * 512 instead of out (for a finalize)
};
cudaError_t launch_attn_batch(const AttnBatch &ab, int batch, void *ws, cudaStream_t stream);
size_t attn_decode_ws_bytes(int32_t k);

// Dense attention over every row [0, n_rows) (one query): items of
// consecutive rows (dense_rows_per_item: 128, 256, 384 or 512, the fewest
// that keep the items at 256 or fewer up to 131,072 rows) through the
// tensor-core attention kernel (fp32 partials), then a finalize.
constexpr int64_t kDenseMaxTiles = 8192;  // rows up to 8192 * 512
static_assert(kDenseMaxTiles * DS4X_TOPK_MAX == DS4X_DENSE_MAX_ROWS, "the ABI's row limit");
int32_t dense_rows_per_item(int64_t n_rows);
size_t dense_attn_ws_bytes(int64_t n_rows);
cudaError_t launch_dense_attn(const uint8_t *kv_rows, int64_t n_rows, const uint16_t *q, float scale, uint16_t *out,
                              float *lse, void *ws, cudaStream_t stream);

// Attention over k selected rows plus the raw sliding window's w ring rows
// (one softmax over both): the two as items of one attention launch (fp32
// partials), then the finalize.
size_t window_attn_ws_bytes();
cudaError_t launch_window_attn(const uint8_t *kv_rows, int64_t n_rows, const int32_t *idx, int32_t k,
                               const uint8_t *ring_rows, int32_t ring_pos, int32_t w, const uint16_t *q, float scale,
                               uint16_t *out, float *lse, void *ws, cudaStream_t stream);

// Chunked prefill: query quantiser and the multi-query scorer.
cudaError_t launch_quantize_query(const float *q, int64_t n_vec, uint8_t *codes, uint8_t *scales,
                                  cudaStream_t stream);
// Workspace of the prefill scorer: the header, then the fp32 scores of up to
// 512 query tokens (one launch's) over n_rows rows.
size_t prefill_ws_bytes(int64_t n_rows, int32_t T);
cudaError_t launch_score_prefill(const uint8_t *idx_rows, int64_t n_rows, const uint8_t *q_codes,
                                 const uint8_t *q_scales, const float *w, int32_t T, int64_t causal_base,
                                 int32_t k, int32_t *out_idx, float *out_score, void *ws, cudaStream_t stream);
// Prefill attention on the tensor cores: n_queries query tokens, each over its
// own k selected rows (idx [n_queries][k]), one persistent CTA per SM.
size_t attn_prefill_ws_bytes();
cudaError_t launch_attn_prefill(const uint8_t *kv_rows, int64_t n_rows, const int32_t *idx, int32_t n_queries,
                                int32_t k, const uint16_t *q, float scale, uint16_t *out, float *lse, void *ws,
                                cudaStream_t stream);
// The same kernel over `items` dense items of rows_per_item consecutive rows
// each (item i: rows i rows_per_item .. below n_rows), all with the one query
// q, writing each item's normalised fp32 output [64][512] and LSE [64].
cudaError_t launch_attn_dense_items(const uint8_t *kv_rows, int64_t n_rows, int32_t rows_per_item, int32_t items,
                                    const uint16_t *q, float scale, float *out_f32, float *lse, void *ws,
                                    cudaStream_t stream);
// Kernel-side copy (device or GPU-addressable pinned host memory on either side).
cudaError_t launch_copy(void *dst, const void *src, size_t bytes, cudaStream_t stream);
cudaError_t launch_attn_decode(const uint8_t *kv_rows, int64_t n_rows, const int32_t *idx,
                               int32_t k, const uint16_t *q, float scale, uint16_t *out,
                               float *lse, void *ws, cudaStream_t stream);

}  // namespace ds4x
