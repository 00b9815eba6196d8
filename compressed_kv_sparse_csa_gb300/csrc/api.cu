// Host side of the C ABI declared in include/ds4x.h: argument checks (all
// before any CUDA call, so a bad call launches nothing), the device
// architecture check, workspace sizing and dispatch to the kernels.
#include <atomic>
#include <cstdlib>
#include <cstring>

#include "ds4x_internal.cuh"

using namespace ds4x;

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Per-device cache of the architecture check: 0 unknown, 1 GB300, 2 other.
std::atomic<int> g_arch_ok[64];

int check_arch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DS4X_ECUDA;
  if (dev >= 0 && dev < 64) {
    const int c = g_arch_ok[dev].load(std::memory_order_relaxed);
    if (c != 0) return c == 1 ? DS4X_OK : DS4X_EARCH;
  }
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    return DS4X_ECUDA;
  }
  const bool ok = (major == 10 && minor == 3);
  if (dev >= 0 && dev < 64) g_arch_ok[dev].store(ok ? 1 : 2, std::memory_order_relaxed);
  return ok ? DS4X_OK : DS4X_EARCH;
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? DS4X_OK : DS4X_ECUDA; }

// DS4X_SCORER=two_stage selects the score-then-select path (A/B and debug);
// the default is the fused tensor-core scorer.
bool use_two_stage() {
  static const bool v = [] {
    const char *e = std::getenv("DS4X_SCORER");
    return e != nullptr && std::strcmp(e, "two_stage") == 0;
  }();
  return v;
}

}  // namespace

extern "C" {

const char *ds4x_status_str(int status) {
  switch (status) {
    case DS4X_OK: return "ok";
    case DS4X_EINVAL: return "invalid argument (null or misaligned pointer, bad size or k)";
    case DS4X_ERANGE: return "rows outside the cache capacity";
    case DS4X_EWORKSPACE: return "workspace too small";
    case DS4X_EARCH: return "device is not compute capability 10.3 (GB300)";
    case DS4X_ECUDA: return "CUDA runtime error";
    case DS4X_ETIMEOUT: return "bounded device wait gave up";
    case DS4X_EDEVICE: return "kernel-detected invalid input (index out of range)";
    case DS4X_EFORMAT: return "not a checkpoint of this layout, or corrupt or truncated";
    case DS4X_EVERSION: return "a checkpoint of another payload version";
    default: return "unknown status";
  }
}

int ds4x_abi_version(void) { return DS4X_ABI_VERSION; }

int64_t ds4x_cache_bytes(int64_t L) {
  if (L < 0) return -1;
  const int64_t ring = int64_t(43) * 256 * DS4X_KV_ROW_BYTES;
  const int64_t csa = int64_t(21) * (L / 4 + 2) * (DS4X_KV_ROW_BYTES + DS4X_IDX_ROW_BYTES);
  const int64_t hca = int64_t(20) * (L / 128 + 2) * DS4X_KV_ROW_BYTES;
  return ring + csa + hca;
}

int ds4x_workspace_init(void *ws, size_t ws_bytes, ds4x_stream_t stream) {
  if (ws == nullptr || !aligned16(ws) || ws_bytes < kWsHeaderBytes) return DS4X_EINVAL;
  const int a = check_arch();
  if (a != DS4X_OK) return a;
  return from_cuda(cudaMemsetAsync(ws, 0, ws_bytes, stream));
}

int ds4x_copy_async(void *dst, const void *src, size_t bytes, ds4x_stream_t stream) {
  if (dst == nullptr || src == nullptr || !aligned16(dst) || !aligned16(src)) return DS4X_EINVAL;
  const uintptr_t d = reinterpret_cast<uintptr_t>(dst), s = reinterpret_cast<uintptr_t>(src);
  if (bytes > 0 && d < s + bytes && s < d + bytes) return DS4X_EINVAL;  // overlapping
  if (bytes == 0) return DS4X_OK;
  const int a = check_arch();
  if (a != DS4X_OK) return a;
  return from_cuda(launch_copy(dst, src, bytes, stream));
}

int ds4x_workspace_status(void *ws, ds4x_stream_t stream, int32_t *status_host) {
  if (ws == nullptr || status_host == nullptr || !aligned16(ws)) return DS4X_EINVAL;
  const int a = check_arch();
  if (a != DS4X_OK) return a;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return DS4X_ECUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, ws, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return DS4X_ECUDA;
  const int32_t zero = 0;
  if (cudaMemcpy(ws, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return DS4X_ECUDA;
  *status_host = v;
  return DS4X_OK;
}

int ds4x_cache_append(uint8_t *kv_rows, uint8_t *idx_rows, int64_t capacity, int64_t pos,
                      const float *kv_in, const float *idx_in, int64_t n, ds4x_stream_t stream) {
  if (kv_rows == nullptr && idx_rows == nullptr) return DS4X_EINVAL;
  if (kv_rows != nullptr && (kv_in == nullptr || !aligned16(kv_in) || !aligned16(kv_rows))) return DS4X_EINVAL;
  if (idx_rows != nullptr && (idx_in == nullptr || !aligned16(idx_in) || !aligned16(idx_rows))) return DS4X_EINVAL;
  if (n < 1 || capacity < 1) return DS4X_EINVAL;
  if (pos < 0 || pos > capacity || n > capacity - pos) return DS4X_ERANGE;
  const int a = check_arch();
  if (a != DS4X_OK) return a;
  return from_cuda(launch_cache_append(kv_rows, idx_rows, pos, kv_in, idx_in, n, stream));
}

size_t ds4x_index_score_topk_workspace(int64_t n_rows, int32_t k) {
  (void)k;
  if (n_rows < 1) n_rows = 1;
  const size_t a = score_two_stage_ws_bytes(n_rows), b = score_fused_ws_bytes();
  return a > b ? a : b;
}

int ds4x_index_score_topk(const uint8_t *idx_rows, int64_t n_rows, const uint16_t *q_bf16,
                          const float *w, int32_t k, int32_t *out_idx, float *out_score, void *ws,
                          size_t ws_bytes, ds4x_stream_t stream) {
  if (idx_rows == nullptr || q_bf16 == nullptr || w == nullptr || out_idx == nullptr || ws == nullptr)
    return DS4X_EINVAL;
  if (!aligned16(idx_rows) || !aligned16(q_bf16) || !aligned16(w) || !aligned16(out_idx) ||
      !aligned16(ws) || (out_score != nullptr && !aligned16(out_score)))
    return DS4X_EINVAL;
  if (n_rows < 1 || n_rows > int64_t(INT32_MAX) || k < 1 || k > DS4X_TOPK_MAX) return DS4X_EINVAL;
  if (ws_bytes < ds4x_index_score_topk_workspace(n_rows, k)) return DS4X_EWORKSPACE;
  const int a = check_arch();
  if (a != DS4X_OK) return a;
  if (use_two_stage())
    return from_cuda(launch_score_two_stage(idx_rows, n_rows, q_bf16, w, k, out_idx, out_score, ws, stream));
  return from_cuda(launch_score_fused(idx_rows, n_rows, q_bf16, w, k, out_idx, out_score, ws, stream));
}

size_t ds4x_sparse_attn_decode_workspace(int32_t k) {
  if (k < 1) k = 1;
  if (k > DS4X_TOPK_MAX) k = DS4X_TOPK_MAX;
  return attn_decode_ws_bytes(k);
}

int ds4x_sparse_attn_decode(const uint8_t *kv_rows, int64_t n_rows, const int32_t *idx, int32_t k,
                            const uint16_t *q_bf16, float softmax_scale, uint16_t *out_bf16,
                            float *lse, void *ws, size_t ws_bytes, ds4x_stream_t stream) {
  if (kv_rows == nullptr || idx == nullptr || q_bf16 == nullptr || out_bf16 == nullptr || ws == nullptr)
    return DS4X_EINVAL;
  if (!aligned16(kv_rows) || !aligned16(idx) || !aligned16(q_bf16) || !aligned16(out_bf16) ||
      !aligned16(ws) || (lse != nullptr && !aligned16(lse)))
    return DS4X_EINVAL;
  if (n_rows < 1 || k < 1 || k > DS4X_TOPK_MAX) return DS4X_EINVAL;
  if (ws_bytes < ds4x_sparse_attn_decode_workspace(k)) return DS4X_EWORKSPACE;
  const int a = check_arch();
  if (a != DS4X_OK) return a;
  return from_cuda(launch_attn_decode(kv_rows, n_rows, idx, k, q_bf16, softmax_scale, out_bf16, lse,
                                      ws, stream));
}

size_t ds4x_csa_decode_step_workspace(int64_t n_rows, int32_t k) {
  const size_t a = ds4x_index_score_topk_workspace(n_rows, k), b = ds4x_sparse_attn_decode_workspace(k);
  return a > b ? a : b;
}

int ds4x_csa_decode_step(const uint8_t *idx_rows, const uint8_t *kv_rows, int64_t n_rows, const uint16_t *q_idx_bf16,
                         const float *w, int32_t k, const uint16_t *q_attn_bf16, float softmax_scale,
                         int32_t *out_idx, float *out_score, uint16_t *out_bf16, float *lse, void *ws,
                         size_t ws_bytes, ds4x_stream_t stream) {
  if (idx_rows == nullptr || kv_rows == nullptr || q_idx_bf16 == nullptr || w == nullptr || q_attn_bf16 == nullptr ||
      out_idx == nullptr || out_bf16 == nullptr || ws == nullptr)
    return DS4X_EINVAL;
  if (!aligned16(idx_rows) || !aligned16(kv_rows) || !aligned16(q_idx_bf16) || !aligned16(w) ||
      !aligned16(q_attn_bf16) || !aligned16(out_idx) || !aligned16(out_bf16) || !aligned16(ws) ||
      (out_score != nullptr && !aligned16(out_score)) || (lse != nullptr && !aligned16(lse)))
    return DS4X_EINVAL;
  if (n_rows < 1 || n_rows > int64_t(INT32_MAX) || k < 1 || k > DS4X_TOPK_MAX) return DS4X_EINVAL;
  if (ws_bytes < ds4x_csa_decode_step_workspace(n_rows, k)) return DS4X_EWORKSPACE;
  const int a = check_arch();
  if (a != DS4X_OK) return a;
  // the attention shares the scorer's workspace header (it only ever sets its status word)
  cudaError_t e = use_two_stage()
                      ? launch_score_two_stage(idx_rows, n_rows, q_idx_bf16, w, k, out_idx, out_score, ws, stream)
                      : launch_score_fused(idx_rows, n_rows, q_idx_bf16, w, k, out_idx, out_score, ws, stream);
  if (e != cudaSuccess) return DS4X_ECUDA;
  return from_cuda(launch_attn_decode(kv_rows, n_rows, out_idx, k, q_attn_bf16, softmax_scale, out_bf16, lse, ws,
                                      stream));
}

size_t ds4x_index_score_topk_batched_workspace(int32_t n_sess, int32_t k) {
  (void)n_sess;
  (void)k;
  return score_fused_ws_bytes();
}

int ds4x_index_score_topk_batched(const uint8_t *const *idx_rows, const int64_t *n_rows, int32_t n_sess,
                                  const uint16_t *q_bf16, const float *w, int32_t k, int32_t *out_idx,
                                  float *out_score, void *ws, size_t ws_bytes, ds4x_stream_t stream) {
  if (idx_rows == nullptr || n_rows == nullptr || q_bf16 == nullptr || w == nullptr || out_idx == nullptr ||
      ws == nullptr)
    return DS4X_EINVAL;
  if (!aligned16(idx_rows) || !aligned16(n_rows) || !aligned16(q_bf16) || !aligned16(w) || !aligned16(out_idx) ||
      !aligned16(ws) || (out_score != nullptr && !aligned16(out_score)))
    return DS4X_EINVAL;
  if (n_sess < 1 || n_sess > DS4X_MAX_SESSIONS || k < 1 || k > DS4X_TOPK_MAX) return DS4X_EINVAL;
  if (ws_bytes < ds4x_index_score_topk_batched_workspace(n_sess, k)) return DS4X_EWORKSPACE;
  const int a = check_arch();
  if (a != DS4X_OK) return a;
  ScoreBatch sb{};
  sb.rows_arr = idx_rows;
  sb.n_arr = n_rows;
  sb.n_sess = n_sess;
  sb.q = q_bf16;
  sb.w = w;
  sb.k = k;
  sb.out_idx = out_idx;
  sb.out_score = out_score;
  return from_cuda(launch_score_batch(sb, 0, ws, stream));
}

int ds4x_sparse_attn_decode_batched(const uint8_t *const *kv_rows, const int64_t *n_rows, int32_t n_sess,
                                    const int32_t *idx, int32_t k, const uint16_t *q_bf16, float softmax_scale,
                                    uint16_t *out_bf16, float *lse, void *ws, size_t ws_bytes,
                                    ds4x_stream_t stream) {
  if (kv_rows == nullptr || n_rows == nullptr || idx == nullptr || q_bf16 == nullptr || out_bf16 == nullptr ||
      ws == nullptr)
    return DS4X_EINVAL;
  if (!aligned16(kv_rows) || !aligned16(n_rows) || !aligned16(idx) || !aligned16(q_bf16) || !aligned16(out_bf16) ||
      !aligned16(ws) || (lse != nullptr && !aligned16(lse)))
    return DS4X_EINVAL;
  if (n_sess < 1 || n_sess > DS4X_MAX_SESSIONS || k < 1 || k > DS4X_TOPK_MAX) return DS4X_EINVAL;
  if (ws_bytes < ds4x_sparse_attn_decode_workspace(k)) return DS4X_EWORKSPACE;
  const int a = check_arch();
  if (a != DS4X_OK) return a;
  AttnBatch ab{};
  ab.kv_arr = kv_rows;
  ab.n_arr = n_rows;
  ab.idx = idx;
  ab.k = k;
  ab.scale = softmax_scale;
  ab.q = q_bf16;
  ab.out = out_bf16;
  ab.lse = lse;
  return from_cuda(launch_attn_batch(ab, n_sess, ws, stream));
}

int ds4x_sparse_attn_prefill(const uint8_t *kv_rows, int64_t n_rows, const int32_t *idx, int32_t n_queries,
                             int32_t k, const uint16_t *q_bf16, float softmax_scale, uint16_t *out_bf16,
                             float *lse, void *ws, size_t ws_bytes, ds4x_stream_t stream) {
  if (kv_rows == nullptr || idx == nullptr || q_bf16 == nullptr || out_bf16 == nullptr || ws == nullptr)
    return DS4X_EINVAL;
  if (!aligned16(kv_rows) || !aligned16(idx) || !aligned16(q_bf16) || !aligned16(out_bf16) || !aligned16(ws) ||
      (lse != nullptr && !aligned16(lse)))
    return DS4X_EINVAL;
  if (n_rows < 1 || n_queries < 1 || n_queries > DS4X_PREFILL_MAX_QUERIES || k < 1 || k > DS4X_TOPK_MAX)
    return DS4X_EINVAL;
  if (ws_bytes < ds4x_sparse_attn_decode_workspace(k) || ws_bytes < attn_prefill_ws_bytes()) return DS4X_EWORKSPACE;
  const int a = check_arch();
  if (a != DS4X_OK) return a;
  return from_cuda(launch_attn_prefill(kv_rows, n_rows, idx, n_queries, k, q_bf16, softmax_scale, out_bf16, lse, ws,
                                       stream));
}

size_t ds4x_dense_attn_decode_workspace(int64_t n_rows) {
  if (n_rows < 1) n_rows = 1;
  if (n_rows > DS4X_DENSE_MAX_ROWS) n_rows = DS4X_DENSE_MAX_ROWS;
  return dense_attn_ws_bytes(n_rows);
}

int ds4x_dense_attn_decode(const uint8_t *kv_rows, int64_t n_rows, const uint16_t *q_bf16, float softmax_scale,
                           uint16_t *out_bf16, float *lse, void *ws, size_t ws_bytes, ds4x_stream_t stream) {
  if (kv_rows == nullptr || q_bf16 == nullptr || out_bf16 == nullptr || ws == nullptr) return DS4X_EINVAL;
  if (!aligned16(kv_rows) || !aligned16(q_bf16) || !aligned16(out_bf16) || !aligned16(ws) ||
      (lse != nullptr && !aligned16(lse)))
    return DS4X_EINVAL;
  if (n_rows < 1 || n_rows > DS4X_DENSE_MAX_ROWS) return DS4X_EINVAL;
  if (ws_bytes < ds4x_dense_attn_decode_workspace(n_rows)) return DS4X_EWORKSPACE;
  const int a = check_arch();
  if (a != DS4X_OK) return a;
  return from_cuda(launch_dense_attn(kv_rows, n_rows, q_bf16, softmax_scale, out_bf16, lse, ws, stream));
}

size_t ds4x_window_sparse_attn_decode_workspace(void) { return window_attn_ws_bytes(); }

int ds4x_window_sparse_attn_decode(const uint8_t *kv_rows, int64_t n_rows, const int32_t *idx, int32_t k,
                                   const uint8_t *ring_rows, int32_t ring_pos, int32_t w, const uint16_t *q_bf16,
                                   float softmax_scale, uint16_t *out_bf16, float *lse, void *ws, size_t ws_bytes,
                                   ds4x_stream_t stream) {
  if (kv_rows == nullptr || idx == nullptr || ring_rows == nullptr || q_bf16 == nullptr || out_bf16 == nullptr ||
      ws == nullptr)
    return DS4X_EINVAL;
  if (!aligned16(kv_rows) || !aligned16(idx) || !aligned16(ring_rows) || !aligned16(q_bf16) ||
      !aligned16(out_bf16) || !aligned16(ws) || (lse != nullptr && !aligned16(lse)))
    return DS4X_EINVAL;
  if (n_rows < 1 || k < 1 || k > DS4X_TOPK_MAX || ring_pos < 0 || ring_pos >= DS4X_RING_ROWS || w < 0 ||
      w > DS4X_RING_ROWS)
    return DS4X_EINVAL;
  if (ws_bytes < ds4x_window_sparse_attn_decode_workspace()) return DS4X_EWORKSPACE;
  const int a = check_arch();
  if (a != DS4X_OK) return a;
  return from_cuda(launch_window_attn(kv_rows, n_rows, idx, k, ring_rows, ring_pos, w, q_bf16, softmax_scale,
                                      out_bf16, lse, ws, stream));
}

int ds4x_quantize_query_e4m3(const float *q, int64_t n_vec128, uint8_t *codes, uint8_t *scales,
                              ds4x_stream_t stream) {
  if (q == nullptr || codes == nullptr || scales == nullptr) return DS4X_EINVAL;
  if (!aligned16(q) || !aligned16(codes) || !aligned16(scales)) return DS4X_EINVAL;
  if (n_vec128 < 1 || n_vec128 > (int64_t(1) << 34)) return DS4X_EINVAL;
  const int a = check_arch();
  if (a != DS4X_OK) return a;
  return from_cuda(launch_quantize_query(q, n_vec128, codes, scales, stream));
}

size_t ds4x_index_score_topk_prefill_workspace(int64_t n_rows, int32_t n_queries, int32_t k) {
  (void)k;
  return prefill_ws_bytes(n_rows, n_queries);
}

int ds4x_index_score_topk_prefill(const uint8_t *idx_rows, int64_t n_rows, const uint8_t *q_codes,
                                  const uint8_t *q_scales, const float *w, int32_t n_queries, int64_t causal_base,
                                  int32_t k, int32_t *out_idx, float *out_score, void *ws, size_t ws_bytes,
                                  ds4x_stream_t stream) {
  if (idx_rows == nullptr || q_codes == nullptr || q_scales == nullptr || w == nullptr || out_idx == nullptr ||
      ws == nullptr)
    return DS4X_EINVAL;
  if (!aligned16(idx_rows) || !aligned16(q_codes) || !aligned16(q_scales) || !aligned16(w) || !aligned16(out_idx) ||
      !aligned16(ws) || (out_score != nullptr && !aligned16(out_score)))
    return DS4X_EINVAL;
  if (n_rows < 1 || n_rows > int64_t(INT32_MAX) || n_queries < 1 || n_queries > DS4X_PREFILL_MAX_QUERIES ||
      k < 1 || k > DS4X_TOPK_MAX)
    return DS4X_EINVAL;
  if (ws_bytes < ds4x_index_score_topk_prefill_workspace(n_rows, n_queries, k)) return DS4X_EWORKSPACE;
  const int a = check_arch();
  if (a != DS4X_OK) return a;
  return from_cuda(launch_score_prefill(idx_rows, n_rows, q_codes, q_scales, w, n_queries, causal_base, k, out_idx,
                                        out_score, ws, stream));
}

}  // extern "C"
