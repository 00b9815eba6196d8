// Chunked-prefill CSA scoring (DS4X README, "Packed prefill implementation":
// batch score/top-k over the packed 68-byte indexer rows for a chunk of
// query tokens).
//
// * quantize_query_kernel: each 128-value query vector (one token, one head)
//   becomes E4M3 codes with one UE8M0 scale per 32 values, with the block
//   scale rule of the cache writer (least e with amax <= 448 * 2^e) and the
//   hardware round-to-nearest-even E4M3 converter; one warp per vector.
// * prefill_prep_kernel: widens each quantised query back to its exact value
//   (an E4M3 value times a power of two has at most four significant bits,
//   so it is exact in bf16 whenever its exponent is in bf16's normal range),
//   and writes, per query token i, the session it is scored as: the same
//   indexer rows with the causal length min(n_rows, causal_base + i).
// * The scoring itself is the fused block-scaled scorer run as a batch of
//   such sessions (launch_score_batch), as many per launch as it has CTAs
//   (one per SM), spread evenly over the launches: every CTA then streams
//   one whole session, so no launch waits on a session with fewer CTAs;
//   its query split gives hi = the exact E4M3 value and lo = 0 for such a
//   query, so every product is exact and the sums are fp32.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ds4x_internal.cuh"

namespace ds4x {
namespace {

constexpr int kQBlock = 32;

__global__ void __launch_bounds__(256) quantize_query_kernel(const float *__restrict__ q, int64_t n_vec,
                                                             uint8_t *__restrict__ codes,
                                                             uint8_t *__restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t v = int64_t(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (v >= n_vec) return;
  // lane owns elements 4 lane .. 4 lane + 3; block b = lane / 8
  const float4 x = reinterpret_cast<const float4 *>(q + v * DS4X_IDX_DIM)[lane];
  float amax = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const int e = block_exponent(amax, 0.875f, 9);  // 448 = 0.875 * 2^9
  const float s = pow2_neg(e);
  const uint32_t lo = cvt_e4m3x2(x.y * s, x.x * s), hi = cvt_e4m3x2(x.w * s, x.z * s);
  reinterpret_cast<uint32_t *>(codes + v * DS4X_IDX_DIM)[lane] = lo | (hi << 16);
  if ((lane & 7) == 0) scales[v * (DS4X_IDX_DIM / kQBlock) + (lane >> 3)] = uint8_t(e + 127);
}

// E4M3FN code -> value (finite codes).
__device__ __forceinline__ float e4m3_code_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  const float mag = e == 0 ? float(m) * __uint_as_float(118u << 23)              // m * 2^-9
                           : float(8u + m) * __uint_as_float((117u + e) << 23);  // (8 + m) * 2^(e - 10)
  return (c & 0x80u) ? -mag : mag;
}

__global__ void __launch_bounds__(256) prefill_prep_kernel(const uint8_t *__restrict__ codes,
                                                           const uint8_t *__restrict__ scales, int32_t T,
                                                           const uint8_t *rows, int64_t n_rows,
                                                           int64_t causal_base, uint16_t *__restrict__ qbf,
                                                           const uint8_t **rows_arr, int64_t *n_arr) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;  // one element
  const int64_t total = int64_t(T) * DS4X_IDX_HEADS * DS4X_IDX_DIM;
  if (i < total) {
    const int64_t vec = i / DS4X_IDX_DIM;
    const int blk = int(i % DS4X_IDX_DIM) / kQBlock;
    const int sb = scales[vec * (DS4X_IDX_DIM / kQBlock) + blk];
    const float scale = sb == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(uint32_t(sb) << 23);
    qbf[i] = __bfloat16_as_ushort(__float2bfloat16_rn(e4m3_code_value(codes[i]) * scale));
  }
  if (i < T) {
    const int64_t vis = causal_base + i;
    rows_arr[i] = rows;
    n_arr[i] = vis < 0 ? 0 : (vis < n_rows ? vis : n_rows);
  }
}

struct PrefillWsLayout {
  size_t fused, qbf, ptrs, lens, total;
};

PrefillWsLayout prefill_layout(int32_t T) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  PrefillWsLayout L;
  L.fused = 0;
  L.qbf = up(score_fused_ws_bytes());
  L.ptrs = L.qbf + up(size_t(T) * DS4X_IDX_HEADS * DS4X_IDX_DIM * sizeof(uint16_t));
  L.lens = L.ptrs + up(size_t(T) * sizeof(void *));
  L.total = L.lens + up(size_t(T) * sizeof(int64_t));
  return L;
}

}  // namespace

cudaError_t launch_quantize_query(const float *q, int64_t n_vec, uint8_t *codes, uint8_t *scales,
                                  cudaStream_t stream) {
  const int warps = 8;
  const int64_t blocks = (n_vec + warps - 1) / warps;
  quantize_query_kernel<<<unsigned(blocks), warps * 32, 0, stream>>>(q, n_vec, codes, scales);
  return cudaGetLastError();
}

size_t prefill_ws_bytes(int32_t T) { return prefill_layout(T < 1 ? 1 : T).total; }

cudaError_t launch_score_prefill(const uint8_t *idx_rows, int64_t n_rows, const uint8_t *q_codes,
                                 const uint8_t *q_scales, const float *w, int32_t T, int64_t causal_base,
                                 int32_t k, int32_t *out_idx, float *out_score, void *ws, cudaStream_t stream) {
  const PrefillWsLayout L = prefill_layout(T);
  char *base = static_cast<char *>(ws);
  uint16_t *qbf = reinterpret_cast<uint16_t *>(base + L.qbf);
  const uint8_t **rows_arr = reinterpret_cast<const uint8_t **>(base + L.ptrs);
  int64_t *n_arr = reinterpret_cast<int64_t *>(base + L.lens);
  const int64_t elems = int64_t(T) * DS4X_IDX_HEADS * DS4X_IDX_DIM;
  prefill_prep_kernel<<<unsigned((elems + 255) / 256), 256, 0, stream>>>(q_codes, q_scales, T, idx_rows, n_rows,
                                                                         causal_base, qbf, rows_arr, n_arr);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int32_t cap = sms < score_fused_max_ctas() ? sms : score_fused_max_ctas();  // sessions per launch
  const int32_t launches = (T + cap - 1) / cap;
  for (int32_t c0 = 0, li = 0; c0 < T; ++li) {
    const int32_t ns = (T - c0 + (launches - li) - 1) / (launches - li);  // the rest, spread evenly
    ScoreBatch sb{};
    sb.rows_arr = rows_arr + c0;
    sb.n_arr = n_arr + c0;
    sb.n_sess = ns;
    sb.q = qbf + size_t(c0) * DS4X_IDX_HEADS * DS4X_IDX_DIM;
    sb.w = w + size_t(c0) * DS4X_IDX_HEADS;
    sb.k = k;
    sb.out_idx = out_idx + size_t(c0) * k;
    sb.out_score = out_score != nullptr ? out_score + size_t(c0) * k : nullptr;
    e = launch_score_batch(sb, 0, base + L.fused, stream);
    if (e != cudaSuccess) return e;
    c0 += ns;
  }
  return cudaSuccess;
}

}  // namespace ds4x
