// Sparse (indexed) decode attention over selected packed KV rows, split over
// row ranges (flash-decoding) with a log-sum-exp combine.
//
// Row layout: DS4X README, "Packed cache ABI" (448 E4M3 codes, 64 FP16 RoPE
// values, 7 UE8M0 scales).  K = V = the dequantised 512-vector, shared by all
// 64 heads.  Split kernel: one CTA per (32-row range, 16-head group) gathers
// and dequantises its rows into shared memory, computes the range's softmax
// statistics (m, l) and unnormalised output; the combine kernel rescales the
// partials by exp(m_s - M) and writes bf16 outputs and the LSE.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ds4x_internal.cuh"

namespace ds4x {
namespace {

constexpr int kRows = 32;   // rows per split (one per lane)
constexpr int kHeads = 16;  // heads per CTA
constexpr int kThreads = 256;
constexpr int kVStride = DS4X_KV_DIM + 1;  // odd stride: conflict-free V[lane][d]
constexpr size_t kSmemBytes =
    (size_t(kRows) * kVStride + size_t(kHeads) * DS4X_KV_DIM + kHeads * kRows) * sizeof(float);

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(uint32_t(b) << 16);
}

// E4M3FN code -> value (finite codes only are ever written).
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  const float mag = e == 0 ? ldexpf(float(m), -9) : ldexpf(1.0f + float(m) * 0.125f, int(e) - 7);
  return (c & 0x80u) ? -mag : mag;
}

struct Partials {
  float *ml;  // [splits][64][2]: running max and sum of exp
  float *o;   // [splits][64][512]: unnormalised output
};

__device__ __forceinline__ Partials partials(void *ws, int splits) {
  char *base = static_cast<char *>(ws) + kWsHeaderBytes;
  Partials p;
  p.ml = reinterpret_cast<float *>(base);
  p.o = reinterpret_cast<float *>(base + size_t(splits) * DS4X_ATTN_HEADS * 2 * sizeof(float));
  return p;
}

__global__ void __launch_bounds__(kThreads)
attn_split_kernel(const uint8_t *__restrict__ kv, int64_t n_rows, const int32_t *__restrict__ idx,
                  int k, const uint16_t *__restrict__ q, float scale, void *ws) {
  extern __shared__ float smem[];
  float *V = smem;                         // [kRows][kVStride]
  float *Q = V + kRows * kVStride;         // [kHeads][512]
  float *P = Q + kHeads * DS4X_KV_DIM;     // [kHeads][kRows]
  __shared__ int64_t rows_s[kRows];

  const int split = blockIdx.x, hg = blockIdx.y, splits = gridDim.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  WsHeader *hdr = static_cast<WsHeader *>(ws);

  if (threadIdx.x < kRows) {
    const int j = split * kRows + threadIdx.x;
    int64_t r = -1;
    if (j < k) {
      r = idx[j];
      if (r < -1 || r >= n_rows) {
        atomicExch(&hdr->status, int32_t(DS4X_EDEVICE));
        r = -1;
      }
    }
    rows_s[threadIdx.x] = r;
  }
  for (int i = threadIdx.x; i < kHeads * DS4X_KV_DIM; i += kThreads) {
    Q[i] = bf16_bits_to_float(q[size_t(hg) * kHeads * DS4X_KV_DIM + i]);
  }
  __syncthreads();

  // gather + dequantise: warp w handles rows w, w+8, ...
  for (int rr = warp; rr < kRows; rr += kThreads / 32) {
    const int64_t r = rows_s[rr];
    float *dst = V + rr * kVStride;
    if (r < 0) {
      for (int d = lane; d < DS4X_KV_DIM; d += 32) dst[d] = 0.0f;
      continue;
    }
    const uint8_t *src = kv + r * DS4X_KV_ROW_BYTES;
    for (int d = lane; d < DS4X_KV_NOPE; d += 32) {
      const int sb = src[DS4X_KV_NOPE + 2 * DS4X_KV_ROPE + d / DS4X_KV_BLOCK];
      dst[d] = e4m3_value(src[d]) * ldexpf(1.0f, sb - 127);
    }
    for (int d = lane; d < DS4X_KV_ROPE; d += 32) {
      const uint16_t hb = uint16_t(src[DS4X_KV_NOPE + 2 * d]) | uint16_t(src[DS4X_KV_NOPE + 2 * d + 1] << 8);
      dst[DS4X_KV_NOPE + d] = __half2float(__ushort_as_half(hb));
    }
  }
  __syncthreads();

  Partials part = partials(ws, splits);
  // logits and softmax statistics: warp w handles heads 2w, 2w+1; lane = row
  const bool valid = rows_s[lane] >= 0;
  for (int hh = 0; hh < kHeads / (kThreads / 32); ++hh) {
    const int h = warp * (kHeads / (kThreads / 32)) + hh;
    const float *qh = Q + h * DS4X_KV_DIM;
    const float *vr = V + lane * kVStride;
    float acc = 0.0f;
#pragma unroll 8
    for (int d = 0; d < DS4X_KV_DIM; ++d) acc = fmaf(qh[d], vr[d], acc);
    const float l = valid ? acc * scale : -INFINITY;
    float m = l;
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float p = (valid && m != -INFINITY) ? expf(l - m) : 0.0f;
    float sum = p;
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    P[h * kRows + lane] = p;
    if (lane == 0) {
      const int head = hg * kHeads + h;
      part.ml[(size_t(split) * DS4X_ATTN_HEADS + head) * 2 + 0] = m;
      part.ml[(size_t(split) * DS4X_ATTN_HEADS + head) * 2 + 1] = sum;
    }
  }
  __syncthreads();

  // unnormalised output: thread t owns columns t and t + 256 of every head
  for (int dd = 0; dd < DS4X_KV_DIM / kThreads; ++dd) {
    const int d = threadIdx.x + dd * kThreads;
    float acc[kHeads];
#pragma unroll
    for (int h = 0; h < kHeads; ++h) acc[h] = 0.0f;
    for (int r = 0; r < kRows; ++r) {
      const float v = V[r * kVStride + d];
#pragma unroll
      for (int h = 0; h < kHeads; ++h) acc[h] = fmaf(P[h * kRows + r], v, acc[h]);
    }
#pragma unroll
    for (int h = 0; h < kHeads; ++h) {
      const int head = hg * kHeads + h;
      part.o[(size_t(split) * DS4X_ATTN_HEADS + head) * DS4X_KV_DIM + d] = acc[h];
    }
  }
}

__global__ void __launch_bounds__(256)
attn_combine_kernel(int splits, uint16_t *__restrict__ out, float *__restrict__ lse, void *ws) {
  const int head = blockIdx.x;
  Partials part = partials(ws, splits);
  float M = -INFINITY;
  for (int s = 0; s < splits; ++s) M = fmaxf(M, part.ml[(size_t(s) * DS4X_ATTN_HEADS + head) * 2]);
  float L = 0.0f;
  for (int s = 0; s < splits; ++s) {
    const float m = part.ml[(size_t(s) * DS4X_ATTN_HEADS + head) * 2];
    if (m != -INFINITY) L += expf(m - M) * part.ml[(size_t(s) * DS4X_ATTN_HEADS + head) * 2 + 1];
  }
  for (int d = threadIdx.x; d < DS4X_KV_DIM; d += blockDim.x) {
    float o = 0.0f;
    for (int s = 0; s < splits; ++s) {
      const float m = part.ml[(size_t(s) * DS4X_ATTN_HEADS + head) * 2];
      if (m != -INFINITY) o += expf(m - M) * part.o[(size_t(s) * DS4X_ATTN_HEADS + head) * DS4X_KV_DIM + d];
    }
    const float v = (L > 0.0f) ? o / L : 0.0f;
    out[size_t(head) * DS4X_KV_DIM + d] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  }
  if (lse != nullptr && threadIdx.x == 0) lse[head] = (L > 0.0f) ? M + logf(L) : -INFINITY;
}

}  // namespace

size_t attn_decode_ws_bytes(int32_t k) {
  const size_t splits = size_t((k + kRows - 1) / kRows);
  return kWsHeaderBytes + splits * DS4X_ATTN_HEADS * (2 + DS4X_KV_DIM) * sizeof(float);
}

cudaError_t launch_attn_decode(const uint8_t *kv_rows, int64_t n_rows, const int32_t *idx,
                               int32_t k, const uint16_t *q, float scale, uint16_t *out,
                               float *lse, void *ws, cudaStream_t stream) {
  static std::atomic<uint64_t> smem_set{0};
  cudaError_t e = set_max_smem_once(attn_split_kernel, int(kSmemBytes), smem_set);
  if (e != cudaSuccess) return e;
  const int splits = (k + kRows - 1) / kRows;
  attn_split_kernel<<<dim3(splits, DS4X_ATTN_HEADS / kHeads), kThreads, kSmemBytes, stream>>>(
      kv_rows, n_rows, idx, k, q, scale, ws);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  attn_combine_kernel<<<DS4X_ATTN_HEADS, 256, 0, stream>>>(splits, out, lse, ws);
  return cudaGetLastError();
}

}  // namespace ds4x
