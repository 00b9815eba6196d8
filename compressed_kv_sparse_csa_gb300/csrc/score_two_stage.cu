// Two-stage CSA indexer score + exact top-k (the score-then-select path DS4X
// keeps for short contexts; DS4X README, "CSA score/top-512 fusion").
//
// Stage 1 writes one sortable 64-bit (score, index) key per row; stage 2 is
// a single-CTA most-significant-byte-first radix select that finds the k-th
// largest key exactly, gathers the k keys at or above it and sorts them.
// CUDA cores only; kept as the simple reference path of the library (forced
// with DS4X_SCORER=two_stage) and for small inputs.
#include "ds4x_internal.cuh"

namespace ds4x {
namespace {

constexpr int kScoreWarps = 8;

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(uint32_t(b) << 16);
}

// E2M1 code -> value (magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6).
__device__ __forceinline__ float e2m1_value(uint32_t c) {
  const uint32_t e = (c >> 1) & 3u, m = c & 1u;
  float mag = e == 0 ? 0.5f * float(m) : ldexpf(1.0f + 0.5f * float(m), int(e) - 1);
  return (c & 8u) ? -mag : mag;
}

__global__ void __launch_bounds__(kScoreWarps * 32)
score_keys_kernel(const uint8_t *__restrict__ rows, int64_t n, const uint16_t *__restrict__ q,
                  const float *__restrict__ w, uint64_t *__restrict__ keys) {
  __shared__ float qT[DS4X_IDX_DIM][DS4X_IDX_HEADS];  // transposed: lane-contiguous heads
  __shared__ float krow[kScoreWarps][DS4X_IDX_DIM];
  for (int i = threadIdx.x; i < DS4X_IDX_HEADS * DS4X_IDX_DIM; i += blockDim.x) {
    qT[i % DS4X_IDX_DIM][i / DS4X_IDX_DIM] = bf16_bits_to_float(q[i]);
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float w0 = w[lane], w1 = w[lane + 32];
  for (int64_t r = int64_t(blockIdx.x) * kScoreWarps + warp; r < n;
       r += int64_t(gridDim.x) * kScoreWarps) {
    const uint8_t *row = rows + r * DS4X_IDX_ROW_BYTES;
    const uint32_t b0 = row[2 * lane], b1 = row[2 * lane + 1];
    const float sc = ldexpf(1.0f, int(row[DS4X_IDX_DIM / 2 + (lane >> 3)]) - 127);
    krow[warp][4 * lane + 0] = e2m1_value(b0 & 15u) * sc;
    krow[warp][4 * lane + 1] = e2m1_value(b0 >> 4) * sc;
    krow[warp][4 * lane + 2] = e2m1_value(b1 & 15u) * sc;
    krow[warp][4 * lane + 3] = e2m1_value(b1 >> 4) * sc;
    __syncwarp();
    float d0 = 0.0f, d1 = 0.0f;
#pragma unroll 8
    for (int j = 0; j < DS4X_IDX_DIM; ++j) {
      const float kj = krow[warp][j];
      d0 = fmaf(qT[j][lane], kj, d0);
      d1 = fmaf(qT[j][lane + 32], kj, d1);
    }
    float s = w0 * fmaxf(d0, 0.0f) + w1 * fmaxf(d1, 0.0f);
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) keys[r] = make_key(s, uint32_t(r));
    __syncwarp();
  }
}

constexpr int kSelThreads = 1024;

// Bitonic sort of kTopKMax keys in shared memory, descending.
__device__ void bitonic_sort_desc_512(uint64_t *a) {
  for (int size = 2; size <= DS4X_TOPK_MAX; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      __syncthreads();
      for (int t = threadIdx.x; t < DS4X_TOPK_MAX / 2; t += blockDim.x) {
        const int i = 2 * t - (t & (stride - 1));
        const int j = i + stride;
        const bool desc = ((i & size) == 0);
        const uint64_t x = a[i], y = a[j];
        if ((x < y) == desc) {
          a[i] = y;
          a[j] = x;
        }
      }
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kSelThreads)
select_topk_kernel(const uint64_t *__restrict__ keys, int64_t n, int k,
                   int32_t *__restrict__ out_idx, float *__restrict__ out_score) {
  __shared__ uint32_t hist[256];
  __shared__ uint64_t sel[DS4X_TOPK_MAX];
  __shared__ uint64_t s_prefix, s_mask;
  __shared__ int s_krem;
  __shared__ uint32_t cnt;

  uint64_t prefix = 0, mask = 0;
  if (n > k) {
    int krem = k;
    for (int d = 7; d >= 0; --d) {
      for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
      __syncthreads();
      for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
        const uint64_t key = keys[i];
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> (8 * d)) & 255u], 1u);
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        int cum = 0, b = 255;
        for (; b > 0; --b) {
          if (cum + int(hist[b]) >= krem) break;
          cum += int(hist[b]);
        }
        s_krem = krem - cum;
        s_prefix = prefix | (uint64_t(b) << (8 * d));
        s_mask = mask | (uint64_t(255) << (8 * d));
      }
      __syncthreads();
      prefix = s_prefix;
      mask = s_mask;
      krem = s_krem;
    }
  }
  // prefix is the k-th largest key (keys are unique) or 0 when n <= k
  if (threadIdx.x == 0) cnt = 0;
  for (int i = threadIdx.x; i < DS4X_TOPK_MAX; i += blockDim.x) sel[i] = 0;
  __syncthreads();
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
    const uint64_t key = keys[i];
    if (key >= prefix) {
      const uint32_t p = atomicAdd(&cnt, 1u);
      if (p < DS4X_TOPK_MAX) sel[p] = key;
    }
  }
  bitonic_sort_desc_512(sel);
  const int valid = n < int64_t(k) ? int(n) : k;
  for (int i = threadIdx.x; i < k; i += blockDim.x) {
    if (i < valid) {
      out_idx[i] = key_index(sel[i]);
      if (out_score) out_score[i] = key_score(sel[i]);
    } else {
      out_idx[i] = -1;
      if (out_score) out_score[i] = __uint_as_float(0x7fc00000u);
    }
  }
}

}  // namespace

size_t score_two_stage_ws_bytes(int64_t n_rows) {
  return kWsHeaderBytes + size_t(n_rows) * sizeof(uint64_t);
}

cudaError_t launch_score_two_stage(const uint8_t *idx_rows, int64_t n_rows, const uint16_t *q,
                                   const float *w, int32_t k, int32_t *out_idx, float *out_score,
                                   void *ws, cudaStream_t stream) {
  uint64_t *keys = reinterpret_cast<uint64_t *>(static_cast<char *>(ws) + kWsHeaderBytes);
  int64_t blocks = (n_rows + kScoreWarps - 1) / kScoreWarps;
  if (blocks > 152 * 16) blocks = 152 * 16;
  score_keys_kernel<<<unsigned(blocks), kScoreWarps * 32, 0, stream>>>(idx_rows, n_rows, q, w, keys);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  select_topk_kernel<<<1, kSelThreads, 0, stream>>>(keys, n_rows, k, out_idx, out_score);
  return cudaGetLastError();
}

}  // namespace ds4x
