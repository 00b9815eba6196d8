// Sparse (indexed) decode attention over the selected packed KV rows.
//
// Row layout: DS4X README, "Packed cache ABI" (448 E4M3 codes, 64 FP16 RoPE
// values, 7 UE8M0 scales).  K = V = the dequantised 512-vector, shared by all
// 64 heads (the indexed attention of the DS4X README, "Nsight Systems").
//
// One kernel, no partials in global memory.  The grid is 16 head groups of 4
// heads, each one cluster of 8 CTAs; CTA s of a cluster takes the selected
// rows [64 s, 64 s + 64):
//   1. cp.async gathers each row's bytes (the 16-byte-aligned span holding
//      the 583-byte row, at most 38 chunks) into that row's slot of shared
//      memory, all rows at once, so the gather costs one memory round trip;
//   2. each warp widens its rows in place to fp16: the E4M3 code values
//      (exact in fp16, |x| <= 448) and the FP16 RoPE values; the block
//      scales 2^(e-127) go to a small fp32 table and are applied in fp32
//      (a power of two, so exactly) to per-block partial sums;
//   3. logits for 4 heads x 64 rows, the split's softmax statistics
//      m = max_j l_j, l = sum_j exp(l_j - m) and the unnormalised partial
//      output o = sum_j exp(l_j - m) v_j;
//   4. the cluster combines its 8 partials through distributed shared
//      memory, o_h = sum_s e^(m_s - M) o_s / sum_s e^(m_s - M) l_s: each CTA
//      finishes 1/8 of the group's 4 x 512 outputs, and the LSE M + log L.
// About 95 KB of shared memory per CTA, so two CTAs fit an SM and all 16
// clusters are resident at once.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ds4x_internal.cuh"

namespace ds4x {
namespace {

constexpr int kCluster = 8;                         // CTAs per cluster (row splits)
constexpr int kRows = DS4X_TOPK_MAX / kCluster;     // 64 selected rows per CTA
constexpr int kHg = 4;                              // heads per cluster
constexpr int kGroups = DS4X_ATTN_HEADS / kHg;      // 16 clusters
constexpr int kThreads = 256;
constexpr int kChunks = 38;                         // 16-byte chunks spanning any 583-byte row
constexpr int kSlotBytes = 2 * DS4X_KV_DIM + 32;    // 1056: fp16 row + pad (rows 32 B apart mod 128)
constexpr int kGroupsPerRow = DS4X_KV_DIM / 4;      // 128 four-value column groups
constexpr int kNopeGroups = DS4X_KV_NOPE / 4;       // 112
constexpr int kBlocks = DS4X_KV_DIM / DS4X_KV_BLOCK;  // 8: 7 scaled E4M3 blocks + the RoPE tail
constexpr int kNopeBlocks = DS4X_KV_NOPE / DS4X_KV_BLOCK;  // 7

constexpr size_t kKhBytes = size_t(kRows) * kSlotBytes;                // 67,584
constexpr size_t kQfBytes = size_t(kHg) * DS4X_KV_DIM * sizeof(float);  // 8,192 (then the partial output)
constexpr size_t kPsBytes = size_t(kRows) * kBlocks * kHg * sizeof(float);  // 8,192
constexpr size_t kRedBytes = size_t(kHg) * DS4X_KV_DIM * sizeof(float);  // 8,192
constexpr size_t kSmemBytes = kKhBytes + kQfBytes + kPsBytes + kRedBytes;
static_assert(kRows * kCluster == DS4X_TOPK_MAX, "clusters cover the maximum k");
static_assert(kChunks * 16 <= kSlotBytes && kSlotBytes % 16 == 0, "a row's bytes fit its slot");
static_assert(kHg * DS4X_KV_DIM == kThreads * 8, "one 16-byte query load per thread");
static_assert(kHg * DS4X_KV_DIM == kCluster * kThreads, "one combined output per thread");

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
               "l"(gmem_src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Two E4M3 codes (low byte: the first) -> their fp16 values, packed (low half: the first).
__device__ __forceinline__ uint32_t e4m3x2_to_half2_bits(uint32_t two_codes) {
  uint32_t h2;
  asm("{ .reg .b16 c; cvt.u16.u32 c, %1; cvt.rn.f16x2.e4m3x2 %0, c; }" : "=r"(h2) : "r"(two_codes));
  return h2;
}
__device__ __forceinline__ float2 half2_bits_to_float2(uint32_t bits) {
  return __half22float2(*reinterpret_cast<const __half2 *>(&bits));
}
// 2^(e - 127) for a UE8M0 code e in 0..254 (e = 0 is the subnormal 2^-127).
__device__ __forceinline__ float ue8m0_value(uint32_t e) {
  return e == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(e << 23);
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Exit guard: waits until every CTA of the cluster is done reading peers.
__device__ __forceinline__ void cluster_wait_peers() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Loads a float from the same shared-memory offset in cluster CTA `rank`.
__device__ __forceinline__ float ld_peer(const float *local, uint32_t rank) {
  uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local)), ra;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra));
  return v;
}

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads, 2)
attn_decode_kernel(AttnBatch ab, WsHeader *hdr) {
  // batch item blockIdx.z: its cache, selected rows, query and output
  const int bz = blockIdx.z;
  const uint8_t *__restrict__ kv = ab.kv_arr != nullptr ? ab.kv_arr[bz] : ab.kv;
  const int64_t n_rows = ab.n_arr != nullptr ? ab.n_arr[bz] : ab.n_rows;
  const int k = ab.k;
  const float scale = ab.scale;
  const int32_t *__restrict__ idx = ab.idx + size_t(bz) * k;
  const uint16_t *__restrict__ q = ab.q + size_t(bz) * DS4X_ATTN_HEADS * DS4X_KV_DIM;
  uint16_t *__restrict__ out = ab.out + size_t(bz) * DS4X_ATTN_HEADS * DS4X_KV_DIM;
  float *__restrict__ lse = ab.lse != nullptr ? ab.lse + size_t(bz) * DS4X_ATTN_HEADS : nullptr;
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned char *Kh = smem;                                                // [64][1056]: raw, then fp16
  float *Qf = reinterpret_cast<float *>(smem + kKhBytes);                 // [4][512]
  float *Opart = Qf;                                                       // [4][512], after the logits
  float4 *Ps = reinterpret_cast<float4 *>(smem + kKhBytes + kQfBytes);    // [64][8] x 4 heads
  float *red = reinterpret_cast<float *>(smem + kKhBytes + kQfBytes + kPsBytes);  // [4][512]
  __shared__ __align__(16) float Pt[kRows][kHg];   // logits, then exp(l - m)
  __shared__ float sc[kRows][kBlocks];             // block scales (1 for the RoPE tail)
  __shared__ float ml[2 * kHg];                    // m[4], l[4] of this split
  __shared__ int64_t rows_s[kRows];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x, hg = blockIdx.y;

  if (tid < kRows) {
    const int j = split * kRows + tid;
    int64_t r = -1;
    if (j < k) {
      r = idx[j];
      if (r < -1 || r >= n_rows) {
        atomicExch(&hdr->status, int32_t(DS4X_EDEVICE));
        r = -1;
      }
    }
    rows_s[tid] = r;
  }
  {
    const uint4 qb = reinterpret_cast<const uint4 *>(q + size_t(hg) * kHg * DS4X_KV_DIM)[tid];
    const uint32_t w[4] = {qb.x, qb.y, qb.z, qb.w};
    float4 *dst = reinterpret_cast<float4 *>(Qf) + 2 * tid;
    dst[0] = make_float4(__uint_as_float(w[0] << 16), __uint_as_float(w[0] & 0xffff0000u),
                         __uint_as_float(w[1] << 16), __uint_as_float(w[1] & 0xffff0000u));
    dst[1] = make_float4(__uint_as_float(w[2] << 16), __uint_as_float(w[2] & 0xffff0000u),
                         __uint_as_float(w[3] << 16), __uint_as_float(w[3] & 0xffff0000u));
  }
  __syncthreads();

  // 1. gather: chunk c of row rr is bytes [a0 + 16 c, a0 + 16 c + 16), a0 the
  // row's start rounded down to 16; chunks past the row's end are skipped and
  // a chunk crossing the end of the buffer is read byte by byte.
  const int64_t total = n_rows * DS4X_KV_ROW_BYTES;
  for (int id = tid; id < kRows * kChunks; id += kThreads) {
    const int rr = id / kChunks, c = id - rr * kChunks;
    const int64_t r = rows_s[rr];
    if (r < 0) continue;
    const int64_t start = r * DS4X_KV_ROW_BYTES;
    const int64_t src = (start & ~int64_t(15)) + 16 * c;
    if (src >= start + DS4X_KV_ROW_BYTES) continue;
    unsigned char *dst = Kh + rr * kSlotBytes + 16 * c;
    if (src + 16 <= total) {
      cp_async16(dst, kv + src);
    } else {
      for (int b = 0; b < 16; ++b)
        if (src + b < total) dst[b] = kv[src + b];
    }
  }
  cp_async_wait_all();
  __syncthreads();

  // 2. widen in place: warp w owns rows 8w..8w+7.  Every lane reads all its
  // inputs of a row (column groups lane + 32 q, four values each) before the
  // warp overwrites the slot with the row's fp16 values.  Skipped rows
  // become zeros.
#pragma unroll 1
  for (int i = 0; i < kRows / (kThreads / 32); ++i) {
    const int rr = warp * (kRows / (kThreads / 32)) + i;
    const int64_t r = rows_s[rr];
    unsigned char *slot = Kh + rr * kSlotBytes;
    uint2 *hrow = reinterpret_cast<uint2 *>(slot);
    if (r < 0) {
#pragma unroll
      for (int q4 = 0; q4 < kGroupsPerRow / 32; ++q4) hrow[lane + 32 * q4] = make_uint2(0u, 0u);
      if (lane < kBlocks) sc[rr][lane] = 0.f;
      continue;
    }
    const int off = int((r * DS4X_KV_ROW_BYTES) & 15);
    const uint32_t *w32 = reinterpret_cast<const uint32_t *>(slot);
    const int sh = (off & 3) * 8;
    uint32_t in[kGroupsPerRow / 32][2];
#pragma unroll
    for (int q4 = 0; q4 < kGroupsPerRow / 32; ++q4) {
      const int g = lane + 32 * q4;
      if (g < kNopeGroups) {  // 4 E4M3 codes
        const int p = off + 4 * g;
        in[q4][0] = __funnelshift_r(w32[p >> 2], w32[(p >> 2) + 1], sh);
        in[q4][1] = 0u;
      } else {  // 4 FP16 values
        const int p = off + DS4X_KV_NOPE + 8 * (g - kNopeGroups);
        const uint32_t a = w32[p >> 2], b = w32[(p >> 2) + 1], c = w32[(p >> 2) + 2];
        in[q4][0] = __funnelshift_r(a, b, sh);
        in[q4][1] = __funnelshift_r(b, c, sh);
      }
    }
    float scale_b = 1.f;
    if (lane < kNopeBlocks) scale_b = ue8m0_value(slot[off + DS4X_KV_NOPE + 2 * DS4X_KV_ROPE + lane]);
    __syncwarp();
#pragma unroll
    for (int q4 = 0; q4 < kGroupsPerRow / 32; ++q4) {
      const int g = lane + 32 * q4;
      if (g < kNopeGroups) {
        hrow[g] = make_uint2(e4m3x2_to_half2_bits(in[q4][0] & 0xffffu), e4m3x2_to_half2_bits(in[q4][0] >> 16));
      } else {
        hrow[g] = make_uint2(in[q4][0], in[q4][1]);
      }
    }
    if (lane < kBlocks) sc[rr][lane] = scale_b;
  }
  __syncthreads();

  // 3a. logits: thread (row tid / 4, column quarter tid % 4), 4 heads; the
  // sum over each 64-column block is scaled by the block's scale.
  {
    const int r = tid >> 2, jq = tid & 3;
    const uint2 *K2 = reinterpret_cast<const uint2 *>(Kh + r * kSlotBytes);
    const float4 *Q4 = reinterpret_cast<const float4 *>(Qf);
    float a[kHg] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int b = 0; b < kBlocks; ++b) {
      float part[kHg] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ii = 0; ii < 4; ++ii) {
        const int c = jq + 16 * b + 4 * ii;
        const uint2 hv = K2[c];
        const float2 x01 = half2_bits_to_float2(hv.x), x23 = half2_bits_to_float2(hv.y);
#pragma unroll
        for (int h = 0; h < kHg; ++h) {
          const float4 y = Q4[h * kGroupsPerRow + c];
          part[h] = fmaf(y.x, x01.x, part[h]);
          part[h] = fmaf(y.y, x01.y, part[h]);
          part[h] = fmaf(y.z, x23.x, part[h]);
          part[h] = fmaf(y.w, x23.y, part[h]);
        }
      }
      const float s = sc[r][b];
#pragma unroll
      for (int h = 0; h < kHg; ++h) a[h] = fmaf(s, part[h], a[h]);
    }
#pragma unroll
    for (int h = 0; h < kHg; ++h) {
      a[h] += __shfl_xor_sync(0xffffffffu, a[h], 1);
      a[h] += __shfl_xor_sync(0xffffffffu, a[h], 2);
    }
    if (jq == 0) {
      const bool valid = rows_s[r] >= 0;
#pragma unroll
      for (int h = 0; h < kHg; ++h) Pt[r][h] = valid ? a[h] * scale : -INFINITY;
    }
  }
  __syncthreads();

  // 3b. split softmax statistics: warp h < 4 takes head h, rows lane, lane + 32.
  if (warp < kHg) {
    const int h = warp;
    const float l0 = Pt[lane][h], l1 = Pt[lane + 32][h];
    float m = fmaxf(l0, l1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float p0 = m == -INFINITY ? 0.f : expf(l0 - m);
    const float p1 = m == -INFINITY ? 0.f : expf(l1 - m);
    Pt[lane][h] = p0;
    Pt[lane + 32][h] = p1;
    float s = p0 + p1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) {
      ml[h] = m;
      ml[kHg + h] = s;
    }
  }
  __syncthreads();
  // weights per (row, block): exp(l - m) times the block scale
  for (int e = tid; e < kRows * kBlocks; e += kThreads) {
    const int r = e / kBlocks, b = e % kBlocks;
    const float s = sc[r][b];
    const float4 p = *reinterpret_cast<const float4 *>(&Pt[r][0]);
    Ps[e] = make_float4(p.x * s, p.y * s, p.z * s, p.w * s);
  }
  __syncthreads();

  // 3c. partial output: thread (column group tid % 128, row half tid / 128).
  {
    const int c = tid & (kGroupsPerRow - 1), half = tid >> 7, b = c >> 4;
    float4 acc[kHg];
#pragma unroll
    for (int h = 0; h < kHg; ++h) acc[h] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int i = 0; i < kRows / 2; ++i) {
      const int r = half * (kRows / 2) + i;
      const uint2 hv = reinterpret_cast<const uint2 *>(Kh + r * kSlotBytes)[c];
      const float2 v01 = half2_bits_to_float2(hv.x), v23 = half2_bits_to_float2(hv.y);
      const float4 p = Ps[r * kBlocks + b];
      const float ph[kHg] = {p.x, p.y, p.z, p.w};
#pragma unroll
      for (int h = 0; h < kHg; ++h) {
        acc[h].x = fmaf(ph[h], v01.x, acc[h].x);
        acc[h].y = fmaf(ph[h], v01.y, acc[h].y);
        acc[h].z = fmaf(ph[h], v23.x, acc[h].z);
        acc[h].w = fmaf(ph[h], v23.y, acc[h].w);
      }
    }
    float4 *red4 = reinterpret_cast<float4 *>(red);
    float4 *O4 = reinterpret_cast<float4 *>(Opart);
    if (half == 1) {
#pragma unroll
      for (int h = 0; h < kHg; ++h) red4[h * kGroupsPerRow + c] = acc[h];
    }
    __syncthreads();
    if (half == 0) {
#pragma unroll
      for (int h = 0; h < kHg; ++h) {
        const float4 o = red4[h * kGroupsPerRow + c];
        O4[h * kGroupsPerRow + c] =
            make_float4(acc[h].x + o.x, acc[h].y + o.y, acc[h].z + o.z, acc[h].w + o.w);
      }
    }
  }

  // 4. combine the cluster's 8 partials through distributed shared memory.
  cluster_sync();
  {
    const int e = int(cluster_rank()) * kThreads + tid;
    const int h = e / DS4X_KV_DIM, d = e % DS4X_KV_DIM;
    float ms[kCluster], ls[kCluster], os[kCluster];
#pragma unroll
    for (int s = 0; s < kCluster; ++s) {
      ms[s] = ld_peer(&ml[h], uint32_t(s));
      ls[s] = ld_peer(&ml[kHg + h], uint32_t(s));
      os[s] = ld_peer(&Opart[h * DS4X_KV_DIM + d], uint32_t(s));
    }
    float M = -INFINITY;
#pragma unroll
    for (int s = 0; s < kCluster; ++s) M = fmaxf(M, ms[s]);
    float L = 0.f, o = 0.f;
#pragma unroll
    for (int s = 0; s < kCluster; ++s) {
      const float f = ms[s] == -INFINITY ? 0.f : expf(ms[s] - M);
      L = fmaf(f, ls[s], L);
      o = fmaf(f, os[s], o);
    }
    const int head = hg * kHg + h;
    out[size_t(head) * DS4X_KV_DIM + d] = __bfloat16_as_ushort(__float2bfloat16_rn(L > 0.f ? o / L : 0.f));
    if (lse != nullptr && d == 0) lse[head] = L > 0.f ? M + logf(L) : -INFINITY;
  }
  cluster_wait_peers();  // peers may still be reading this CTA's partials
}

}  // namespace

size_t attn_decode_ws_bytes(int32_t) { return kWsHeaderBytes; }

cudaError_t launch_attn_batch(const AttnBatch &ab, int batch, void *ws, cudaStream_t stream) {
  static std::atomic<uint64_t> smem_set{0};
  cudaError_t e = set_max_smem_once(attn_decode_kernel, int(kSmemBytes), smem_set);
  if (e != cudaSuccess) return e;
  attn_decode_kernel<<<dim3(kCluster, kGroups, batch), kThreads, kSmemBytes, stream>>>(ab,
                                                                                      static_cast<WsHeader *>(ws));
  return cudaGetLastError();
}

cudaError_t launch_attn_decode(const uint8_t *kv_rows, int64_t n_rows, const int32_t *idx,
                               int32_t k, const uint16_t *q, float scale, uint16_t *out,
                               float *lse, void *ws, cudaStream_t stream) {
  AttnBatch ab{};
  ab.kv = kv_rows;
  ab.n_rows = n_rows;
  ab.idx = idx;
  ab.k = k;
  ab.q = q;
  ab.scale = scale;
  ab.out = out;
  ab.lse = lse;
  return launch_attn_batch(ab, 1, ws, stream);
}

}  // namespace ds4x
