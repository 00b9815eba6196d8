// Sparse (indexed) decode attention over the selected packed KV rows.
//
// Row layout: DS4X README, "Packed cache ABI" (448 E4M3 codes, 64 FP16 RoPE
// values, 7 UE8M0 scales).  K = V = the dequantised 512-vector, shared by all
// 64 heads (the indexed attention of the DS4X README, "Nsight Systems").
//
// One kernel, no partials in global memory.  The grid is 64 / HG head groups
// of HG heads (HG = 4, 8 or 16: the fewest heads whose grid fits one
// resident wave, else 16), each one cluster of 8 CTAs; CTA s of a cluster
// takes the selected rows [64 s, 64 s + 64):
//   1. cp.async gathers each row's bytes (the 16-byte-aligned span holding
//      the 583-byte row, at most 38 chunks) into that row's slot of shared
//      memory, all rows at once, so the gather costs one memory round trip;
//   2. each warp widens its rows in place to fp16: the E4M3 code values
//      (exact in fp16, |x| <= 448) and the FP16 RoPE values; the block
//      scales 2^(e-127) go to a small fp32 table;
//   3. logits for HG heads x 64 rows on the tensor cores (mma.sync
//      m16n8k16, fp16 operands, fp32 sums; each head's bf16 query scaled
//      by a power of two into fp16, exact for every value within 2^24 of
//      the head's largest), each 64-column partial sum scaled by the
//      row's block scale in fp32; the split's softmax statistics
//      m = max_j l_j, l = sum_j exp(l_j - m); the unnormalised partial
//      output o = sum_j exp(l_j - m) v_j on the tensor cores too, per
//      64-column block with the weights exp(l_j - m) s_jb / max_j s_jb as
//      fp16 pairs hi + lo (22 significant bits; the ratio an exact power
//      of two);
//   4. the cluster combines its 8 partials through distributed shared
//      memory, o_h = sum_s e^(m_s - M) o_s / sum_s e^(m_s - M) l_s: each CTA
//      finishes 1/8 of the group's HG x 512 outputs, and the LSE M + log L.
// About 106 KB (HG = 4), 99 KB (HG = 8) or 107 KB (HG = 16) of shared memory
// per CTA, so two CTAs fit an SM: from HG = 8 on, the partial output reuses
// the row slots and the logit halves the weight buffer, and HG = 16 makes
// its weights and output MMAs in two passes of 8 heads.  The n = 8 side of
// every MMA is 8 of the group's heads: with HG = 4 half of it is zero rows.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ds4x_internal.cuh"

namespace ds4x {
namespace {

constexpr int kCluster = 8;                         // CTAs per cluster (row splits)
constexpr int kRows = DS4X_TOPK_MAX / kCluster;     // 64 selected rows per CTA
constexpr int kThreads = 256;
constexpr int kChunks = 38;                         // 16-byte chunks spanning any 583-byte row
constexpr int kSlotBytes = 2 * DS4X_KV_DIM + 16;    // 1040: fp16 row + pad (8 rows cover all 32 banks)
constexpr int kGroupsPerRow = DS4X_KV_DIM / 4;      // 128 four-value column groups
constexpr int kNopeGroups = DS4X_KV_NOPE / 4;       // 112
constexpr int kBlocks = DS4X_KV_DIM / DS4X_KV_BLOCK;  // 8: 7 scaled E4M3 blocks + the RoPE tail
constexpr int kNopeBlocks = DS4X_KV_NOPE / DS4X_KV_BLOCK;  // 7

// Tensor-core operands (mma.sync m16n8k16, fp16 in, fp32 accumulate): the
// query as B of the logits (8 rows: the HG heads, then zero rows), the
// softmax weights as B of the output (per 64-column block, 8 rows of 64
// weights, as an fp16 pair hi + lo).
constexpr int kQhStride = 2 * DS4X_KV_DIM + 16;     // 1040 bytes per query row
constexpr int kPbStride = 2 * kRows + 16;           // 144 bytes per weight row
constexpr size_t kKhBytes = size_t(kRows) * kSlotBytes;                     // 66,560
constexpr size_t kPbBytes = size_t(2) * kBlocks * 8 * kPbStride;            // 18,432: hi and lo parts

// Partial-output rows, in floats: 512 + 4, so the MMA fragments' stores (4
// heads x 8 columns per warp) hit 32 banks and every row stays 16-byte aligned.
constexpr int kOpStride = DS4X_KV_DIM + 4;

// Per head-group size: HG = 4 keeps the partial output (8 KB) and the logit
// halves (2 KB) in their own space; HG >= 8 puts the partial output (16 or
// 32 KB) over the row slots once the output MMAs are done and the logit
// halves (4 or 8 KB) over the weight buffer before the weights are written.
template <int HG>
struct Cfg {
  static_assert(HG == 4 || HG == 8 || HG == 16, "4, 8 or 16 heads per cluster");
  static constexpr int kGroups = DS4X_ATTN_HEADS / HG;
  static constexpr bool kShared = HG >= 8;
  static constexpr int kNT = HG > 8 ? HG / 8 : 1;  // 8-head n tiles of the logits, passes of the output
  static constexpr int kPH = HG > 8 ? 8 : HG;      // heads per output pass
  static constexpr size_t kQhBytes = size_t(8 * kNT) * kQhStride;  // query rows: the heads, then zero rows
  static constexpr size_t kOpBytes = size_t(HG) * kOpStride * sizeof(float);
  static constexpr size_t kRedBytes = size_t(2) * kRows * HG * sizeof(float);
  static constexpr size_t kSmemBytes =
      kShared ? kKhBytes + kQhBytes + kPbBytes : kKhBytes + kQhBytes + kPbBytes + kOpBytes + kRedBytes;
  static_assert(kSmemBytes + 8 * 1024 <= 113 * 1024, "two CTAs per SM (with up to 8 KB of static shared memory)");
  static_assert(!kShared || (kOpBytes <= kKhBytes && kRedBytes <= kPbBytes), "reused buffers fit");
};
static_assert(kRows * kCluster == DS4X_TOPK_MAX, "clusters cover the maximum k");
static_assert(kChunks * 16 <= kSlotBytes && kSlotBytes % 16 == 0, "a row's bytes fit its slot");
static_assert(4 * DS4X_KV_DIM == kThreads * 8, "one 16-byte query load per thread per 4 heads");
static_assert(4 * DS4X_KV_DIM == kCluster * kThreads, "one combined output per thread per 4 heads");
static_assert(kThreads / 32 == kBlocks && kRows == 4 * 16, "warp w: output block w; logits: 4 row tiles x 2 block halves");

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
// 2^(e - 127) for a UE8M0 code e in 0..254 (e = 0 is the subnormal 2^-127).
__device__ __forceinline__ float ue8m0_value(uint32_t e) {
  return e == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(e << 23);
}

// Warp-level tensor-core helpers (fp16 operands from shared memory).
__device__ __forceinline__ void ldsm_x4(const void *p, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
}
__device__ __forceinline__ void ldsm_x4_trans(const void *p, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
}
__device__ __forceinline__ void ldsm_x2(const void *p, uint32_t (&r)[2]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
}
// d += a (16x16, row) * b (16x8, col), fp16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
               "{%0,%1,%2,%3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// 2^e for |e| <= 126 (so that 2^-e is a normal float too).
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float(uint32_t(e + 127) << 23); }
// The query scale exponent of a head whose largest |value| is m: m 2^e lies
// in [2^14, 2^15) (clamped to |e| <= 126; 0 for an all-zero head).
__device__ __forceinline__ int query_exp(float m) {
  if (!(m > 0.f)) return 0;
  const int e = 14 - (int((__float_as_uint(m) >> 23) & 0xffu) - 127);
  return e < -126 ? -126 : (e > 126 ? 126 : e);
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
// Loads N consecutive floats (16-byte aligned for N = 4, 8 for N = 2) from
// the same shared-memory offset in cluster CTA `rank`.
template <int N>
__device__ __forceinline__ void ld_peer_vec(const float *local, uint32_t rank, float (&v)[N]) {
  uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local)), ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  if constexpr (N == 4) {
    asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]) : "r"(ra));
  } else if constexpr (N == 2) {
    asm volatile("ld.shared::cluster.v2.f32 {%0,%1}, [%2];" : "=f"(v[0]), "=f"(v[1]) : "r"(ra));
  } else {
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v[0]) : "r"(ra));
  }
}
__device__ __forceinline__ float ld_peer(const float *local, uint32_t rank) {
  uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local)), ra;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra));
  return v;
}

// With ab.out_f32 set, item b's normalised output goes there in fp32 (for a
// finalize) instead of to ab.out.
template <int HG>
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads, 2)
attn_decode_kernel(AttnBatch ab, WsHeader *hdr) {
  using C = Cfg<HG>;
  constexpr int kQLoads = HG / 4;  // 16-byte query loads (and combined outputs) per thread
  // batch item blockIdx.z: its cache, selected rows, query and output
  const int bz = blockIdx.z;
  const uint8_t *__restrict__ kv = ab.kv_arr != nullptr ? ab.kv_arr[bz] : ab.kv;
  const int64_t n_rows = ab.n_arr != nullptr ? ab.n_arr[bz] : ab.n_rows;
  const int k = ab.k;
  const float scale = ab.scale;
  const int32_t *__restrict__ idx = ab.idx + size_t(bz) * k;
  const uint16_t *__restrict__ q = ab.q + (ab.q_shared ? size_t(0) : size_t(bz) * DS4X_ATTN_HEADS * DS4X_KV_DIM);
  // fp32 output (window + sparse items) for a finalize, else bf16
  const bool f32_out = ab.out_f32 != nullptr;
  uint16_t *__restrict__ out = f32_out ? nullptr : ab.out + size_t(bz) * DS4X_ATTN_HEADS * DS4X_KV_DIM;
  float *__restrict__ lse = ab.lse != nullptr ? ab.lse + size_t(bz) * DS4X_ATTN_HEADS : nullptr;
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned char *Kh = smem;                                   // [64][1040]: raw row, then fp16
  unsigned char *Qh = smem + kKhBytes;                        // [8][1040]: scaled query, fp16
  unsigned char *Pb = Qh + C::kQhBytes;                       // [hi, lo][8 blocks][8][144]: weights, fp16
  float *Opart = C::kShared ? reinterpret_cast<float *>(Kh)                 // [HG][516]
                            : reinterpret_cast<float *>(Pb + kPbBytes);
  float *red = C::kShared ? reinterpret_cast<float *>(Pb) : Opart + HG * kOpStride;  // [2][64][HG]
  // odd row strides: a warp reading one column over 32 rows hits 32 banks
  __shared__ float Pt[kRows][HG + 1];              // logits, then exp(l - m)
  __shared__ float sc[kRows][kBlocks + 1];         // block scales (1 for the RoPE tail)
  __shared__ float ml[2 * HG];                     // m[HG], l[HG] of this split
  __shared__ float qmax[kQLoads][kThreads / 32];   // per load and warp: largest |q| of its head
  __shared__ float sbmax[kBlocks];                 // per block: largest row scale
  __shared__ float sbinv[kBlocks];                 // ... and its reciprocal (exact: a power of two)
  __shared__ float fw[HG][kCluster];               // combine weights e^(m_s - M) per head and split
  __shared__ float fl[HG];                         // ... and their sum L per head
  __shared__ int64_t rows_s[kRows];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x, hg = blockIdx.y;

  // the zero rows HG..7 of the query operand and of every weight block
  if (HG < 8) {
    constexpr int kZero = (HG < 8 ? 8 - HG : 1) * kPbStride / 16;  // 16-byte words of a block's zero rows
    for (int i = tid; i < (8 - HG) * kQhStride / 16; i += kThreads)
      reinterpret_cast<uint4 *>(Qh + HG * kQhStride)[i] = make_uint4(0u, 0u, 0u, 0u);
    for (int i = tid; i < 2 * kBlocks * kZero; i += kThreads) {
      const int blk = i / kZero, j = i % kZero;  // blk: part * 8 + block
      reinterpret_cast<uint4 *>(Pb + blk * 8 * kPbStride + HG * kPbStride)[j] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  // Launched as a programmatic dependent of the previous kernel (the scorer
  // that wrote idx): everything above reads no input; wait for it here.  Its
  // own dependents (a finalize, a copy of the output) may be scheduled from
  // now on; they wait for its completion.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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
  // query: load j of thread t holds 8 values of head 4 j + t / 64 (two warps per head)
  float qv[kQLoads][8];
#pragma unroll
  for (int j = 0; j < kQLoads; ++j) {
    const uint4 qb = reinterpret_cast<const uint4 *>(q + size_t(hg) * HG * DS4X_KV_DIM)[j * kThreads + tid];
    const uint32_t w[4] = {qb.x, qb.y, qb.z, qb.w};
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      qv[j][2 * i] = __uint_as_float(w[i] << 16);
      qv[j][2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
      m = fmaxf(m, fmaxf(fabsf(qv[j][2 * i]), fabsf(qv[j][2 * i + 1])));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) qmax[j][warp] = m;
  }
  __syncthreads();
  // head h's largest |q|: load h / 4, warps 2 (h % 4) and 2 (h % 4) + 1
  auto head_qmax = [&](int h) { return fmaxf(qmax[h >> 2][2 * (h & 3)], qmax[h >> 2][2 * (h & 3) + 1]); };

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
  // while the rows are in flight: head h's query scaled by 2^e_h so that its
  // largest value lies in [2^14, 2^15): every bf16 value in that range is
  // exact in fp16, and the logits are scaled back by 2^-e_h (exactly)
#pragma unroll
  for (int j = 0; j < kQLoads; ++j) {
    const int hq = 4 * j + (tid >> 6);
    const float s = pow2f(query_exp(head_qmax(hq)));
    __half hv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) hv[i] = __float2half_rn(qv[j][i] * s);
    *reinterpret_cast<uint4 *>(Qh + hq * kQhStride + 16 * (tid & 63)) = *reinterpret_cast<const uint4 *>(hv);
  }
  cp_async_wait_all();
  __syncthreads();

  // 2. widen in place: warp w owns rows 8w..8w+7, four at a time.  Every lane
  // reads all its inputs of the four rows (column groups lane + 32 q, four
  // values each) before the warp overwrites the slots with fp16 values.
  // Skipped rows become zeros with scale 0.
#pragma unroll 1
  for (int i = 0; i < kRows / (kThreads / 32); i += 4) {
    uint32_t in[4][kGroupsPerRow / 32][2];
    float scale_b[4];
    int64_t rv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int rr = warp * (kRows / (kThreads / 32)) + i + u;
      rv[u] = rows_s[rr];
      const unsigned char *slot = Kh + rr * kSlotBytes;
      const int off = rv[u] >= 0 ? int((rv[u] * DS4X_KV_ROW_BYTES) & 15) : 0;
      const uint32_t *w32 = reinterpret_cast<const uint32_t *>(slot);
      const int sh = (off & 3) * 8;
#pragma unroll
      for (int q4 = 0; q4 < kGroupsPerRow / 32; ++q4) {
        const int g = lane + 32 * q4;
        if (g < kNopeGroups) {  // 4 E4M3 codes
          const int p = off + 4 * g;
          in[u][q4][0] = __funnelshift_r(w32[p >> 2], w32[(p >> 2) + 1], sh);
          in[u][q4][1] = 0u;
        } else {  // 4 FP16 values
          const int p = off + DS4X_KV_NOPE + 8 * (g - kNopeGroups);
          const uint32_t a = w32[p >> 2], b = w32[(p >> 2) + 1], c = w32[(p >> 2) + 2];
          in[u][q4][0] = __funnelshift_r(a, b, sh);
          in[u][q4][1] = __funnelshift_r(b, c, sh);
        }
      }
      scale_b[u] = 1.f;
      if (lane < kNopeBlocks) scale_b[u] = ue8m0_value(slot[off + DS4X_KV_NOPE + 2 * DS4X_KV_ROPE + lane]);
    }
    __syncwarp();
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int rr = warp * (kRows / (kThreads / 32)) + i + u;
      uint2 *hrow = reinterpret_cast<uint2 *>(Kh + rr * kSlotBytes);
      const bool valid = rv[u] >= 0;
#pragma unroll
      for (int q4 = 0; q4 < kGroupsPerRow / 32; ++q4) {
        const int g = lane + 32 * q4;
        uint2 hv;
        if (!valid) hv = make_uint2(0u, 0u);
        else if (g < kNopeGroups)
          hv = make_uint2(e4m3x2_to_half2_bits(in[u][q4][0] & 0xffffu), e4m3x2_to_half2_bits(in[u][q4][0] >> 16));
        else
          hv = make_uint2(in[u][q4][0], in[u][q4][1]);
        hrow[g] = hv;
      }
      if (lane < kBlocks) sc[rr][lane] = valid ? scale_b[u] : 0.f;
    }
  }
  __syncthreads();

  // 3a. logits on the tensor cores: warp w takes rows 16 (w % 4) .. + 16 and
  // blocks 4 (w / 4) .. + 4; each block's 64-column partial sum is scaled by
  // the row's block scale.  C fragment: rows g and g + 8 (g = lane / 4),
  // heads 8 n + 2 (lane % 4) and + 1 of n tile n (heads HG..7 are the zero
  // rows); each key fragment serves every n tile.
  {
    const int mt = warp & 3, bh = warp >> 2, g = lane >> 2, hc = 2 * (lane & 3);
    const int r0 = 16 * mt + g, r1 = r0 + 8;
    const unsigned char *a_base = Kh + (16 * mt + (lane & 7) + ((lane >> 3) & 1) * 8) * kSlotBytes + ((lane >> 4) & 1) * 16;
    const unsigned char *b_base = Qh + (lane & 7) * kQhStride + ((lane >> 3) & 1) * 16;
    float tot[C::kNT][4];
#pragma unroll
    for (int nt = 0; nt < C::kNT; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) tot[nt][j] = 0.f;
#pragma unroll
    for (int bi = 0; bi < 4; ++bi) {
      const int blk = 4 * bh + bi;
      float acc[C::kNT][4];
#pragma unroll
      for (int nt = 0; nt < C::kNT; ++nt)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[nt][j] = 0.f;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const int k0 = DS4X_KV_BLOCK * blk + 16 * ks;  // columns k0 .. k0 + 15
        uint32_t af[4];
        ldsm_x4(a_base + 2 * k0, af);
#pragma unroll
        for (int nt = 0; nt < C::kNT; ++nt) {
          uint32_t bf[2];
          ldsm_x2(b_base + 8 * nt * kQhStride + 2 * k0, bf);
          mma_16816(acc[nt], af, bf);
        }
      }
      const float s0 = sc[r0][blk], s1 = sc[r1][blk];
#pragma unroll
      for (int nt = 0; nt < C::kNT; ++nt) {
        tot[nt][0] = fmaf(s0, acc[nt][0], tot[nt][0]);
        tot[nt][1] = fmaf(s0, acc[nt][1], tot[nt][1]);
        tot[nt][2] = fmaf(s1, acc[nt][2], tot[nt][2]);
        tot[nt][3] = fmaf(s1, acc[nt][3], tot[nt][3]);
      }
    }
    float *rb = red + bh * kRows * HG;
#pragma unroll
    for (int nt = 0; nt < C::kNT; ++nt) {
      const int h = 8 * nt + hc;
      if (h < HG) {
        rb[r0 * HG + h] = tot[nt][0];
        rb[r0 * HG + h + 1] = tot[nt][1];
        rb[r1 * HG + h] = tot[nt][2];
        rb[r1 * HG + h + 1] = tot[nt][3];
      }
    }
  }
  __syncthreads();
  for (int e = tid; e < kRows * HG; e += kThreads) {
    const int r = e / HG, h = e % HG;
    const float unscale = pow2f(-query_exp(head_qmax(h)));
    const float l = (red[r * HG + h] + red[kRows * HG + r * HG + h]) * unscale;
    Pt[r][h] = rows_s[r] >= 0 ? l * scale : -INFINITY;
  }
  __syncthreads();

  // 3b. split softmax statistics: warp w takes heads w, w + 8, ... (< HG),
  // rows lane, lane + 32; the warps without a head (every warp, for HG >= 8,
  // after its heads) find each block's largest row scale.
  for (int h = warp; h < HG; h += kThreads / 32) {
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
      ml[HG + h] = s;
    }
  }
  if (HG >= 8 || warp >= HG) {
    constexpr int kPer = kBlocks / (kThreads / 32 - (HG >= 8 ? 0 : HG));  // blocks per warp: 1 or 2
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int blk = kPer * (HG >= 8 ? warp : warp - HG) + j;
      float m = fmaxf(sc[lane][blk], sc[lane + 32][blk]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) {
        sbmax[blk] = m;
        sbinv[blk] = m > 0.f ? 1.0f / m : 0.f;
      }
    }
  }
  __syncthreads();
  // 3c/3d, per pass of up to 8 heads (HG = 16: two passes over one weight
  // buffer; the accumulators stay in registers until the row slots are done).
  // 3c. output weights per block: exp(l - m) times the row's block scale over
  // the block's largest (a power of two at most 1, exact), as fp16 hi + lo
  // (hi the rounded weight, lo the rounded remainder: 22 significant bits).
  // 3d. partial output on the tensor cores: warp w takes block w (columns
  // 64 w .. + 64, four 16-column tiles); A = the rows' values transposed, B =
  // the block's weights; the block's largest scale goes back on at the end.
  const int g = lane >> 2, hc = 2 * (lane & 3);
  float acc[C::kNT][4][4];
#pragma unroll
  for (int pass = 0; pass < C::kNT; ++pass) {
    if (pass > 0) __syncthreads();  // the previous pass's MMAs have read the weights
    {
      // thread t: row t % 64, blocks 2 (t / 64) and + 1; the row's scale
      // ratios once, each head's exp(l - m) once
      static_assert(2 * (kThreads / kRows) == kBlocks, "two blocks per thread");
      const int r = tid % kRows, b0 = 2 * (tid / kRows);
      float ratio[2];
#pragma unroll
      for (int j = 0; j < 2; ++j)
        ratio[j] = sbmax[b0 + j] > 0.f ? sc[r][b0 + j] * sbinv[b0 + j] : 0.f;  // exact: powers of two
#pragma unroll
      for (int hl = 0; hl < C::kPH; ++hl) {
        const float pe = Pt[r][C::kPH * pass + hl];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int blk = b0 + j;
          const float w = pe * ratio[j];
          const __half hi = __float2half_rn(w);
          const __half lo = __float2half_rn(w - __half2float(hi));
          reinterpret_cast<__half *>(Pb + (blk * 8 + hl) * kPbStride)[r] = hi;
          reinterpret_cast<__half *>(Pb + ((kBlocks + blk) * 8 + hl) * kPbStride)[r] = lo;
        }
      }
    }
    __syncthreads();
    const int blk = warp;
#pragma unroll
    for (int t = 0; t < 4; ++t)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[pass][t][j] = 0.f;
    const unsigned char *pb = Pb + blk * 8 * kPbStride + (lane & 7) * kPbStride + ((lane >> 3) & 1) * 16;
#pragma unroll
    for (int ks = 0; ks < kRows / 16; ++ks) {
      uint32_t bh[2], bl[2];
      ldsm_x2(pb + 32 * ks, bh);
      ldsm_x2(pb + kBlocks * 8 * kPbStride + 32 * ks, bl);
      const unsigned char *a_base =
          Kh + (16 * ks + (lane & 7) + ((lane >> 4) & 1) * 8) * kSlotBytes + ((lane >> 3) & 1) * 16;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        uint32_t af[4];
        ldsm_x4_trans(a_base + 2 * (DS4X_KV_BLOCK * blk + 16 * t), af);
        mma_16816(acc[pass][t], af, bh);
        mma_16816(acc[pass][t], af, bl);
      }
    }
  }
  {
    const int blk = warp;
    const float smax = sbmax[blk];
    if (C::kShared) __syncthreads();  // the partial output goes over the row slots the other warps read
#pragma unroll
    for (int pass = 0; pass < C::kNT; ++pass) {
      const int h = C::kPH * pass + hc;
      if (hc < C::kPH) {
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int d0 = DS4X_KV_BLOCK * blk + 16 * t + g;
          Opart[h * kOpStride + d0] = acc[pass][t][0] * smax;
          Opart[(h + 1) * kOpStride + d0] = acc[pass][t][1] * smax;
          Opart[h * kOpStride + d0 + 8] = acc[pass][t][2] * smax;
          Opart[(h + 1) * kOpStride + d0 + 8] = acc[pass][t][3] * smax;
        }
      }
    }
  }

  // 4. combine the cluster's 8 partials through distributed shared memory:
  // warp 0 turns the 8 splits' (m, l) into each head's weights
  // f_s = e^(m_s - M), the sum L = sum_s f_s l_s and the LSE; then every
  // thread reads its 8 partial outputs and divides sum_s f_s o_s by L.
  cluster_sync();
  if (warp < HG / 4) {
    // lane = split s (8) x head h (4 per warp)
    const int s = lane & (kCluster - 1), h = 4 * warp + (lane >> 3);
    const float ms = ld_peer(&ml[h], uint32_t(s)), ls = ld_peer(&ml[HG + h], uint32_t(s));
    float M = ms;
#pragma unroll
    for (int o = 1; o < kCluster; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float f = ms == -INFINITY ? 0.f : expf(ms - M);
    float L = f * ls;
#pragma unroll
    for (int o = 1; o < kCluster; o <<= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    fw[h][s] = f;
    if (s == 0) fl[h] = L;
    if (s == 0 && lse != nullptr && cluster_rank() == 0) lse[hg * HG + h] = L > 0.f ? M + logf(L) : -INFINITY;
  }
  __syncthreads();
  {
    // HG / 4 consecutive outputs of one head per thread: one vector load per peer
    constexpr int kV = kQLoads;
    const int e = (int(cluster_rank()) * kThreads + tid) * kV;
    const int h = e / DS4X_KV_DIM, d = e % DS4X_KV_DIM;
    float os[kCluster][kV];
#pragma unroll
    for (int s = 0; s < kCluster; ++s) ld_peer_vec<kV>(&Opart[h * kOpStride + d], uint32_t(s), os[s]);
    const float L = fl[h];
    float of[kV];
    uint16_t ob[kV];
#pragma unroll
    for (int v = 0; v < kV; ++v) {
      float o = 0.f;
#pragma unroll
      for (int s = 0; s < kCluster; ++s) o = fmaf(fw[h][s], os[s][v], o);
      of[v] = L > 0.f ? o / L : 0.f;
      ob[v] = __bfloat16_as_ushort(__float2bfloat16_rn(of[v]));
    }
    if (f32_out) {  // the item's normalised output in fp32, for the finalize
      float *fdst = ab.out_f32 + (size_t(bz) * DS4X_ATTN_HEADS + size_t(hg * HG + h)) * DS4X_KV_DIM + d;
      if (kV == 4) {
        *reinterpret_cast<float4 *>(fdst) = make_float4(of[0], of[kV > 1 ? 1 : 0], of[kV > 2 ? 2 : 0], of[kV > 3 ? 3 : 0]);
      } else if (kV == 2) {
        *reinterpret_cast<float2 *>(fdst) = make_float2(of[0], of[kV > 1 ? 1 : 0]);
      } else {
        fdst[0] = of[0];
      }
    } else if (kV == 4) {
      uint16_t *dst = out + size_t(hg * HG + h) * DS4X_KV_DIM + d;
      *reinterpret_cast<uint2 *>(dst) = make_uint2(uint32_t(ob[0]) | (uint32_t(ob[kV > 1 ? 1 : 0]) << 16),
                                                   uint32_t(ob[kV > 2 ? 2 : 0]) | (uint32_t(ob[kV > 3 ? 3 : 0]) << 16));
    } else if (kV == 2) {
      uint16_t *dst = out + size_t(hg * HG + h) * DS4X_KV_DIM + d;
      *reinterpret_cast<uint32_t *>(dst) = uint32_t(ob[0]) | (uint32_t(ob[kV > 1 ? 1 : 0]) << 16);
    } else {
      out[size_t(hg * HG + h) * DS4X_KV_DIM + d] = ob[0];
    }
  }
  cluster_wait_peers();  // peers may still be reading this CTA's partials
}

}  // namespace

size_t attn_decode_ws_bytes(int32_t) { return kWsHeaderBytes; }

template <int HG>
cudaError_t launch_attn_hg(const AttnBatch &ab, int batch, void *ws, cudaStream_t stream) {
  using C = Cfg<HG>;
  static std::atomic<uint64_t> smem_set{0};
  cudaError_t e = set_max_smem_once(attn_decode_kernel<HG>, int(C::kSmemBytes), smem_set);
  if (e != cudaSuccess) return e;
  // Programmatic stream serialisation: the CTAs may start while the previous
  // kernel finishes (it lets them go from its tail); the kernel waits for it
  // before reading anything.
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(kCluster, C::kGroups, unsigned(batch));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_decode_kernel<HG>, ab, static_cast<WsHeader *>(ws));
}

cudaError_t launch_attn_batch(const AttnBatch &ab, int batch, void *ws, cudaStream_t stream) {
  // the fewest heads per cluster whose grid fits one wave (two CTAs per SM):
  // the most CTAs, the shortest latency; beyond that 16, a quarter of the
  // CTAs of 4 heads for about twice the MMAs each (no zero rows)
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int64_t wave = 2 * int64_t(sms);
  if (int64_t(batch) * kCluster * Cfg<4>::kGroups <= wave) return launch_attn_hg<4>(ab, batch, ws, stream);
  if (int64_t(batch) * kCluster * Cfg<8>::kGroups <= wave) return launch_attn_hg<8>(ab, batch, ws, stream);
  return launch_attn_hg<16>(ab, batch, ws, stream);
}

namespace {

// The dense attention's workspace: the status header, then per item i the
// LSEs [i][64] and the normalised outputs [i][64][512], fp32.
struct DenseWsLayout {
  int32_t rows_per_item, items;
  size_t lse, o, total;
};
DenseWsLayout dense_layout(int64_t n_rows) {
  DenseWsLayout L{};
  L.rows_per_item = dense_rows_per_item(n_rows);
  L.items = int32_t((n_rows + L.rows_per_item - 1) / L.rows_per_item);
  L.lse = kWsHeaderBytes;
  L.o = L.lse + ((size_t(L.items) * DS4X_ATTN_HEADS * sizeof(float) + 255) / 256) * 256;
  L.total = L.o + size_t(L.items) * DS4X_ATTN_HEADS * DS4X_KV_DIM * sizeof(float);
  return L;
}

constexpr int kFinDims = 128;                      // output dims per block
constexpr int kFinParts = 4;                       // item groups per block
constexpr int kFinThreads = kFinDims * kFinParts;  // 512
constexpr int kFinSplit = DS4X_KV_DIM / kFinDims;  // blocks per head

// The split-KV combine over T items, block (h, c): head h, dims 128 c ..
// 128 c + 127.  With M the largest item LSE, o = sum_t e^(lse_t - M) o_t /
// sum_t e^(lse_t - M) (o_t each item's normalised output), lse = M + log sum_t
// e^(lse_t - M).  Thread (p, d) sums items p, p + 4, ... of dim d (eight loads
// in flight), the four sums are added in a fixed order.  Item weights in
// shared memory (T floats).  Launched as a programmatic dependent of the
// items' attention: it waits for it first.
__global__ void __launch_bounds__(kFinThreads) dense_finalize_kernel(const float *__restrict__ lse_part,
                                                                     const float *__restrict__ o_part, int T,
                                                                     uint16_t *__restrict__ out,
                                                                     float *__restrict__ lse) {
  extern __shared__ float fsh[];  // [T]: e^(lse_t - M)
  __shared__ float red[kFinThreads / 32];
  __shared__ float osum[kFinParts][kFinDims];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int h = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = kFinThreads / 32;
  float m = -INFINITY;
  for (int t = tid; t < T; t += kFinThreads) m = fmaxf(m, lse_part[size_t(t) * DS4X_ATTN_HEADS + h]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) red[warp] = m;
  __syncthreads();
  float M = red[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) M = fmaxf(M, red[w]);
  __syncthreads();  // red is reused below
  float sum = 0.f;
  for (int t = tid; t < T; t += kFinThreads) {
    const float l = lse_part[size_t(t) * DS4X_ATTN_HEADS + h];
    const float f = (l == -INFINITY || M == -INFINITY) ? 0.f : expf(l - M);
    fsh[t] = f;
    sum += f;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane == 0) red[warp] = sum;
  __syncthreads();
  float L = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) L += red[w];
  const int dd = tid % kFinDims, part = tid / kFinDims;
  const int d = kFinDims * blockIdx.y + dd;
  const float *op = o_part + size_t(h) * DS4X_KV_DIM + d;
  constexpr size_t kItem = size_t(DS4X_ATTN_HEADS) * DS4X_KV_DIM;  // floats between items
  float o = 0.f;
  int t = part;
  for (; t + 7 * kFinParts < T; t += 8 * kFinParts) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = op[size_t(t + u * kFinParts) * kItem];
#pragma unroll
    for (int u = 0; u < 8; ++u) o = fmaf(fsh[t + u * kFinParts], v[u], o);
  }
  for (; t < T; t += kFinParts) o = fmaf(fsh[t], op[size_t(t) * kItem], o);
  osum[part][dd] = o;
  __syncthreads();
  if (part == 0) {
    const float tot = (osum[0][dd] + osum[1][dd]) + (osum[2][dd] + osum[3][dd]);
    out[size_t(h) * DS4X_KV_DIM + d] = __bfloat16_as_ushort(__float2bfloat16_rn(L > 0.f ? tot / L : 0.f));
  }
  if (blockIdx.y == 0 && tid == 0 && lse != nullptr) lse[h] = L > 0.f ? M + logf(L) : -INFINITY;
}

cudaError_t launch_finalize(const float *lse_part, const float *o_part, int T, uint16_t *out, float *lse,
                            cudaStream_t stream) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(DS4X_ATTN_HEADS, kFinSplit);
  cfg.blockDim = dim3(kFinThreads);
  cfg.dynamicSmemBytes = size_t(T) * sizeof(float);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];  // programmatic stream serialisation (the kernel waits first thing)
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, dense_finalize_kernel, lse_part, o_part, T, out, lse);
}

}  // namespace

int32_t dense_rows_per_item(int64_t n_rows) {
  const int64_t per = (n_rows + 128 * 256 - 1) / (128 * 256);  // 128-row tiles per item
  return int32_t(128 * (per < 1 ? 1 : (per > 4 ? 4 : per)));
}

size_t dense_attn_ws_bytes(int64_t n_rows) { return dense_layout(n_rows < 1 ? 1 : n_rows).total; }

namespace {

// The window + sparse attention's workspace: the status header, the two
// items' LSEs [2][64] and normalised outputs [2][64][512] (fp32), their index
// lists [2][512], row-array pointers [2] and row counts [2].
struct WindowWsLayout {
  size_t lse, o, idx, ptrs, lens, total;
};
constexpr WindowWsLayout window_layout() {
  WindowWsLayout L{};
  L.lse = kWsHeaderBytes;
  L.o = L.lse + 2 * DS4X_ATTN_HEADS * sizeof(float);
  L.idx = L.o + size_t(2) * DS4X_ATTN_HEADS * DS4X_KV_DIM * sizeof(float);
  L.ptrs = L.idx + 2 * DS4X_TOPK_MAX * sizeof(int32_t);
  L.lens = L.ptrs + 2 * sizeof(void *);
  L.total = L.lens + 2 * sizeof(int64_t);
  return L;
}

// Item 0: the caller's k selected rows; item 1: the window, ring slots
// ring_pos, ring_pos - 1, ... (mod DS4X_RING_ROWS), w of them.
__global__ void __launch_bounds__(DS4X_TOPK_MAX) window_prep_kernel(const uint8_t *kv_rows, int64_t n_rows,
                                                                    const int32_t *__restrict__ idx, int32_t k,
                                                                    const uint8_t *ring_rows, int32_t ring_pos,
                                                                    int32_t w, int32_t *__restrict__ idx2,
                                                                    const uint8_t **ptrs, int64_t *lens) {
  // launched as a programmatic dependent: the previous kernel (the scorer that
  // wrote idx, or the previous call's finalize, which reads this workspace) is
  // complete past this wait
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int j = threadIdx.x;
  idx2[j] = j < k ? idx[j] : -1;
  idx2[DS4X_TOPK_MAX + j] = j < w ? (ring_pos - j + DS4X_RING_ROWS) % DS4X_RING_ROWS : -1;
  if (j == 0) {
    ptrs[0] = kv_rows;
    ptrs[1] = ring_rows;
    lens[0] = n_rows;
    lens[1] = DS4X_RING_ROWS;
  }
}

}  // namespace

size_t window_attn_ws_bytes() { return window_layout().total; }

cudaError_t launch_window_attn(const uint8_t *kv_rows, int64_t n_rows, const int32_t *idx, int32_t k,
                               const uint8_t *ring_rows, int32_t ring_pos, int32_t w, const uint16_t *q, float scale,
                               uint16_t *out, float *lse, void *ws, cudaStream_t stream) {
  constexpr WindowWsLayout L = window_layout();
  char *base = static_cast<char *>(ws);
  float *lse_part = reinterpret_cast<float *>(base + L.lse);
  float *o_part = reinterpret_cast<float *>(base + L.o);
  int32_t *idx2 = reinterpret_cast<int32_t *>(base + L.idx);
  const uint8_t **ptrs = reinterpret_cast<const uint8_t **>(base + L.ptrs);
  int64_t *lens = reinterpret_cast<int64_t *>(base + L.lens);
  cudaError_t e = launch_pdl(window_prep_kernel, 1u, unsigned(DS4X_TOPK_MAX), 0, stream, kv_rows, n_rows, idx, k,
                             ring_rows, ring_pos, w, idx2, ptrs, lens);
  if (e != cudaSuccess) return e;
  AttnBatch ab{};
  ab.kv_arr = ptrs;
  ab.n_arr = lens;
  ab.idx = idx2;
  ab.k = DS4X_TOPK_MAX;
  ab.scale = scale;
  ab.q = q;
  ab.q_shared = true;
  ab.lse = lse_part;
  ab.out_f32 = o_part;
  e = launch_attn_batch(ab, 2, ws, stream);
  if (e != cudaSuccess) return e;
  return launch_finalize(lse_part, o_part, 2, out, lse, stream);
}

cudaError_t launch_dense_attn(const uint8_t *kv_rows, int64_t n_rows, const uint16_t *q, float scale, uint16_t *out,
                              float *lse, void *ws, cudaStream_t stream) {
  if (n_rows < 1 || n_rows > kDenseMaxTiles * DS4X_TOPK_MAX) return cudaErrorInvalidValue;
  const DenseWsLayout L = dense_layout(n_rows);
  char *base = static_cast<char *>(ws);
  float *lse_part = reinterpret_cast<float *>(base + L.lse);
  float *o_part = reinterpret_cast<float *>(base + L.o);
  cudaError_t e = launch_attn_dense_items(kv_rows, n_rows, L.rows_per_item, L.items, q, scale, o_part, lse_part, ws,
                                          stream);
  if (e != cudaSuccess) return e;
  return launch_finalize(lse_part, o_part, L.items, out, lse, stream);
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
