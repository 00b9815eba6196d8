// Chunked-prefill CSA score + per-query exact top-k (DS4X README, "Packed
// prefill implementation": batch score/top-k over the packed 68-byte indexer
// rows for a chunk of query tokens).
//
// The prefill scorer is a dense contraction: every query token scores every
// history row it can see.  It runs in two kernels per launch of up to
// 2 x (SMs) query tokens:
//
// * prefill_score_kernel, one CTA per pair of query tokens, streams the key
//   tiles the pair can see once and scores them for both tokens with one
//   block-scaled tcgen05.mma kind::mxf8f6f4 per 32-element K step: M = 128
//   rows, N = 128 = the two tokens' 64 heads, K = 32; A = the E2M1 keys with
//   their own UE8M0 scales (in tensor memory, one code per byte, as in the
//   decode scorer), B = the tokens' E4M3 query codes with their UE8M0 scales
//   per 32 elements, exactly as the query quantiser wrote them (so every
//   product is exact and the tensor core sums in fp32).  Roles: warp 20
//   copies two tiles per bulk copy into a five-stage ring; converter
//   warpgroups 0-1 (tile i: warpgroup i % 2) write each tile's A operand and
//   scale factors; warps 21-23 issue the four MMAs of a tile (tile i by warp
//   21 + i % 3); epilogue warpgroups 2-4 (tile i: warpgroup 2 + i % 3) read the row's 128
//   accumulators and write both tokens' scores
//   s = sum_h w_h * ReLU(acc_h), in fp32, for the rows each token can see.
// * prefill_topk_kernel, one CTA per query token, takes the exact top-k of the
//   token's visible scores (score descending, lower row first): all keys in
//   shared memory when they fit, else histogram passes over the scores (which
//   the score kernel left in L2) that narrow the range of the k-th key, and
//   an index-order pass for a run of equal scores.
#include "ds4x_internal.cuh"
#include "select512.cuh"
#include "tc_ptx.cuh"

namespace ds4x {
namespace {

using namespace ptx;

constexpr int kTileRows = 128;
constexpr int kTileBytes = kTileRows * DS4X_IDX_ROW_BYTES;  // 8704
constexpr int kStageTiles = 2;
constexpr int kStageBytes = kStageTiles * kTileBytes;
constexpr int kStages = 5;
constexpr int kPair = 2;                                  // query tokens per CTA
constexpr int kN = kPair * DS4X_IDX_HEADS;                // 128: B rows = the MMA's N
constexpr int kConvWG = 2;                                // converter warpgroups 0-1 (tile i: i % 2)
constexpr int kEpiWG = 3;                                 // epilogue warpgroups 2-4 (tile i: 2 + i % 3)
constexpr int kProducerWarp = 4 * (kConvWG + kEpiWG);     // 20
constexpr int kMmaWarp = kProducerWarp + 1;               // 21: allocates tensor memory; 21-23 issue MMAs
constexpr int kMmaWarps = 3;
constexpr int kThreads = 32 * (kMmaWarp + kMmaWarps);     // 768
constexpr int kASlots = 3;                                // tensor-memory A ring
constexpr int kDSlots = 3;                                // accumulator ring, 128 columns a slot
// mbarriers indexed by tile modulo a multiple of the ring size and of the
// waiters' rotation, so each waiter waits on every phase of its barriers
constexpr int kAFullBars = 3;                             // afull[i % 3]: waited by issuer i % 3
constexpr int kAEmptyBars = 6;                            // aempty[i % 6]: waited by the converter of tile i + 3
constexpr int kDFullBars = 3;                             // dfull[i % 3]: waited by epilogue WG i % 3
static_assert(kAFullBars % kASlots == 0 && kAFullBars % kMmaWarps == 0, "afull: one issuer per barrier");
static_assert(kAEmptyBars % kASlots == 0 && kAEmptyBars % kConvWG == 0, "aempty: one converter WG per barrier");
static_assert(kDFullBars % kDSlots == 0 && kDFullBars % kEpiWG == 0, "dfull: one epilogue WG per barrier");
static_assert(kStageTiles == kConvWG, "each converter warpgroup takes one tile of every stage");
constexpr uint32_t kDCol0 = 0;                            // D slot d: columns [128 d, 128 d + 128)
constexpr uint32_t kACol0 = kN * kDSlots;                 // 384: A slot a: 32 columns from 384 + 32 a
constexpr uint32_t kSfaCol0 = kACol0 + 32 * kASlots;      // 480: SFA of A slot a: 4 columns
constexpr uint32_t kSfbCol = kSfaCol0 + 4 * kASlots;      // 492: SFB, columns +0 .. +3 (B row n: column n / 32)
constexpr int kTmemCols = 512;
static_assert(kSfbCol % 4 == 0 && kSfbCol + 4 <= uint32_t(kTmemCols), "tensor-memory map");
constexpr uint32_t kLbo = 128, kSbo = 1024;
constexpr uint32_t kIdesc = idesc_mxf8f6f4_e2m1_e4m3(kN);
constexpr unsigned long long kTimeoutNs = 500ull * 1000 * 1000;  // a bounded wait gives up after 0.5 s
constexpr int kMinSmem = 120 * 1024;                      // more than half an SM: one CTA per SM (512 TMEM columns)

__device__ __forceinline__ uint32_t op_offset(int r, int kk) {
  return uint32_t(r >> 3) * kSbo + uint32_t(kk >> 4) * kLbo + uint32_t(r & 7) * 16 + uint32_t(kk & 15);
}

struct __align__(1024) PSmem {
  uint8_t bq[kN * DS4X_IDX_DIM];                // the pair's query codes (B), K-major, converter K order
  uint8_t stage[kStages][kStageBytes];          // raw tile ring, two tiles a stage
  alignas(16) float wq[kN];                     // head weights: token 0's 64, then token 1's
  uint32_t sfb[kN];                             // UE8M0 scale words of the B rows
  unsigned long long full[kStages], empty[kStages];
  unsigned long long afull[kAFullBars], aempty[kAEmptyBars], dfull[kDFullBars];
  int drel[kDSlots];                            // epilogue warps that released the slot so far
  uint32_t tmem_base;
  int abort_flag;
};

struct PrefillArgs {
  const uint8_t *rows;
  int64_t n_rows;
  const uint8_t *q_codes;   // [T][64][128]
  const uint8_t *q_scales;  // [T][64][4]
  const float *w;           // [T][64]
  int64_t causal_base;
  int32_t q0, nq;           // this launch: query tokens q0 .. q0 + nq - 1
  float *scores;            // [nq][score_stride(n_rows)]: token q0 + j in row j
  int32_t k;
  int32_t *out_idx;         // [T][k]
  float *out_score;         // [T][k] or null
};

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded mbarrier wait (as in the decode scorer): on time-out the CTA is
// marked aborted and the workspace status gets DS4X_ETIMEOUT.
__device__ bool wait_bar(PSmem &sm, unsigned long long *bar, uint32_t parity, WsHeader *hdr) {
  const uint32_t b = smem_u32(bar);
  if (mbar_try_wait(b, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(b, parity)) return true;
    if (*reinterpret_cast<volatile int *>(&sm.abort_flag)) return false;
    if (globaltimer() - t0 > kTimeoutNs) {
      atomicExch(&hdr->status, int32_t(DS4X_ETIMEOUT));
      *reinterpret_cast<volatile int *>(&sm.abort_flag) = 1;
      return false;
    }
  }
}

__device__ __forceinline__ int ld_acquire_shared(const int *p) {
  int v;
  asm volatile("ld.acquire.cta.shared::cta.s32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add_shared(int *p, int v) {
  asm volatile("red.release.cta.shared::cta.add.s32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}

__device__ bool wait_seq(PSmem &sm, const int *p, int target, WsHeader *hdr) {
  if (ld_acquire_shared(p) >= target) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    for (int it = 0; it < 64; ++it)
      if (ld_acquire_shared(p) >= target) return true;
    if (*reinterpret_cast<volatile int *>(&sm.abort_flag)) return false;
    if (globaltimer() - t0 > kTimeoutNs) {
      atomicExch(&hdr->status, int32_t(DS4X_ETIMEOUT));
      *reinterpret_cast<volatile int *>(&sm.abort_flag) = 1;
      return false;
    }
  }
}

// Used only while shutting down after a time-out: no bulk copy or MMA may
// still write this CTA's memory when it exits.
__device__ void drain_bar(unsigned long long *bar, uint32_t parity) {
  const uint32_t b = smem_u32(bar);
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(b, parity) && globaltimer() - t0 < kTimeoutNs / 5) {
  }
}

__device__ __forceinline__ void fma_f32x2(float &a0, float &a1, float w0, float w1, float x0, float x1) {
  asm("{\n\t.reg .b64 a, w, x;\n\tmov.b64 a, {%0, %1};\n\tmov.b64 w, {%2, %3};\n\tmov.b64 x, {%4, %5};\n\t"
      "fma.rn.f32x2 a, w, x, a;\n\tmov.b64 {%0, %1}, a;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(w0), "f"(w1), "f"(x0), "f"(x1));
}

// Score rows are n_rows floats rounded up to a multiple of four (16-byte rows).
__host__ __device__ __forceinline__ int64_t score_stride(int64_t n_rows) { return (n_rows + 3) & ~int64_t(3); }

// Rows query token q (absolute) may see: min(n_rows, causal_base + q), at least 0.
__device__ __forceinline__ int64_t visible_rows(const PrefillArgs &a, int64_t q) {
  const int64_t v = a.causal_base + q;
  return v < 0 ? 0 : (v < a.n_rows ? v : a.n_rows);
}

__global__ void __launch_bounds__(kThreads, 1) prefill_score_kernel(PrefillArgs a, WsHeader *__restrict__ hdr) {
  // launched as a programmatic dependent: the previous kernel is complete and
  // visible past this wait; the next kernel's CTAs may be scheduled from now on
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ uint8_t smem_raw[];
  PSmem &sm = *reinterpret_cast<PSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int j0 = kPair * int(blockIdx.x);  // this CTA's tokens: q0 + j0 and q0 + j0 + 1
  int64_t vis[kPair];
#pragma unroll
  for (int j = 0; j < kPair; ++j) vis[j] = j0 + j < a.nq ? visible_rows(a, int64_t(a.q0) + j0 + j) : 0;
  const int64_t n_vis = vis[0] > vis[1] ? vis[0] : vis[1];
  if (n_vis == 0) return;  // uniform across the CTA, before any barrier or allocation
  const int n_tiles = int((n_vis + kTileRows - 1) / kTileRows);
  const int n_copies = (n_tiles + kStageTiles - 1) / kStageTiles;

  // tiles 2j and 2j + 1 -> stage j % kStages, one bulk copy (producer thread)
  auto issue_stage = [&](int j) {
    const int s = j % kStages;
    const int64_t r0 = int64_t(kStageTiles) * j * kTileRows;
    const int64_t left = n_vis - r0;
    const int nr = left < kStageTiles * kTileRows ? int(left) : kStageTiles * kTileRows;
    const uint32_t bytes = uint32_t(nr) * DS4X_IDX_ROW_BYTES;
    const uint32_t bulk = bytes & ~15u;
    const uint8_t *src = a.rows + r0 * DS4X_IDX_ROW_BYTES;
    for (uint32_t b = bulk; b < bytes; b += 4)  // ragged tail
      *reinterpret_cast<uint32_t *>(sm.stage[s] + b) = *reinterpret_cast<const uint32_t *>(src + b);
    mbar_arrive_expect_tx(smem_u32(&sm.full[s]), bulk);
    bulk_g2s(smem_u32(sm.stage[s]), src, bulk, smem_u32(&sm.full[s]));
  };

  // ---- set-up -------------------------------------------------------------
  if (tid == kProducerWarp * 32) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), kStageTiles * kTileRows);  // each converter thread, once per stage
    }
    for (int j = 0; j < kAFullBars; ++j) mbar_init(smem_u32(&sm.afull[j]), kTileRows);
    for (int j = 0; j < kAEmptyBars; ++j) mbar_init(smem_u32(&sm.aempty[j]), 1);
    for (int j = 0; j < kDFullBars; ++j) mbar_init(smem_u32(&sm.dfull[j]), 1);
    for (int j = 0; j < kDSlots; ++j) sm.drel[j] = 0;
    sm.abort_flag = 0;
    fence_mbar_init();
    for (int j = 0; j < kStages && j < n_copies; ++j) issue_stage(j);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&sm.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (tid < 2 * kN) {
    // B row 64 j + h = token j's head h; thread t: row t / 2, elements 64 (t % 2) .. + 63,
    // each group of eight stored even elements first (the converter's K order)
    const int n = tid >> 1, j = n / DS4X_IDX_HEADS, h = n % DS4X_IDX_HEADS, half = tid & 1;
    const bool valid = vis[j] > 0;
    const int64_t qv = int64_t(a.q0) + j0 + j;
    uint4 raw[4] = {};
    if (valid) {
      const uint4 *src =
          reinterpret_cast<const uint4 *>(a.q_codes + (qv * DS4X_IDX_HEADS + h) * DS4X_IDX_DIM + 64 * half);
#pragma unroll
      for (int c = 0; c < 4; ++c) raw[c] = src[c];
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {  // 16 elements: groups of eight (x, y) and (z, w)
      const uint4 v = raw[c];
      const uint4 o = make_uint4(__byte_perm(v.x, v.y, 0x6420), __byte_perm(v.x, v.y, 0x7531),
                                 __byte_perm(v.z, v.w, 0x6420), __byte_perm(v.z, v.w, 0x7531));
      *reinterpret_cast<uint4 *>(sm.bq + op_offset(n, 64 * half + 16 * c)) = o;
    }
    if (half == 0) {
      sm.sfb[n] = valid ? *reinterpret_cast<const uint32_t *>(a.q_scales + (qv * DS4X_IDX_HEADS + h) * 4)
                        : 0x7f7f7f7fu;
      sm.wq[n] = valid ? a.w[qv * DS4X_IDX_HEADS + h] : 0.0f;
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sm.tmem_base;
  if (warp < 4) {
    // B column n's scale factors: lane n % 32 of every sub-partition, column kSfbCol + n / 32
    const uint32_t lanes = uint32_t(32 * warp) << 16;
    tc_st_x4(tmem_base + lanes + kSfbCol, sm.sfb[lane], sm.sfb[32 + lane], sm.sfb[64 + lane], sm.sfb[96 + lane]);
    tc_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == kProducerWarp) {
    // ---- producer -----------------------------------------------------------
    if (lane == 0) {
      int issued = min(kStages, n_copies);
      for (int j = issued; j < n_copies; ++j) {
        if (!wait_bar(sm, &sm.empty[j % kStages], ((j / kStages) - 1) & 1, hdr)) break;
        issue_stage(j);
        issued = j + 1;
      }
      if (*reinterpret_cast<volatile int *>(&sm.abort_flag)) {
        for (int j = max(0, issued - kStages); j < issued; ++j) drain_bar(&sm.full[j % kStages], (j / kStages) & 1);
      }
    }
  } else if (warp >= kMmaWarp) {
    // ---- MMA issuers: warp kMmaWarp + m takes tiles m, m + 3, ... ------------
    if (lane == 0) {
      const uint64_t bdesc = smem_desc_noswizzle(smem_u32(sm.bq), kLbo, kSbo);
      int issued = 0;
      for (int i = warp - kMmaWarp; i < n_tiles; i += kMmaWarps) {
        const int as = i % kASlots, d = i % kDSlots;
        if (!wait_bar(sm, &sm.afull[i % kAFullBars], (i / kAFullBars) & 1, hdr)) break;
        if (i >= kDSlots && !wait_seq(sm, &sm.drel[d], 4 * (i / kDSlots), hdr)) break;
        tc_fence_after();
        mma_mxf8f6f4_ta_k128_1b(tmem_base + kDCol0 + uint32_t(kN * d), tmem_base + kACol0 + uint32_t(32 * as), bdesc,
                                kIdesc, tmem_base + kSfaCol0 + uint32_t(4 * as), tmem_base + kSfbCol);
        tc_commit(smem_u32(&sm.aempty[i % kAEmptyBars]));
        tc_commit(smem_u32(&sm.dfull[i % kDFullBars]));
        issued = i + 1;
      }
      if (*reinterpret_cast<volatile int *>(&sm.abort_flag) && issued > 0) {
        const int i = issued - 1;
        drain_bar(&sm.dfull[i % kDFullBars], (i / kDFullBars) & 1);
      }
    }
  } else if (warp < 4 * kConvWG) {
    // ---- converters: raw row -> A slot (one code per byte) + scale word --------
    const int r = tid & 127;
    const uint32_t lane_base = uint32_t(32 * (warp & 3)) << 16;
    for (int i = warp / 4; i < n_tiles; i += kConvWG) {
      const int j = i / kStageTiles, st = j % kStages, as = i % kASlots;
      wait_bar(sm, &sm.full[st], (j / kStages) & 1, hdr);
      uint32_t wd[17];
      const uint32_t *rp = reinterpret_cast<const uint32_t *>(sm.stage[st] + (i % kStageTiles) * kTileBytes +
                                                               r * DS4X_IDX_ROW_BYTES);
#pragma unroll
      for (int t = 0; t < 17; ++t) wd[t] = rp[t];
      mbar_arrive(smem_u32(&sm.empty[st]));
      // the slot's previous tile i - 3 committed on aempty[(i - 3) % 6], its use (i - 3) / 6 of that barrier
      if (i >= kASlots) wait_bar(sm, &sm.aempty[(i - kASlots) % kAEmptyBars], ((i - kASlots) / kAEmptyBars) & 1, hdr);
      uint32_t av[32];
#pragma unroll
      for (int t = 0; t < 16; ++t) {  // even codes of the group in column 2t, odd ones in 2t + 1, bits 5-2
        av[2 * t] = (wd[t] & 0x0f0f0f0fu) << 2;
        av[2 * t + 1] = (wd[t] & 0xf0f0f0f0u) >> 2;
      }
      tc_st_x32(tmem_base + lane_base + kACol0 + uint32_t(32 * as), av);
      tc_st_x1(tmem_base + lane_base + kSfaCol0 + uint32_t(4 * as + (warp & 3)), wd[16]);
      tc_wait_st();
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.afull[i % kAFullBars]));
    }
  } else {
    // ---- epilogue: 128 accumulators -> two tokens' scores ---------------------
    const int r = tid & 127, role = (warp - 4 * kConvWG) / 4;
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    const float4 *w4 = reinterpret_cast<const float4 *>(sm.wq);
    for (int i = role; i < n_tiles; i += kEpiWG) {
      const int d = i % kDSlots;
      const bool ok = wait_bar(sm, &sm.dfull[i % kDFullBars], (i / kDFullBars) & 1, hdr);
      tc_fence_after();
      const uint32_t d_t = tmem_base + lane_base + kDCol0 + uint32_t(kN * d);
      const int64_t row = int64_t(i) * kTileRows + r;
#pragma unroll
      for (int j = 0; j < kPair; ++j) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t v0[16], v1[16];
          const uint32_t c0 = uint32_t(DS4X_IDX_HEADS * j + 32 * half);
          tc_ld_x16(d_t + c0, v0);
          tc_ld_x16(d_t + c0 + 16u, v1);
          tc_wait_ld();
          if (j == kPair - 1 && half == 1) {  // this warp has read its lanes of the slot
            tc_fence_before();
            __syncwarp();
            if (lane == 0) red_release_add_shared(&sm.drel[d], 1);
          }
#pragma unroll
          for (int g = 0; g < 8; ++g) {  // heads 32 half + 4 g .. + 3 of token j
            const float4 wv = w4[16 * j + 8 * half + g];
            const uint32_t *v = g < 4 ? v0 + 4 * g : v1 + 4 * (g - 4);
            fma_f32x2(acc[0], acc[1], wv.x, wv.y, fmaxf(__uint_as_float(v[0]), 0.0f),
                      fmaxf(__uint_as_float(v[1]), 0.0f));
            fma_f32x2(acc[2], acc[3], wv.z, wv.w, fmaxf(__uint_as_float(v[2]), 0.0f),
                      fmaxf(__uint_as_float(v[3]), 0.0f));
          }
        }
        if (ok && row < vis[j])
          a.scores[int64_t(j0 + j) * score_stride(a.n_rows) + row] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Per-query exact top-k of the scores the score kernel wrote.
// ---------------------------------------------------------------------------
constexpr int kHistBuckets = 4096;
constexpr int kUnroll = 8;  // float4 score loads a thread keeps in flight per pass step

struct __align__(16) TSmem {
  unsigned long long list[kSelCap];      // keys of the boundary range (or all keys when they fit)
  unsigned long long best[DS4X_TOPK_MAX];  // winners collected so far
  unsigned long long tmp[DS4X_TOPK_MAX];   // select_top's output
  unsigned long long sortbuf[2 * DS4X_TOPK_MAX];
  uint32_t hist[kHistBuckets];
  SelShared sel;
  int wsum[kSelThreads / 32];
  uint32_t red_lo[kSelThreads / 32], red_hi[kSelThreads / 32];
  unsigned long long red_key[kSelThreads / 32];
  int bstar, above, bcnt, n_above, n_list;
};

__global__ void __launch_bounds__(kSelThreads, 2) prefill_topk_kernel(PrefillArgs a) {
  // launched as a programmatic dependent: the previous kernel is complete and
  // visible past this wait; the next kernel's CTAs may be scheduled from now on
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ uint8_t tsm_raw[];
  TSmem &sm = *reinterpret_cast<TSmem *>((reinterpret_cast<uintptr_t>(tsm_raw) + 15) & ~uintptr_t(15));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int jq = blockIdx.x;
  const int64_t qv = int64_t(a.q0) + jq;
  const int64_t n = visible_rows(a, qv);
  const int k = a.k;
  const float *__restrict__ s = a.scores + int64_t(jq) * score_stride(a.n_rows);
  int32_t *out_idx = a.out_idx + qv * k;
  float *out_score = a.out_score != nullptr ? a.out_score + qv * k : nullptr;
  const int need0 = int(n < k ? n : k);
  int m = 0;  // winners in best[]
  if (n <= kSelCap) {
#pragma unroll
    for (int q = 0; q < kSelPerThread; ++q) {  // every load in flight at once
      const int i = tid + q * kSelThreads;
      sm.list[i] = i < n ? make_key(s[i], uint32_t(i)) : 0ull;
    }
    bar512();
    if (n > 0) m = select_top(sm.list, int(n), need0, sm.best, sm.hist, sm.sortbuf, sm.sel, tid);
  } else {
    const float4 *__restrict__ s4 = reinterpret_cast<const float4 *>(s);
    const int64_t n4 = (n + 3) / 4;
    int need = need0;
    {
      // A sample of 512 scores (every st-th row), sorted, gives a key T with
      // about twice need keys at or above it; one pass collects those.  When
      // at least need keys are at or above T, the top need are all among them.
      const int64_t st = (n + kSelThreads - 1) / kSelThreads;
      const int ns = int((n + st - 1) / st);
      const unsigned long long sk = tid < ns ? make_key(s[int64_t(tid) * st], uint32_t(int64_t(tid) * st)) : 0ull;
      const unsigned long long srt_s = block_sort512_desc(sk, sm.sortbuf, tid);
      const int64_t want = (2 * int64_t(need) * ns + n - 1) / n + 4;  // sample rank of T (1-based)
      const int rt = int(want < ns ? want : ns) - 1;
      if (tid == rt) sm.red_key[0] = srt_s;
      bar512();
      const unsigned long long t_key = sm.red_key[0];
      // Each warp appends into its own segment of the list with a running
      // count (the same in every lane: no shared atomics, which serialise a
      // pass this long); a segment's unused slots are zero keys (padding,
      // which the selection skips).  A warp with more keys than its segment
      // holds sends the token to the histogram path below.
      constexpr int kSeg = kSelCap / (kSelThreads / 32);  // 576 slots a warp
      unsigned long long *seg = sm.list + warp * kSeg;
      const unsigned lt = (1u << lane) - 1u;
      int wcount = 0;
      for (int64_t t0 = 0; t0 < n4; t0 += kUnroll * kSelThreads) {
        float4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int64_t t4 = t0 + u * kSelThreads + tid;
          v[u] = t4 < n4 ? s4[t4] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int64_t e0 = 4 * (t0 + u * kSelThreads + tid);
          const float x[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const unsigned long long key = e0 + c < n ? make_key(x[c], uint32_t(e0 + c)) : 0ull;
            const bool take = key != 0ull && key >= t_key;
            const unsigned msk = __ballot_sync(0xffffffffu, take);
            const int p = wcount + __popc(msk & lt);
            if (take && p < kSeg) seg[p] = key;
            wcount += __popc(msk);
          }
        }
      }
      for (int i = wcount + lane; i < kSeg; i += 32) seg[i] = 0ull;
      if (lane == 0) sm.wsum[warp] = wcount;
      bar512();
      int cnt = 0;
      bool over = false;
      for (int w = 0; w < kSelThreads / 32; ++w) {
        cnt += sm.wsum[w];
        over = over || sm.wsum[w] > kSeg;
      }
      if (cnt >= need && !over) {
        m = select_top(sm.list, kSelCap, need, sm.best, sm.hist, sm.sortbuf, sm.sel, tid);
        need = 0;
      }
      bar512();
    }
    // Otherwise (rare: the sample fell short, or too many keys share T's
    // score): the range [lo, hi] of ordered score bits still undecided, cut
    // into 4096 buckets per level: the first level is the top 12 bits; each
    // later level is the previous level's boundary bucket.
    uint32_t lo = 0u, hi = ~0u;
    // each level narrows the range by 2^12 (at most three levels: the last
    // has one value per bucket, taken by select_top or the tie pass)
    for (int level = 0; need > 0 && level < 4; ++level) {
      const uint32_t range = hi - lo;
      const int shift = range < uint32_t(kHistBuckets) ? 0 : (32 - __clz(int(range))) - 12;  // range >> shift < 4096
      for (int b = tid; b < kHistBuckets; b += kSelThreads) sm.hist[b] = 0u;
      if (tid == 0) {
        sm.n_above = 0;
        sm.n_list = 0;
      }
      bar512();
      for (int64_t t0 = 0; t0 < n4; t0 += kUnroll * kSelThreads) {
        float4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int64_t t4 = t0 + u * kSelThreads + tid;
          v[u] = t4 < n4 ? s4[t4] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int64_t e0 = 4 * (t0 + u * kSelThreads + tid);
          const float x[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint32_t o = float_to_ordered(x[c]);
            const bool in = e0 + c < n && o >= lo && o <= hi;
            const int b = in ? int((o - lo) >> shift) : -1;
            // one atomic per distinct bucket of the warp (the busy buckets are few)
            const unsigned same = __match_any_sync(0xffffffffu, b);
            if (in && lane == __ffs(same) - 1) atomicAdd(&sm.hist[b], uint32_t(__popc(same)));
          }
        }
      }
      bar512();
      {  // the bucket holding the need-th largest: thread t owns buckets [4095 - 8t - 7, 4095 - 8t]
        const int btop = kHistBuckets - 1 - 8 * tid;
        int local = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) local += int(sm.hist[btop - q]);
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        if (lane == 31) sm.wsum[warp] = incl;
        bar512();
        int before = incl - local;
        for (int w = 0; w < warp; ++w) before += sm.wsum[w];
        if (before < need && before + local >= need) {
          int acc = before;
          for (int q = 0; q < 8; ++q) {
            const int c = int(sm.hist[btop - q]);
            if (acc + c >= need) {
              sm.bstar = btop - q;
              sm.above = acc;
              sm.bcnt = c;
              break;
            }
            acc += c;
          }
        }
        bar512();
      }
      const int bstar = sm.bstar, above = sm.above, bcnt = sm.bcnt;
      const uint32_t fl = lo + (uint32_t(bstar) << shift);
      const uint32_t top = uint32_t(bstar + 1) << shift;                      // may pass hi (or wrap to 0)
      const uint32_t ce = (top - 1u) > (hi - lo) ? hi : lo + (top - 1u);     // the bucket's largest value
      const bool fits = bcnt <= kSelCap;
      // keys above the bucket are winners; the bucket's keys are the candidates for the rest
      for (int64_t t0 = 0; t0 < n4; t0 += kUnroll * kSelThreads) {
        float4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int64_t t4 = t0 + u * kSelThreads + tid;
          v[u] = t4 < n4 ? s4[t4] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {  // warp_append is called by every lane
          const int64_t e0 = 4 * (t0 + u * kSelThreads + tid);
          const float x[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int64_t t = e0 + c;
            const uint32_t o = float_to_ordered(x[c]);
            const bool win = t < n && o > ce && o <= hi;
            const bool cand = fits && t < n && o >= fl && o <= ce;
            const int pw = warp_append(&sm.n_above, win);
            const int pc = warp_append(&sm.n_list, cand);
            if (win) sm.best[m + pw] = (static_cast<unsigned long long>(o) << 32) | uint32_t(~uint32_t(t));
            if (cand) sm.list[pc] = (static_cast<unsigned long long>(o) << 32) | uint32_t(~uint32_t(t));
          }
        }
      }
      bar512();
      m += above;
      need -= above;
      if (fits) {
        const int mm = select_top(sm.list, bcnt, need, sm.tmp, sm.hist, sm.sortbuf, sm.sel, tid);
        for (int i = tid; i < mm; i += kSelThreads) sm.best[m + i] = sm.tmp[i];
        bar512();
        m += mm;
        need = 0;
      } else if (fl == ce) {
        // one score value shared by more rows than fit: the lowest rows win
        int taken = 0;
        for (int64_t t0 = 0; t0 < n && taken < need; t0 += kSelThreads) {
          const int64_t t = t0 + tid;
          const bool p = t < n && float_to_ordered(s[t]) == fl;
          const unsigned msk = __ballot_sync(0xffffffffu, p);
          if (lane == 0) sm.wsum[warp] = __popc(msk);
          bar512();
          int before = 0, total = 0;
          for (int w = 0; w < kSelThreads / 32; ++w) {
            before += w < warp ? sm.wsum[w] : 0;
            total += sm.wsum[w];
          }
          const int rank = taken + before + __popc(msk & ((1u << lane) - 1u));
          if (p && rank < need) sm.best[m + rank] = (static_cast<unsigned long long>(fl) << 32) | uint32_t(~uint32_t(t));
          taken += total;
          bar512();
        }
        m += need;
        need = 0;
        bar512();
      } else {
        lo = fl;  // narrow to the boundary bucket
        hi = ce;
      }
    }
  }
  const unsigned long long srt = block_sort512_desc(tid < m ? sm.best[tid] : 0ull, sm.sortbuf, tid);
  if (tid < k) {
    if (tid < m) {
      out_idx[tid] = key_index(srt);
      if (out_score) out_score[tid] = key_score(srt);
    } else {
      out_idx[tid] = -1;
      if (out_score) out_score[tid] = __uint_as_float(0x7fc00000u);
    }
  }
}

constexpr int kMaxQPerLaunch = 512;  // query tokens whose scores the workspace holds at once

}  // namespace

size_t prefill_ws_bytes(int64_t n_rows, int32_t T) {
  if (n_rows < 1) n_rows = 1;
  if (T < 1) T = 1;
  const int64_t q = T < kMaxQPerLaunch ? T + (T & 1) : kMaxQPerLaunch;
  return kWsHeaderBytes + size_t(q) * size_t(score_stride(n_rows)) * sizeof(float);
}

cudaError_t launch_score_prefill(const uint8_t *idx_rows, int64_t n_rows, const uint8_t *q_codes,
                                 const uint8_t *q_scales, const float *w, int32_t T, int64_t causal_base,
                                 int32_t k, int32_t *out_idx, float *out_score, void *ws, cudaStream_t stream) {
  static std::atomic<uint64_t> smem_a{0}, smem_b{0};
  const int smem_score = int(sizeof(PSmem) + 1024) > kMinSmem ? int(sizeof(PSmem) + 1024) : kMinSmem;
  const int smem_topk = int(sizeof(TSmem) + 16);
  cudaError_t e = set_max_smem_once(prefill_score_kernel, smem_score, smem_a);
  if (e != cudaSuccess) return e;
  if ((e = set_max_smem_once(prefill_topk_kernel, smem_topk, smem_b)) != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  // one wave of pairs per launch, so a launch's scores stay in L2 for its top-k
  int qpl = 2 * sms;
  if (qpl > kMaxQPerLaunch) qpl = kMaxQPerLaunch;
  WsHeader *hdr = static_cast<WsHeader *>(ws);
  PrefillArgs pa{};
  pa.rows = idx_rows;
  pa.n_rows = n_rows;
  pa.q_codes = q_codes;
  pa.q_scales = q_scales;
  pa.w = w;
  pa.causal_base = causal_base;
  pa.scores = reinterpret_cast<float *>(static_cast<char *>(ws) + kWsHeaderBytes);
  pa.k = k;
  pa.out_idx = out_idx;
  pa.out_score = out_score;
  for (int32_t q0 = 0; q0 < T; q0 += qpl) {
    pa.q0 = q0;
    pa.nq = T - q0 < qpl ? T - q0 : qpl;
    if ((e = launch_pdl(prefill_score_kernel, unsigned((pa.nq + kPair - 1) / kPair), kThreads, size_t(smem_score),
                        stream, pa, hdr)) != cudaSuccess)
      return e;
    if ((e = launch_pdl(prefill_topk_kernel, unsigned(pa.nq), kSelThreads, size_t(smem_topk), stream, pa)) !=
        cudaSuccess)
      return e;
  }
  return cudaSuccess;
}

}  // namespace ds4x
