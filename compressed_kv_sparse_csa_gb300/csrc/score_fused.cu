// Fused CSA indexer score + exact top-k on the fifth-generation tensor cores.
//
// DS4X README, "Optimization details" / "CSA score/top-512 fusion": the
// scorer reads the packed 68-byte MXFP4 rows directly, every scorer CTA keeps
// an exact local top-512 of sortable (score, index) keys, and the local lists
// are merged into the exact top-512 without materialising the score array.
// This is a GB300 design of that method:
//
//  * one persistent CTA per SM streams a contiguous range of 128-row tiles
//    (8,704 bytes each) from HBM with 1-D bulk copies into a ring of shared-
//    memory stages (warp 16);
//  * four warpgroups (thread = row) dequantise their tile: each byte of two
//    E2M1 codes goes through the hardware e2m1x2 -> f16x2 converter, then
//    one f16x2 multiply applies the block's scale relative to the row's
//    largest block scale 2^e_ref; the 64 words are written straight into
//    tensor memory as the A operand of the MMA (no shared-memory round trip);
//  * warp 17 issues tcgen05.mma kind::f16 (M = 128 rows, N = 64 heads,
//    K = 16, eight per tile) with the query as the B operand in shared
//    memory; fp32 accumulators land in tensor memory;
//  * the same warpgroup reads its rows' 64 accumulators back and forms
//    s = 2^e_ref * sum_h (w_h / 2^(a_h+1)) * (acc_h + |acc_h|), which is
//    sum_h w_h * ReLU(q_h . k) exactly up to fp32 rounding;
//  * every key stays in shared memory; after the stream an exact range-
//    bucketed selection keeps the CTA's top 512; the last CTA to finish
//    merges the CTAs' top-16 sets, fetching more from any CTA whose 16th key
//    beats the tentative cut (so the result is exact for any input), sorts
//    the winners and writes the outputs.
//
// The query is held in fp16 with a per-head power-of-two scale 2^a_h that
// puts the head's largest |q| in [2^15, 2^16): every bf16 element within
// 2^-32 of its head's maximum converts exactly; the keys are exact in fp16
// whenever a row's block exponents differ by at most 23.
#include <cuda_fp16.h>

#include "ds4x_internal.cuh"
#include "tc_ptx.cuh"

namespace ds4x {
namespace {

using namespace ptx;

constexpr int kTileRows = 128;
constexpr int kTileBytes = kTileRows * DS4X_IDX_ROW_BYTES;  // 8704
constexpr int kStages = 10;
constexpr int kWG = 4;                    // converter/epilogue warpgroups
constexpr int kWGThreads = 128 * kWG;     // 512
constexpr int kProducerWarp = kWGThreads / 32;
constexpr int kMmaWarp = kProducerWarp + 1;
constexpr int kThreads = kWGThreads + 64;  // 576
constexpr int kChunkTiles = 64;
constexpr int kLocalK = DS4X_TOPK_MAX;   // 512
constexpr int kKeysCap = kLocalK + kChunkTiles * kTileRows;  // 8704
constexpr int kSelPerThread = 18;         // kSelPerThread * 512 >= kKeysCap and >= 256 * 16 + 512
constexpr int kTopM = 16;
constexpr int kHistBuckets = 4096;
constexpr int kMaxCtas = 256;
constexpr int kTmemCols = 512;
constexpr uint32_t kBqBytes = DS4X_IDX_HEADS * DS4X_IDX_DIM * 2;  // 16384
constexpr uint32_t kBqSbo = (DS4X_IDX_DIM / 8) * 128;           // 2048: next 8 heads
constexpr uint32_t kBqLbo = 128;                                 // next 8 K elements
constexpr uint32_t kIdesc = idesc_f16_f32(128, DS4X_IDX_HEADS);
constexpr unsigned long long kTimeoutNs = 500ull * 1000 * 1000;  // a bounded wait gives up after 0.5 s
constexpr uint32_t kBarSel = 1;           // named barrier of the 512 warpgroup threads

struct SelShared {
  unsigned long long kmin, kmax;
  int nz, bstar, above, bcnt, out_cnt, list_cnt;
  unsigned long long red_min[16], red_max[16];
  int red_cnt[16];
  int scan[16];
};

struct __align__(1024) Smem {
  uint8_t bq[kBqBytes];                      // query, fp16, canonical no-swizzle K-major
  uint8_t stage[kStages][kTileBytes];        // raw tile ring
  unsigned long long keys[kKeysCap];         // [0, 512): carried local top; then the chunk's keys
  unsigned long long out[kLocalK];
  unsigned long long top16[kTopM];
  uint32_t hist[kHistBuckets];
  alignas(16) float wq[DS4X_IDX_HEADS];      // w_h * 2^-(a_h + 1)
  unsigned long long full[kStages], empty[kStages], afull[kWG], accfull[kWG];
  SelShared sel;
  uint32_t tmem_base;
  int abort_flag;
  int is_last;
};

struct FusedWs {
  WsHeader hdr;
  unsigned long long lists[kMaxCtas][kLocalK];  // per CTA: top-16 first, then the rest
  int cnt[kMaxCtas];                            // valid keys in the CTA's list
  unsigned long long th16[kMaxCtas];            // CTA's 16th largest key (0: none beyond the top 16)
};

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded mbarrier wait: on time-out the CTA is marked aborted and the
// workspace status gets DS4X_ETIMEOUT.
__device__ bool wait_bar(Smem &sm, unsigned long long *bar, uint32_t parity, WsHeader *hdr) {
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

// Bounded wait used only while shutting down after a time-out, so that no
// bulk copy or MMA is still writing into this CTA's memory when it exits.
__device__ void drain_bar(unsigned long long *bar, uint32_t parity) {
  const uint32_t b = smem_u32(bar);
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(b, parity) && globaltimer() - t0 < kTimeoutNs / 5) {
  }
}

__device__ __forceinline__ float pow2f(int e) {  // exact 2^e for e in [-126, 127]
  return __uint_as_float(uint32_t(e + 127) << 23);
}

__device__ __forceinline__ float scale_by_pow2(float s, int e) {
  if (e >= -126 && e <= 127) return s * pow2f(e);
  return ldexpf(s, e);
}

// ---------------------------------------------------------------------------
// Exact selection of the K largest nonzero keys of list[0, n) into out[]
// (unsorted), by all 512 warpgroup threads.  Keys are distinct.  The key
// range [kmin, kmax] is cut into at most 4096 power-of-two buckets; keys in
// buckets above the one holding the K-th key are taken, and the boundary
// bucket is either taken whole, sorted (<= 512 keys) or cut again.
// list[] is clobbered.  Returns the number of keys written to out.
// ---------------------------------------------------------------------------
__device__ void bitonic_desc(unsigned long long *a, int n_pow2, int tid) {
  for (int size = 2; size <= n_pow2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      named_bar_sync(kBarSel, kWGThreads);
      for (int t = tid; t < n_pow2 / 2; t += kWGThreads) {
        const int i = 2 * t - (t & (stride - 1));
        const int j = i + stride;
        const bool desc = ((i & size) == 0);
        const unsigned long long x = a[i], y = a[j];
        if ((x < y) == desc) {
          a[i] = y;
          a[j] = x;
        }
      }
    }
  }
  named_bar_sync(kBarSel, kWGThreads);
}

__device__ int select_top(unsigned long long *list, int n, int K, unsigned long long *out, uint32_t *hist,
                          SelShared &sh, int tid) {
  const int lane = tid & 31, warp = tid >> 5;
  if (tid == 0) sh.out_cnt = 0;
  named_bar_sync(kBarSel, kWGThreads);
  int need = K;
  int cur_n = n;
  while (need > 0) {
    unsigned long long v[kSelPerThread];
    unsigned long long lmin = ~0ull, lmax = 0;
    int lcnt = 0;
#pragma unroll
    for (int q = 0; q < kSelPerThread; ++q) {
      const int i = tid + q * kWGThreads;
      v[q] = i < cur_n ? list[i] : 0ull;
      if (v[q] != 0) {
        lmin = min(lmin, v[q]);
        lmax = max(lmax, v[q]);
        ++lcnt;
      }
    }
    for (int o = 16; o > 0; o >>= 1) {
      lmin = min(lmin, __shfl_xor_sync(0xffffffffu, lmin, o));
      lmax = max(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
      lcnt += __shfl_xor_sync(0xffffffffu, lcnt, o);
    }
    if (lane == 0) {
      sh.red_min[warp] = lmin;
      sh.red_max[warp] = lmax;
      sh.red_cnt[warp] = lcnt;
    }
    named_bar_sync(kBarSel, kWGThreads);
    unsigned long long kmin = ~0ull, kmax = 0;
    int nz = 0;
    for (int w = 0; w < kWGThreads / 32; ++w) {
      kmin = min(kmin, sh.red_min[w]);
      kmax = max(kmax, sh.red_max[w]);
      nz += sh.red_cnt[w];
    }
    if (nz <= need) {  // everything left is selected
#pragma unroll
      for (int q = 0; q < kSelPerThread; ++q)
        if (v[q] != 0) out[atomicAdd(&sh.out_cnt, 1)] = v[q];
      named_bar_sync(kBarSel, kWGThreads);
      break;
    }
    const unsigned long long range = kmax - kmin;
    const int shift = range < kHistBuckets ? 0 : (64 - __clzll((long long)range)) - 12;
    for (int b = tid; b < kHistBuckets; b += kWGThreads) hist[b] = 0;
    named_bar_sync(kBarSel, kWGThreads);
#pragma unroll
    for (int q = 0; q < kSelPerThread; ++q)
      if (v[q] != 0) atomicAdd(&hist[(v[q] - kmin) >> shift], 1u);
    named_bar_sync(kBarSel, kWGThreads);
    // thread t owns the 8 buckets [4095 - 8t - 7, 4095 - 8t]; t = 0 owns the top
    const int btop = kHistBuckets - 1 - 8 * tid;
    int local = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) local += int(hist[btop - q]);
    int incl = local;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) sh.scan[warp] = incl;
    named_bar_sync(kBarSel, kWGThreads);
    int above = incl - local;
    for (int w = 0; w < warp; ++w) above += sh.scan[w];
    if (above < need && above + local >= need) {
      int acc = above;
      for (int q = 0; q < 8; ++q) {
        const int c = int(hist[btop - q]);
        if (acc + c >= need) {
          sh.bstar = btop - q;
          sh.above = acc;
          sh.bcnt = c;
          break;
        }
        acc += c;
      }
    }
    if (tid == 0) sh.list_cnt = 0;
    named_bar_sync(kBarSel, kWGThreads);
    const int bstar = sh.bstar, bcnt = sh.bcnt;
    need -= sh.above;
#pragma unroll
    for (int q = 0; q < kSelPerThread; ++q) {
      if (v[q] == 0) continue;
      const int b = int((v[q] - kmin) >> shift);
      if (b > bstar) out[atomicAdd(&sh.out_cnt, 1)] = v[q];
      else if (b == bstar) list[atomicAdd(&sh.list_cnt, 1)] = v[q];
    }
    named_bar_sync(kBarSel, kWGThreads);
    cur_n = bcnt;
    if (bcnt == need) {
      for (int i = tid; i < bcnt; i += kWGThreads) out[sh.out_cnt + i] = list[i];
      named_bar_sync(kBarSel, kWGThreads);
      if (tid == 0) sh.out_cnt += bcnt;
      named_bar_sync(kBarSel, kWGThreads);
      break;
    }
    if (bcnt <= kWGThreads) {
      for (int i = bcnt + tid; i < kWGThreads; i += kWGThreads) list[i] = 0;
      bitonic_desc(list, kWGThreads, tid);
      for (int i = tid; i < need; i += kWGThreads) out[sh.out_cnt + i] = list[i];
      named_bar_sync(kBarSel, kWGThreads);
      if (tid == 0) sh.out_cnt += need;
      named_bar_sync(kBarSel, kWGThreads);
      break;
    }
    // the boundary bucket still holds more than 512 keys: cut its range again
  }
  named_bar_sync(kBarSel, kWGThreads);
  return sh.out_cnt;
}

__global__ void __launch_bounds__(kThreads, 1)
score_fused_kernel(const uint8_t *__restrict__ rows, int64_t n_rows, const uint16_t *__restrict__ q,
                   const float *__restrict__ w, int k, int32_t *__restrict__ out_idx,
                   float *__restrict__ out_score, FusedWs *__restrict__ ws) {
  extern __shared__ uint8_t smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x;
  const int64_t n_tiles_total = (n_rows + kTileRows - 1) / kTileRows;
  const int64_t tile_begin = n_tiles_total * blockIdx.x / G;
  const int64_t tile_end = n_tiles_total * (blockIdx.x + 1) / G;
  const int n_tiles = int(tile_end - tile_begin);
  WsHeader *hdr = &ws->hdr;

  // ---- set-up -------------------------------------------------------------
  if (tid == kProducerWarp * 32) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), kTileRows);
    }
    for (int g = 0; g < kWG; ++g) {
      mbar_init(smem_u32(&sm.afull[g]), kTileRows);
      mbar_init(smem_u32(&sm.accfull[g]), 1);
    }
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&sm.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (tid < kWGThreads) {
    // query -> fp16 B operand with a per-head power-of-two scale
    for (int h = warp * 4; h < warp * 4 + 4; ++h) {
      const uint2 raw = reinterpret_cast<const uint2 *>(q + h * DS4X_IDX_DIM)[lane];
      float x[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xffff0000u),
                    __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xffff0000u)};
      float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      int a = 0;
      if (amax > 0.0f) {
        int F;
        frexpf(amax, &F);  // amax in [2^(F-1), 2^F)
        a = 16 - F;        // scaled max in [2^15, 2^16)
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int kk = 4 * lane + e;
        const __half hv = __float2half_rn(ldexpf(x[e], a));
        const uint32_t off = (h >> 3) * kBqSbo + (kk >> 3) * kBqLbo + (h & 7) * 16 + (kk & 7) * 2;
        *reinterpret_cast<__half *>(sm.bq + off) = hv;
      }
      if (lane == 0) sm.wq[h] = ldexpf(w[h], -a - 1);
    }
    for (int i = tid; i < kKeysCap; i += kWGThreads) sm.keys[i] = 0ull;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sm.tmem_base;

  if (warp == kProducerWarp) {
    // ---- producer: bulk-copy tiles into the stage ring ---------------------
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < n_tiles; ++i) {
        const int s = i % kStages;
        if (i >= kStages && !wait_bar(sm, &sm.empty[s], ((i / kStages) - 1) & 1, hdr)) break;
        const int64_t tile = tile_begin + i;
        const int64_t r0 = tile * kTileRows;
        const int nr = n_rows - r0 < kTileRows ? int(n_rows - r0) : kTileRows;
        const uint32_t bytes = uint32_t(nr) * DS4X_IDX_ROW_BYTES;
        const uint32_t bulk = bytes & ~15u;
        const uint8_t *src = rows + r0 * DS4X_IDX_ROW_BYTES;
        for (uint32_t b = bulk; b < bytes; b += 4)  // ragged tail of the last tile
          *reinterpret_cast<uint32_t *>(sm.stage[s] + b) = *reinterpret_cast<const uint32_t *>(src + b);
        mbar_arrive_expect_tx(smem_u32(&sm.full[s]), bulk);
        bulk_g2s(smem_u32(sm.stage[s]), src, bulk, smem_u32(&sm.full[s]));
        issued = i + 1;
      }
      if (*reinterpret_cast<volatile int *>(&sm.abort_flag)) {
        for (int i = max(0, issued - kStages); i < issued; ++i) drain_bar(&sm.full[i % kStages], (i / kStages) & 1);
      }
    }
  } else if (warp == kMmaWarp) {
    // ---- MMA issuer ---------------------------------------------------------
    if (lane == 0) {
      const uint32_t bq = smem_u32(sm.bq);
      int issued = 0;
      for (int i = 0; i < n_tiles; ++i) {
        const int g = i % kWG;
        if (!wait_bar(sm, &sm.afull[g], (i / kWG) & 1, hdr)) break;
        tc_fence_after();
        const uint32_t d_t = tmem_base + uint32_t(g * 128);
        const uint32_t a_t = d_t + 64;
#pragma unroll
        for (int kk = 0; kk < DS4X_IDX_DIM / 16; ++kk) {
          mma_f16_ta(d_t, a_t + uint32_t(kk * 8), smem_desc_noswizzle(bq + kk * 256, kBqLbo, kBqSbo), kIdesc,
                     kk > 0);
        }
        tc_commit(smem_u32(&sm.accfull[g]));
        issued = i + 1;
      }
      if (*reinterpret_cast<volatile int *>(&sm.abort_flag)) {
        for (int i = max(0, issued - kWG); i < issued; ++i) drain_bar(&sm.accfull[i % kWG], (i / kWG) & 1);
      }
    }
  } else {
    // ---- warpgroups: dequantise -> TMEM, then the ReLU-weighted epilogue -----
    const int g = warp / 4;
    const int r = tid & 127;                             // row within the tile == TMEM lane
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    const uint32_t d_t = tmem_base + lane_base + uint32_t(g * 128);
    const uint32_t a_t = d_t + 64;
    int m = 0;  // keys in the carried local top list
    for (int c0 = 0; c0 < n_tiles; c0 += kChunkTiles) {
      const int c1 = min(n_tiles, c0 + kChunkTiles);
      for (int i = c0 + ((g - c0 % kWG) + kWG) % kWG; i < c1; i += kWG) {
        const int s = i % kStages;
        bool ok = wait_bar(sm, &sm.full[s], (i / kStages) & 1, hdr);
        uint32_t wd[17];
        const uint32_t *rp = reinterpret_cast<const uint32_t *>(sm.stage[s] + r * DS4X_IDX_ROW_BYTES);
#pragma unroll
        for (int t = 0; t < 17; ++t) wd[t] = rp[t];
        mbar_arrive(smem_u32(&sm.empty[s]));
        // block scales relative to the row's largest block exponent
        int eb[4], eref = -1000;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          eb[b] = int((wd[16] >> (8 * b)) & 0xffu) - 127;
          eref = max(eref, eb[b]);
        }
        uint32_t f2[4];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int d = max(eb[b] - eref, -24);
          const uint32_t h = d >= -14 ? uint32_t(15 + d) << 10 : (1u << (d + 24));  // fp16 2^d
          f2[b] = h | (h << 16);
        }
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t a[32];
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const uint32_t word = wd[half * 8 + t];
            const uint32_t f = f2[(half * 8 + t) >> 2];
            a[4 * t + 0] = hmul2(e2m1x2_to_f16x2(word), f);
            a[4 * t + 1] = hmul2(e2m1x2_to_f16x2(word >> 8), f);
            a[4 * t + 2] = hmul2(e2m1x2_to_f16x2(word >> 16), f);
            a[4 * t + 3] = hmul2(e2m1x2_to_f16x2(word >> 24), f);
          }
          tc_st_x32(a_t + uint32_t(half * 32), a);
        }
        tc_wait_st();
        tc_fence_before();
        mbar_arrive(smem_u32(&sm.afull[g]));
        ok = wait_bar(sm, &sm.accfull[g], (i / kWG) & 1, hdr) && ok;
        tc_fence_after();
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        {
          uint32_t d0[32], d1[32];
          tc_ld_x32(d_t, d0);
          tc_ld_x32(d_t + 32u, d1);
          tc_wait_ld();
          const float4 *wq4 = reinterpret_cast<const float4 *>(sm.wq);
#pragma unroll
          for (int h4 = 0; h4 < 16; ++h4) {
            const float4 wv = wq4[h4];
            const uint32_t *src = h4 < 8 ? d0 + 4 * h4 : d1 + 4 * (h4 - 8);
            const float x0 = __uint_as_float(src[0]), x1 = __uint_as_float(src[1]);
            const float x2 = __uint_as_float(src[2]), x3 = __uint_as_float(src[3]);
            acc[0] = fmaf(wv.x, x0 + fabsf(x0), acc[0]);
            acc[1] = fmaf(wv.y, x1 + fabsf(x1), acc[1]);
            acc[2] = fmaf(wv.z, x2 + fabsf(x2), acc[2]);
            acc[3] = fmaf(wv.w, x3 + fabsf(x3), acc[3]);
          }
        }
        const float s_row = scale_by_pow2((acc[0] + acc[1]) + (acc[2] + acc[3]), eref);
        const int64_t row = (tile_begin + i) * kTileRows + r;
        sm.keys[kLocalK + (i - c0) * kTileRows + r] =
            (ok && row < n_rows) ? make_key(s_row, uint32_t(row)) : 0ull;
      }
      tc_fence_before();
      named_bar_sync(kBarSel, kWGThreads);
      // exact local top-512 of the carried keys and this chunk's keys
      const int n_in = kLocalK + (c1 - c0) * kTileRows;
      m = select_top(sm.keys, n_in, kLocalK, sm.out, sm.hist, sm.sel, tid);
      for (int i = tid; i < kKeysCap; i += kWGThreads) sm.keys[i] = i < m ? sm.out[i] : 0ull;
      named_bar_sync(kBarSel, kWGThreads);
    }

    // ---- publish this CTA's list: top-16 first, then the rest ---------------
    for (int i = tid; i < kLocalK; i += kWGThreads) sm.keys[kLocalK + i] = sm.keys[i];
    named_bar_sync(kBarSel, kWGThreads);
    const int m16 = select_top(sm.keys + kLocalK, m, kTopM, sm.top16, sm.hist, sm.sel, tid);
    unsigned long long th = 0ull;
    if (m > kTopM) {
      th = ~0ull;
      for (int i = 0; i < m16; ++i) th = min(th, sm.top16[i]);
    }
    const int c = blockIdx.x;
    for (int i = tid; i < kTopM; i += kWGThreads) ws->lists[c][i] = i < m16 ? sm.top16[i] : 0ull;
    if (tid == 0) sm.sel.list_cnt = 0;
    named_bar_sync(kBarSel, kWGThreads);
    for (int i = tid; i < m; i += kWGThreads) {
      const unsigned long long key = sm.keys[i];
      if (key < th) ws->lists[c][kTopM + atomicAdd(&sm.sel.list_cnt, 1)] = key;
    }
    if (tid == 0) {
      ws->cnt[c] = m;
      ws->th16[c] = th;
    }
    __threadfence();
    named_bar_sync(kBarSel, kWGThreads);
    if (tid == 0) {
      const unsigned int ticket = atomicAdd(&hdr->ticket, 1u);
      sm.is_last = (ticket == unsigned(G - 1));
    }
    named_bar_sync(kBarSel, kWGThreads);

    if (sm.is_last) {
      // ---- global merge (last CTA to finish) ----------------------------------
      __threadfence();
      const int kk = k;
      for (int i = tid; i < G * kTopM; i += kWGThreads) {
        sm.keys[i] = reinterpret_cast<volatile unsigned long long *>(ws->lists[i / kTopM])[i % kTopM];
      }
      named_bar_sync(kBarSel, kWGThreads);
      int sel_n = select_top(sm.keys, G * kTopM, kk, sm.out, sm.hist, sm.sel, tid);
      unsigned long long cut = 0ull;
      if (sel_n == kk) {
        cut = ~0ull;
        for (int i = 0; i < sel_n; ++i) cut = min(cut, sm.out[i]);
      }
      // CTAs whose 16th key beats the cut may hold more winners: fetch them
      bool fell_back = false;
      int fill = 0;
      for (int cc = 0; cc < G; ++cc) {
        const int cnt = reinterpret_cast<volatile int *>(ws->cnt)[cc];
        const unsigned long long t16 = reinterpret_cast<volatile unsigned long long *>(ws->th16)[cc];
        if (cnt <= kTopM || t16 <= cut) continue;
        if (!fell_back) {
          for (int i = tid; i < sel_n; i += kWGThreads) sm.keys[i] = sm.out[i];
          fill = sel_n;
          fell_back = true;
          named_bar_sync(kBarSel, kWGThreads);
        }
        const int extra = cnt - kTopM;
        if (fill + extra > kKeysCap) {
          sel_n = select_top(sm.keys, fill, kk, sm.out, sm.hist, sm.sel, tid);
          for (int i = tid; i < sel_n; i += kWGThreads) sm.keys[i] = sm.out[i];
          fill = sel_n;
          named_bar_sync(kBarSel, kWGThreads);
        }
        for (int i = tid; i < extra; i += kWGThreads)
          sm.keys[fill + i] = reinterpret_cast<volatile unsigned long long *>(ws->lists[cc])[kTopM + i];
        fill += extra;
        named_bar_sync(kBarSel, kWGThreads);
      }
      if (fell_back) {
        sel_n = select_top(sm.keys, fill, kk, sm.out, sm.hist, sm.sel, tid);
        if (tid == 0) atomicAdd(&hdr->fallback, 1u);
      }
      for (int i = tid; i < kLocalK; i += kWGThreads) sm.keys[i] = i < sel_n ? sm.out[i] : 0ull;
      bitonic_desc(sm.keys, kLocalK, tid);
      for (int i = tid; i < kk; i += kWGThreads) {
        if (i < sel_n) {
          out_idx[i] = key_index(sm.keys[i]);
          if (out_score) out_score[i] = key_score(sm.keys[i]);
        } else {
          out_idx[i] = -1;
          if (out_score) out_score[i] = __uint_as_float(0x7fc00000u);
        }
      }
      if (tid == 0) hdr->ticket = 0u;  // ready for the next call on this workspace
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace

size_t score_fused_ws_bytes() { return sizeof(FusedWs); }

int score_fused_max_ctas() { return kMaxCtas; }

cudaError_t launch_score_fused(const uint8_t *idx_rows, int64_t n_rows, const uint16_t *q, const float *w,
                               int32_t k, int32_t *out_idx, float *out_score, void *ws, cudaStream_t stream) {
  static std::atomic<uint64_t> smem_set{0};
  const int smem_bytes = int(sizeof(Smem)) + 1024;
  cudaError_t e = set_max_smem_once(score_fused_kernel, smem_bytes, smem_set);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int64_t tiles = (n_rows + kTileRows - 1) / kTileRows;
  const int cap = sms < kMaxCtas ? sms : kMaxCtas;
  const int grid = tiles < cap ? int(tiles) : cap;
  score_fused_kernel<<<grid, kThreads, smem_bytes, stream>>>(idx_rows, n_rows, q, w, k, out_idx, out_score,
                                                             static_cast<FusedWs *>(ws));
  return cudaGetLastError();
}

}  // namespace ds4x
