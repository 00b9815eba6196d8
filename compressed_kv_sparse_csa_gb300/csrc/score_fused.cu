// Fused CSA indexer score + exact top-k on the fifth-generation tensor cores.
//
// DS4X README, "Optimization details" / "CSA score/top-512 fusion": the
// scorer reads the packed 68-byte MXFP4 rows directly, every scorer CTA keeps
// an exact local top-512 of sortable (score, index) keys, and the local lists
// are merged into the exact top-512 without materialising the score array.
// This is a GB300 design of that method.  One persistent CTA per SM:
//
//  * warp 16 streams the CTA's contiguous range of 128-row tiles (8,704 bytes
//    each) from HBM with 1-D bulk copies into a ring of shared-memory stages;
//  * converter warpgroups 0-1 (thread = row) dequantise a tile: each byte of
//    two E2M1 codes goes through the hardware e2m1x2 -> f16x2 converter, then
//    one f16x2 multiply applies the block's scale relative to the row's
//    largest block scale 2^e_ref; the 64 words go straight into a tensor-
//    memory A slot (four-slot ring), never through shared memory;
//  * warp 17 issues the tile's eight tcgen05.mma kind::f16 (M = 128 rows,
//    N = 64 heads, K = 16) against the fp16 query (B, shared memory) into a
//    tensor-memory accumulator slot (four-slot ring) and commits the tile's
//    completion to both rings.  The issuing warp competes for issue slots
//    with the converter and epilogue warps, so those keep their FP32-pipe
//    work small (the epilogue's ReLU runs on the integer pipe);
//  * epilogue warpgroups 2-3 read a row's 64 accumulators back and form
//    s = 2^e_ref * sum_h (w_h / 2^a_h) * ReLU(acc_h) with the ReLU as a
//    signed-integer max on the float bits and packed f32x2 FMAs, which is
//    sum_h w_h * ReLU(q_h . k) up to fp32 rounding; each key goes into shared
//    memory and into a fixed 8,192-bucket histogram of its score bits;
//  * after the stream one scan of the histogram locates the CTA's 512th and
//    16th keys; one pass keeps the keys at or above the 512th key's bucket
//    (a superset of the local top-512) and resolves the exact top-16; the
//    CTA publishes both; the last CTA to finish sorts the CTAs' top-16
//    sets together (a register-blocked bitonic merge of the sorted lists),
//    fetches the supersets of any CTA whose 16th key beats the k-th key (so
//    the result is exact for every input) and writes the outputs.
//
// The query is held in fp16 with a per-head power-of-two scale 2^a_h that
// puts the head's largest |q| in [2^15, 2^16): every bf16 element within
// 2^-32 of its head's maximum converts exactly.  Keys are exact in fp16
// whenever a row's block exponents differ by at most 23.
#include <cuda_fp16.h>

#include "ds4x_internal.cuh"
#include "tc_ptx.cuh"

namespace ds4x {
namespace {

using namespace ptx;

constexpr int kTileRows = 128;
constexpr int kTileBytes = kTileRows * DS4X_IDX_ROW_BYTES;  // 8704
constexpr int kStages = 8;
constexpr int kConvWG = 2;                 // converter warpgroups: warps 0-7
constexpr int kEpiWG = 2;                  // epilogue warpgroups: warps 8-15
constexpr int kWGThreads = 128 * (kConvWG + kEpiWG);  // 512
constexpr int kProducerWarp = kWGThreads / 32;        // 16
constexpr int kMmaWarp = kProducerWarp + 1;           // 17: allocates tensor memory, issues MMAs
constexpr int kThreads = kWGThreads + 64;             // 576
constexpr int kSlots = 4;                  // TMEM A ring and D ring depth
constexpr int kErefRing = 8;
constexpr int kChunkTiles = 64;
constexpr int kLocalK = DS4X_TOPK_MAX;     // 512
constexpr int kKeysCap = kLocalK + kChunkTiles * kTileRows;  // 8704
constexpr int kSelPerThread = 18;          // 18 * 512 >= kKeysCap and >= 256 * 16 + 512
constexpr int kTopM = 16;
constexpr int kPubCap = 1024;              // keys a CTA may publish (its top-16, then a superset of the rest)
constexpr int kBuckets = 8192;             // fixed score-bit histogram (16-bit counters, 2 per word)
constexpr int kHistWords = 4096;
constexpr int kMaxCtas = 256;
constexpr int kTmemCols = 512;
constexpr uint32_t kDCol0 = 0;             // D slot j: columns [64j, 64j + 64)
constexpr uint32_t kACol0 = 256;           // A slot j: columns [256 + 64j, 256 + 64j + 64)
constexpr uint32_t kBqBytes = DS4X_IDX_HEADS * DS4X_IDX_DIM * 2;  // 16384
constexpr uint32_t kBqSbo = (DS4X_IDX_DIM / 8) * 128;           // 2048: next 8 heads
constexpr uint32_t kBqLbo = 128;                                 // next 8 K elements
constexpr uint32_t kIdesc = idesc_f16_f32(128, DS4X_IDX_HEADS);
constexpr unsigned long long kTimeoutNs = 500ull * 1000 * 1000;  // a bounded wait gives up after 0.5 s
constexpr uint32_t kBarSel = 1;            // named barrier of the 512 warpgroup threads

struct SelShared {
  unsigned long long red_min[16], red_max[16];
  int red_cnt[16];
  int scan[16];
  int bstar, above, bcnt, out_cnt, list_cnt, n16, nb16;
  int c512_b, c512_above, c16_b, c16_above, c16_cnt, total;
};

struct __align__(1024) Smem {
  uint8_t bq[kBqBytes];                       // query, fp16, canonical no-swizzle K-major
  uint8_t stage[kStages][kTileBytes];         // raw tile ring
  unsigned long long keys[kKeysCap];          // [0, 512): carried keys; then the chunk's keys
  unsigned long long out[kLocalK];
  unsigned long long sortbuf[2 * kLocalK];
  unsigned long long top16[32];
  unsigned long long b16[32];
  uint32_t hist[kHistWords];                  // fixed histogram, or the adaptive one inside select_top
  alignas(16) float wq[DS4X_IDX_HEADS];       // w_h * 2^-a_h
  int eref[kErefRing][kTileRows];
  unsigned long long full[kStages], empty[kStages];
  unsigned long long afull[kSlots], aempty[kSlots], dfull[kSlots], dempty[kSlots];
  unsigned long long ereff[kErefRing];
  SelShared sel;
  int fetch[kMaxCtas];
  uint32_t tmem_base;
  int abort_flag;
  int is_last;
};

struct FusedWs {
  WsHeader hdr;
  unsigned long long lists[kMaxCtas][kPubCap];  // per CTA: its top-16 (descending), then the rest
  int cnt[kMaxCtas];                            // entries in the CTA's list
  unsigned long long th16[kMaxCtas];            // CTA's 16th largest key (0: the list is all it has)
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

__device__ __forceinline__ float scale_by_pow2(float s, int e) {
  if (e >= -126 && e <= 127) return s * __uint_as_float(uint32_t(e + 127) << 23);
  return ldexpf(s, e);
}

// Fixed histogram bucket of a key: the top 14 bits of its ordered score bits
// (sign, exponent, 4 mantissa bits), non-positive scores in bucket 0.
// Non-decreasing in the key.
__device__ __forceinline__ int fixed_bucket(unsigned long long key) {
  const int b = int(uint32_t(key >> 32) >> 18) - kBuckets;
  return b < 0 ? 0 : b;
}

__device__ __forceinline__ void hist_add(uint32_t *hist, int b) {
  atomicAdd(&hist[b >> 1], 1u << ((b & 1) * 16));
}

__device__ __forceinline__ void bar512() { named_bar_sync(kBarSel, kWGThreads); }

// Warp-aggregated append: every lane of the warp calls it; lanes with pred
// get consecutive slots from *counter (one shared atomic per warp instead of
// one per lane, which would serialise on the single address).
__device__ __forceinline__ int warp_append(int *counter, bool pred) {
  const unsigned mask = __ballot_sync(0xffffffffu, pred);
  const int lane = threadIdx.x & 31;
  int base = 0;
  if (mask != 0u) {
    const int leader = __ffs(mask) - 1;
    if (lane == leader) base = atomicAdd(counter, __popc(mask));
    base = __shfl_sync(0xffffffffu, base, leader);
  }
  return base + __popc(mask & ((1u << lane) - 1u));
}

__device__ __forceinline__ unsigned long long ld_cg(const unsigned long long *p) { return __ldcg(p); }

// ---------------------------------------------------------------------------
// Sorting helpers (descending).  Zero keys are padding and sort last.
// ---------------------------------------------------------------------------

// One warp: lane i returns the i-th largest of the 32 values.
__device__ unsigned long long warp_sort32_desc(unsigned long long v, int lane) {
  for (int size = 2; size <= 32; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, stride);
      const bool keep_max = ((lane & size) == 0) == ((lane & stride) == 0);
      v = keep_max ? max(v, o) : min(v, o);
    }
  }
  return v;
}

// All 512 warpgroup threads: thread t returns the t-th largest of the 512
// values (bitonic network; strides below 32 by shuffles, the rest through a
// double-buffered shared array, one barrier per such stage).
__device__ unsigned long long block_sort512_desc(unsigned long long v, unsigned long long *buf, int tid) {
  int pb = 0;
  for (int size = 2; size <= kWGThreads; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      unsigned long long o;
      if (stride >= 32) {
        buf[pb * kWGThreads + tid] = v;
        bar512();
        o = buf[pb * kWGThreads + (tid ^ stride)];
        pb ^= 1;
      } else {
        o = __shfl_xor_sync(0xffffffffu, v, stride);
      }
      const bool keep_max = ((tid & size) == 0) == ((tid & stride) == 0);
      v = keep_max ? max(v, o) : min(v, o);
    }
  }
  return v;
}

// ---------------------------------------------------------------------------
// Exact selection of the K largest nonzero keys of list[0, n) into out[]
// (unsorted), by all 512 warpgroup threads.  Keys are distinct.  The key
// range [kmin, kmax] is cut into at most 4096 power-of-two buckets; keys in
// buckets above the one holding the K-th key are taken, and the boundary
// bucket is taken whole, sorted (<= 512 keys) or cut again.  list[] and
// hist[] are clobbered; sortbuf holds 1024 keys.  Returns the number of
// keys written to out.
// ---------------------------------------------------------------------------
__device__ int select_top(unsigned long long *list, int n, int K, unsigned long long *out, uint32_t *hist,
                          unsigned long long *sortbuf, SelShared &sh, int tid) {
  constexpr int kAdaptBuckets = 4096;
  const int lane = tid & 31, warp = tid >> 5;
  if (tid == 0) sh.out_cnt = 0;
  bar512();
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
    for (int b = tid; b < kAdaptBuckets; b += kWGThreads) hist[b] = 0;
    bar512();
    unsigned long long kmin = ~0ull, kmax = 0;
    int nz = 0;
    for (int w = 0; w < kWGThreads / 32; ++w) {
      kmin = min(kmin, sh.red_min[w]);
      kmax = max(kmax, sh.red_max[w]);
      nz += sh.red_cnt[w];
    }
    if (nz <= need) {  // everything left is selected
#pragma unroll
      for (int q = 0; q < kSelPerThread; ++q) {
        const int pos = warp_append(&sh.out_cnt, v[q] != 0);
        if (v[q] != 0) out[pos] = v[q];
      }
      bar512();
      break;
    }
    const unsigned long long range = kmax - kmin;
    const int shift = range < kAdaptBuckets ? 0 : (64 - __clzll((long long)range)) - 12;
#pragma unroll
    for (int q = 0; q < kSelPerThread; ++q)
      if (v[q] != 0) atomicAdd(&hist[(v[q] - kmin) >> shift], 1u);
    bar512();
    // thread t owns the 8 buckets [4095 - 8t - 7, 4095 - 8t]; t = 0 owns the top
    const int btop = kAdaptBuckets - 1 - 8 * tid;
    int local = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) local += int(hist[btop - q]);
    int incl = local;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) sh.scan[warp] = incl;
    bar512();
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
    bar512();
    const int bstar = sh.bstar, bcnt = sh.bcnt;
    need -= sh.above;
#pragma unroll
    for (int q = 0; q < kSelPerThread; ++q) {
      const int b = v[q] != 0 ? int((v[q] - kmin) >> shift) : -1;
      const int po = warp_append(&sh.out_cnt, b > bstar);
      const int pl = warp_append(&sh.list_cnt, b == bstar);
      if (b > bstar) out[po] = v[q];
      else if (b == bstar) list[pl] = v[q];
    }
    bar512();
    cur_n = bcnt;
    const int base = sh.out_cnt;
    if (bcnt == need) {
      for (int i = tid; i < bcnt; i += kWGThreads) out[base + i] = list[i];
      bar512();
      if (tid == 0) sh.out_cnt += bcnt;
      bar512();
      break;
    }
    if (bcnt <= 32) {
      if (warp == 0) {
        const unsigned long long s = warp_sort32_desc(lane < bcnt ? list[lane] : 0ull, lane);
        if (lane < need) out[base + lane] = s;
      }
      bar512();
      if (tid == 0) sh.out_cnt += need;
      bar512();
      break;
    }
    if (bcnt <= kWGThreads) {
      const unsigned long long s = block_sort512_desc(tid < bcnt ? list[tid] : 0ull, sortbuf, tid);
      if (tid < need) out[base + tid] = s;
      bar512();
      if (tid == 0) sh.out_cnt += need;
      bar512();
      break;
    }
    // the boundary bucket still holds more than 512 keys: cut its range again
  }
  bar512();
  return sh.out_cnt;
}

// The K largest nonzero keys of keys[0, n) (n <= 4096, distinct, zeros are
// padding), written to out[0, K') sorted descending, K' = min(K, nonzero
// count); returns K', or -1 when a bucket is too crowded for this method
// (the caller then falls back to select_top).  A counting sort: the key range
// is cut into 4096 power-of-two buckets, a prefix scan over the buckets from
// the top gives every bucket its first output slot, each key is scattered to
// that slot plus its arrival order, and keys sharing a bucket re-rank among
// their bucket-mates.  keys[], hist[] and fill[] (4096 words) are clobbered.
__device__ int merge_topk_sorted(unsigned long long *keys, int n, int K, unsigned long long *out, uint32_t *hist,
                                 uint32_t *fill, SelShared &sh, int tid) {
  constexpr int kB = 4096, kPer = 8, kCrowd = 64;
  const int lane = tid & 31, warp = tid >> 5;
  unsigned long long v[kPer];
  unsigned long long lmin = ~0ull, lmax = 0;
  int lcnt = 0;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int i = tid + q * kWGThreads;
    v[q] = i < n ? keys[i] : 0ull;
    if (v[q] != 0ull) {
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
  for (int b = tid; b < kB; b += kWGThreads) {
    hist[b] = 0u;
    fill[b] = 0u;
  }
  bar512();
  unsigned long long kmin = ~0ull, kmax = 0;
  int nz = 0;
  for (int w = 0; w < kWGThreads / 32; ++w) {
    kmin = min(kmin, sh.red_min[w]);
    kmax = max(kmax, sh.red_max[w]);
    nz += sh.red_cnt[w];
  }
  const int kout = nz < K ? nz : K;
  if (kout == 0) return 0;
  const unsigned long long range = kmax - kmin;
  const int shift = range < kB ? 0 : (64 - __clzll((long long)range)) - 12;
  int bk[kPer];
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    bk[q] = v[q] != 0ull ? kB - 1 - int((v[q] - kmin) >> shift) : -1;  // bucket 0 holds the highest keys
    if (bk[q] >= 0) atomicAdd(&hist[bk[q]], 1u);
  }
  bar512();
  // exclusive prefix over the buckets in order 0 (top) .. 4095; thread t owns [8t, 8t + 8)
  uint32_t c8[8];
  int local = 0;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    c8[q] = hist[8 * tid + q];
    local += int(c8[q]);
  }
  int incl = local;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sh.scan[warp] = incl;
  bar512();
  int first = incl - local, crowd = 0;
  for (int w = 0; w < warp; ++w) first += sh.scan[w];
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    if (first < kout && int(c8[q]) > kCrowd) crowd = 1;
    hist[8 * tid + q] = uint32_t(first) | (c8[q] << 16);  // first slot | count
    first += int(c8[q]);
  }
  const int wcrowd = __any_sync(0xffffffffu, crowd);
  if (lane == 0) sh.red_cnt[warp] = wcrowd;
  bar512();
  int crowded = 0;
  for (int w = 0; w < kWGThreads / 32; ++w) crowded |= sh.red_cnt[w];
  if (crowded) {
    bar512();
    for (int q = 0; q < kPer; ++q) {  // hand the keys back to the caller
      const int i = tid + q * kWGThreads;
      if (i < n) keys[i] = v[q];
    }
    bar512();
    return -1;
  }
  // scatter every key of a bucket that starts before kout (keys[] is free now)
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    if (bk[q] < 0) continue;
    const uint32_t w = hist[bk[q]];
    const int f = int(w & 0xffffu);
    if (f < kout) keys[f + int(atomicAdd(&fill[bk[q]], 1u))] = v[q];
  }
  bar512();
  // final slots: keys alone in their bucket keep the bucket's slot; others
  // count the bucket-mates above them
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    if (bk[q] < 0) continue;
    const uint32_t w = hist[bk[q]];
    const int f = int(w & 0xffffu), c = int(w >> 16);
    if (f >= kout) continue;
    int rank = 0;
    for (int u = 0; u < c && c > 1; ++u) rank += keys[f + u] > v[q];
    if (f + rank < kout) out[f + rank] = v[q];
  }
  bar512();
  return kout;
}

// Cuts of the fixed histogram at the 512 and 16 largest keys: the bucket
// holding the K-th key, the number of keys in higher buckets and (for K = 16)
// in that bucket.  b = -1 when there are at most K keys.
__device__ void hist_cuts(const uint32_t *hist, SelShared &sh, int tid) {
  const int lane = tid & 31, warp = tid >> 5;
  // thread t owns words [4095 - 8t - 7, 4095 - 8t] = buckets [8191 - 16t - 15, 8191 - 16t]
  uint32_t c[16];
  int local = 0;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const uint32_t wv = hist[kHistWords - 1 - 8 * tid - q];
    c[2 * q] = wv >> 16;  // the odd (higher) bucket of the word first
    c[2 * q + 1] = wv & 0xffffu;
    local += int(c[2 * q] + c[2 * q + 1]);
  }
  int incl = local;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sh.scan[warp] = incl;
  if (tid == 0) {
    sh.c512_b = -1;
    sh.c16_b = -1;
    sh.c16_cnt = 0;
  }
  bar512();
  int above = incl - local, total = 0;
  for (int w = 0; w < kWGThreads / 32; ++w) {
    if (w < warp) above += sh.scan[w];
    total += sh.scan[w];
  }
  const int bhigh = kBuckets - 1 - 16 * tid;
  if (above < kLocalK && above + local >= kLocalK) {
    int acc = above;
    for (int q = 0; q < 16; ++q) {
      if (acc + int(c[q]) >= kLocalK) {
        sh.c512_b = bhigh - q;
        sh.c512_above = acc;
        break;
      }
      acc += int(c[q]);
    }
  }
  if (above < kTopM && above + local >= kTopM) {
    int acc = above;
    for (int q = 0; q < 16; ++q) {
      if (acc + int(c[q]) >= kTopM) {
        sh.c16_b = bhigh - q;
        sh.c16_above = acc;
        sh.c16_cnt = int(c[q]);
        break;
      }
      acc += int(c[q]);
    }
  }
  if (tid == 0) sh.total = total;
  bar512();
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
    for (int j = 0; j < kSlots; ++j) {
      mbar_init(smem_u32(&sm.afull[j]), kTileRows);
      mbar_init(smem_u32(&sm.aempty[j]), 1);
      mbar_init(smem_u32(&sm.dfull[j]), 1);
      mbar_init(smem_u32(&sm.dempty[j]), kTileRows);
    }
    for (int j = 0; j < kErefRing; ++j) mbar_init(smem_u32(&sm.ereff[j]), kTileRows);
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
      if (lane == 0) sm.wq[h] = ldexpf(w[h], -a);
    }
    for (int i = tid; i < kKeysCap; i += kWGThreads) sm.keys[i] = 0ull;
    for (int i = tid; i < kHistWords; i += kWGThreads) sm.hist[i] = 0u;
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
        const int64_t r0 = (tile_begin + i) * kTileRows;
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
      const uint64_t bdesc = smem_desc_noswizzle(smem_u32(sm.bq), kBqLbo, kBqSbo);
      int issued = 0;
      for (int i = 0; i < n_tiles; ++i) {
        const int j = i % kSlots;
        if (!wait_bar(sm, &sm.afull[j], (i / kSlots) & 1, hdr)) break;
        if (i >= kSlots && !wait_bar(sm, &sm.dempty[j], ((i / kSlots) - 1) & 1, hdr)) break;
        tc_fence_after();
        mma_f16_ta_k128(tmem_base + kDCol0 + uint32_t(64 * j), tmem_base + kACol0 + uint32_t(64 * j), bdesc,
                        kIdesc);
        tc_commit(smem_u32(&sm.aempty[j]));
        tc_commit(smem_u32(&sm.dfull[j]));
        issued = i + 1;
      }
      if (*reinterpret_cast<volatile int *>(&sm.abort_flag)) {
        for (int i = max(0, issued - kSlots); i < issued; ++i) drain_bar(&sm.dfull[i % kSlots], (i / kSlots) & 1);
      }
    }
  } else if (warp < kProducerWarp) {
    const int r = tid & 127;  // row within the tile == TMEM lane
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    const bool is_conv = warp < 4 * kConvWG;
    const int role_wg = is_conv ? warp / 4 : (warp - 4 * kConvWG) / 4;
    const int n_role_wg = is_conv ? kConvWG : kEpiWG;
    int carried = 0;  // keys carried from earlier chunks, in keys[0, carried)
    for (int c0 = 0; c0 < n_tiles; c0 += kChunkTiles) {
      const int c1 = min(n_tiles, c0 + kChunkTiles);
      for (int i = c0 + role_wg; i < c1; i += n_role_wg) {
        const int j = i % kSlots;
        const int er = i % kErefRing;
        if (is_conv) {
          // ---- convert: raw row -> fp16 A slot ------------------------------
          const int s = i % kStages;
          wait_bar(sm, &sm.full[s], (i / kStages) & 1, hdr);
          uint32_t wd[17];
          const uint32_t *rp = reinterpret_cast<const uint32_t *>(sm.stage[s] + r * DS4X_IDX_ROW_BYTES);
#pragma unroll
          for (int t = 0; t < 17; ++t) wd[t] = rp[t];
          mbar_arrive(smem_u32(&sm.empty[s]));
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
          if (i >= kSlots) wait_bar(sm, &sm.aempty[j], ((i / kSlots) - 1) & 1, hdr);
          sm.eref[er][r] = eref;
          mbar_arrive(smem_u32(&sm.ereff[er]));
          const uint32_t a_t = tmem_base + lane_base + kACol0 + uint32_t(64 * j);
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
          mbar_arrive(smem_u32(&sm.afull[j]));
        } else {
          // ---- epilogue: accumulators -> score -> key --------------------------
          bool ok = wait_bar(sm, &sm.dfull[j], (i / kSlots) & 1, hdr);
          ok = wait_bar(sm, &sm.ereff[er], (i / kErefRing) & 1, hdr) && ok;
          const int eref = sm.eref[er][r];
          tc_fence_after();
          const uint32_t d_t = tmem_base + lane_base + kDCol0 + uint32_t(64 * j);
          uint32_t d0[32], d1[32];
          tc_ld_x32(d_t, d0);
          tc_ld_x32(d_t + 32u, d1);
          tc_wait_ld();
          tc_fence_before();
          mbar_arrive(smem_u32(&sm.dempty[j]));
          // ReLU(x) as max(int bits, 0): a negative float (or -0) has negative
          // int bits, a positive one keeps its bits
          unsigned long long acc2[4] = {0ull, 0ull, 0ull, 0ull};
          const ulonglong2 *wq2 = reinterpret_cast<const ulonglong2 *>(sm.wq);
#pragma unroll
          for (int h4 = 0; h4 < 16; ++h4) {
            const ulonglong2 wv = wq2[h4];
            const uint32_t *src = h4 < 8 ? d0 + 4 * h4 : d1 + 4 * (h4 - 8);
            const unsigned long long r01 = uint64_t(uint32_t(max(int(src[0]), 0))) |
                                           (uint64_t(uint32_t(max(int(src[1]), 0))) << 32);
            const unsigned long long r23 = uint64_t(uint32_t(max(int(src[2]), 0))) |
                                           (uint64_t(uint32_t(max(int(src[3]), 0))) << 32);
            acc2[(2 * h4) & 3] = ffma2(wv.x, r01, acc2[(2 * h4) & 3]);
            acc2[(2 * h4 + 1) & 3] = ffma2(wv.y, r23, acc2[(2 * h4 + 1) & 3]);
          }
          float part[8];
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            part[2 * p] = __uint_as_float(uint32_t(acc2[p]));
            part[2 * p + 1] = __uint_as_float(uint32_t(acc2[p] >> 32));
          }
          const float sum = ((part[0] + part[1]) + (part[2] + part[3])) + ((part[4] + part[5]) + (part[6] + part[7]));
          const float s_row = scale_by_pow2(sum, eref);
          const int64_t row = (tile_begin + i) * kTileRows + r;
          unsigned long long key = 0ull;
          if (ok && row < n_rows) {
            key = make_key(s_row, uint32_t(row));
            hist_add(sm.hist, fixed_bucket(key));
          }
          sm.keys[kLocalK + (i - c0) * kTileRows + r] = key;
        }
      }
      bar512();

      // ---- end of chunk: keep a superset of the local top-512 ---------------
      hist_cuts(sm.hist, sm.sel, tid);
      const int n_in = kLocalK + (c1 - c0) * kTileRows;
      const int b512 = sm.sel.c512_b;  // -1: at most 512 keys, keep all
      const int b16 = sm.sel.c16_b;    // -1: at most 16 keys
      const bool last_chunk = c1 == n_tiles;
      const bool b16_small = b16 < 0 || sm.sel.c16_cnt <= 32;
      unsigned long long v[kSelPerThread];
#pragma unroll
      for (int qq = 0; qq < kSelPerThread; ++qq) {
        const int i = tid + qq * kWGThreads;
        v[qq] = i < n_in ? sm.keys[i] : 0ull;
      }
      if (tid == 0) {
        sm.sel.list_cnt = 0;
        sm.sel.n16 = 0;
        sm.sel.nb16 = 0;
      }
      bar512();
      {
        // one shared atomic per warp for the whole pass
        unsigned masks[kSelPerThread];
        int total = 0;
#pragma unroll
        for (int qq = 0; qq < kSelPerThread; ++qq) {
          const int b = v[qq] != 0ull ? fixed_bucket(v[qq]) : -2;
          masks[qq] = __ballot_sync(0xffffffffu, b >= b512 && b >= 0);
          total += __popc(masks[qq]);
        }
        int base = 0;
        if (lane == 0 && total > 0) base = atomicAdd(&sm.sel.list_cnt, total);
        base = __shfl_sync(0xffffffffu, base, 0);
        const unsigned lt = (1u << lane) - 1u;
#pragma unroll
        for (int qq = 0; qq < kSelPerThread; ++qq) {
          if (masks[qq] & (1u << lane)) sm.keys[base + __popc(masks[qq] & lt)] = v[qq];
          base += __popc(masks[qq]);
        }
      }
      bar512();
      int n_keep = sm.sel.list_cnt;
      if (last_chunk && b16_small) {
        // the top-16 lies in the kept keys: those above the 16th key's bucket,
        // and the members of that bucket
        for (int i0 = 0; i0 < n_keep; i0 += kWGThreads) {
          const int i = i0 + tid;
          const unsigned long long key = i < n_keep ? sm.keys[i] : 0ull;
          const int b = key != 0ull ? fixed_bucket(key) : -2;
          const bool top = b >= 0 && (b16 < 0 || b > b16);
          const bool bnd = b >= 0 && b16 >= 0 && b == b16;
          const int pt = warp_append(&sm.sel.n16, top);
          const int pb = warp_append(&sm.sel.nb16, bnd);
          if (top) sm.top16[pt] = key;
          if (bnd) sm.b16[pb] = key;
        }
      }
      for (int i = n_keep + tid; i < kKeysCap; i += kWGThreads) sm.keys[i] = 0ull;
      bar512();
      if (n_keep > (last_chunk ? kPubCap : kLocalK)) {  // a wide boundary bucket: reduce exactly to 512
        const int m = select_top(sm.keys, n_keep, kLocalK, sm.out, sm.hist, sm.sortbuf, sm.sel, tid);
        for (int i = tid; i < kKeysCap; i += kWGThreads) sm.keys[i] = i < m ? sm.out[i] : 0ull;
        bar512();
        n_keep = m;
      }
      carried = n_keep;
      // histogram of the carried keys for the next chunk
      for (int i = tid; i < kHistWords; i += kWGThreads) sm.hist[i] = 0u;
      bar512();
      if (!last_chunk) {
        for (int i = tid; i < carried; i += kWGThreads) hist_add(sm.hist, fixed_bucket(sm.keys[i]));
        bar512();
      }
    }

    // ---- exact top-16 of this CTA (sorted) and the list it publishes ---------
    const int m = carried;
    int n_top;
    if (m <= kTopM) {
      n_top = m;
      if (warp == 0) {
        const unsigned long long t = warp_sort32_desc(lane < m ? sm.keys[lane] : 0ull, lane);
        if (lane < kTopM) sm.top16[lane] = t;
      }
      bar512();
    } else if (sm.sel.c16_b >= 0 && sm.sel.c16_cnt <= 32) {
      // the keys above the 16th key's bucket, plus the best of that bucket
      const int n_above = sm.sel.n16, need = kTopM - n_above;
      if (warp == 0) {
        const unsigned long long bsorted = warp_sort32_desc(lane < sm.sel.nb16 ? sm.b16[lane] : 0ull, lane);
        const unsigned long long shifted = __shfl_sync(0xffffffffu, bsorted, (lane - n_above) & 31);
        const unsigned long long cand =
            lane < n_above ? sm.top16[lane] : (lane < n_above + need ? shifted : 0ull);
        const unsigned long long srt = warp_sort32_desc(cand, lane);
        if (lane < kTopM) sm.top16[lane] = srt;
      }
      bar512();
      n_top = kTopM;
    } else {
      // a wide 16th-key bucket: exact selection over the kept keys
      for (int i = tid; i < m; i += kWGThreads) sm.sortbuf[i] = sm.keys[i];
      bar512();
      const int n16 = select_top(sm.sortbuf, m, kTopM, sm.top16, sm.hist, sm.keys + kPubCap, sm.sel, tid);
      if (warp == 0) {
        const unsigned long long srt = warp_sort32_desc(lane < n16 ? sm.top16[lane] : 0ull, lane);
        if (lane < kTopM) sm.top16[lane] = srt;
      }
      bar512();
      n_top = kTopM;
    }
    const unsigned long long th = (m > kTopM) ? sm.top16[kTopM - 1] : 0ull;
    const int c = blockIdx.x;
    for (int i = tid; i < kTopM; i += kWGThreads) ws->lists[c][i] = i < n_top ? sm.top16[i] : 0ull;
    if (tid == 0) sm.sel.list_cnt = 0;
    bar512();
    for (int i0 = 0; i0 < m; i0 += kWGThreads) {
      const int i = i0 + tid;
      const unsigned long long key = i < m ? sm.keys[i] : ~0ull;
      const int p = warp_append(&sm.sel.list_cnt, key < th);
      if (key < th) ws->lists[c][kTopM + p] = key;
    }
    bar512();
    if (tid == 0) {
      ws->cnt[c] = kTopM + sm.sel.list_cnt;
      ws->th16[c] = th;
    }
    __threadfence();
    bar512();
    if (tid == 0) {
      const unsigned int ticket = atomicAdd(&hdr->ticket, 1u);
      sm.is_last = (ticket == unsigned(G - 1));
    }
    bar512();

    if (sm.is_last) {
      // ---- global merge (last CTA to finish) ----------------------------------
      __threadfence();
      const int kk = k;
      // the CTAs' top-16 lists, then the k largest of them, sorted
      {
        unsigned long long cand[8];  // all loads in flight before the stores
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int i = tid + q * kWGThreads;
          cand[q] = i < G * kTopM ? ld_cg(&ws->lists[i / kTopM][i % kTopM]) : 0ull;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) sm.keys[tid + q * kWGThreads] = cand[q];
      }
      bar512();
      int sel_n = merge_topk_sorted(sm.keys, G * kTopM, kk, sm.out, sm.hist,
                                    reinterpret_cast<uint32_t *>(sm.stage[0]), sm.sel, tid);
      bool sorted_ok = sel_n >= 0;
      if (!sorted_ok) sel_n = select_top(sm.keys, G * kTopM, kk, sm.out, sm.hist, sm.sortbuf, sm.sel, tid);
      unsigned long long cut = 0ull;
      if (sel_n == kk) {
        if (sorted_ok) {
          cut = sm.out[kk - 1];
        } else {
          unsigned long long m0 = ~0ull;
          for (int i = 0; i < sel_n; ++i) m0 = min(m0, sm.out[i]);
          cut = m0;
        }
      }
      // CTAs whose 16th key beats the k-th candidate may hold more winners
      // (select_top above reuses list_cnt, so reset it here)
      bar512();
      if (tid == 0) sm.sel.list_cnt = 0;
      bar512();
      for (int c0 = 0; c0 < G; c0 += kWGThreads) {
        const int cc = c0 + tid;
        const unsigned long long t16 = cc < G ? ld_cg(&ws->th16[cc]) : 0ull;
        const bool f = t16 != 0ull && t16 > cut;
        const int p = warp_append(&sm.sel.list_cnt, f);
        if (f) sm.fetch[p] = cc;
      }
      bar512();
      const int n_fetch = min(sm.sel.list_cnt, G);
      if (n_fetch == 0 && sorted_ok) {
        for (int e = tid; e < kk; e += kWGThreads) {
          if (e < sel_n) {
            out_idx[e] = key_index(sm.out[e]);
            if (out_score) out_score[e] = key_score(sm.out[e]);
          } else {
            out_idx[e] = -1;
            if (out_score) out_score[e] = __uint_as_float(0x7fc00000u);
          }
        }
      } else {
        // exact fallback: the current winners plus every flagged CTA's list
        for (int i = tid; i < kKeysCap; i += kWGThreads) sm.keys[i] = 0ull;
        bar512();
        for (int i = tid; i < sel_n; i += kWGThreads) sm.keys[i] = sm.out[i];
        int fill = sel_n;
        bar512();
        for (int f = 0; f < n_fetch; ++f) {
          const int cc = sm.fetch[f];
          const int extra = __ldcg(&ws->cnt[cc]) - kTopM;
          if (fill + extra > kKeysCap) {
            sel_n = select_top(sm.keys, fill, kk, sm.out, sm.hist, sm.sortbuf, sm.sel, tid);
            for (int i = tid; i < kKeysCap; i += kWGThreads) sm.keys[i] = i < sel_n ? sm.out[i] : 0ull;
            fill = sel_n;
            bar512();
          }
          for (int i = tid; i < extra; i += kWGThreads) sm.keys[fill + i] = ld_cg(&ws->lists[cc][kTopM + i]);
          fill += extra;
          bar512();
        }
        sel_n = select_top(sm.keys, fill, kk, sm.out, sm.hist, sm.sortbuf, sm.sel, tid);
        if (tid == 0) atomicAdd(&hdr->fallback, 1u);
        const unsigned long long srt = block_sort512_desc(tid < sel_n ? sm.out[tid] : 0ull, sm.sortbuf, tid);
        if (tid < kk) {
          if (tid < sel_n) {
            out_idx[tid] = key_index(srt);
            if (out_score) out_score[tid] = key_score(srt);
          } else {
            out_idx[tid] = -1;
            if (out_score) out_score[tid] = __uint_as_float(0x7fc00000u);
          }
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
