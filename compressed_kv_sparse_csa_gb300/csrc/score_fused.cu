// Fused CSA indexer score + exact top-k on the fifth-generation tensor cores.
//
// DS4X README, "Optimization details" / "CSA score/top-512 fusion": the
// scorer reads the packed 68-byte MXFP4 rows directly, every scorer CTA keeps
// an exact local top-512 of sortable (score, index) keys, and the local lists
// are merged into the exact top-512 without materialising the score array.
// This is a GB300 design of that method.  One persistent CTA per SM:
//
//  * warp 20 streams the CTA's contiguous range of 128-row tiles from HBM,
//    two tiles (17,408 bytes) per 1-D bulk copy, into a ring of five
//    shared-memory stages (fewer, larger copies keep the copy engine near the
//    HBM rate);
//  * converter warpgroups 0-1 (tile i: warpgroup i % 2, thread = row) move a
//    tile into tensor memory as the MMA's A operand: each E2M1 code gets its
//    own byte in bits 5-2 (the container is read as bits 5-0; bits 7-6 are
//    ignored), the even codes of each group of eight in one 32-bit column and
//    the odd ones in the next (a mask and a shift per column; the query
//    pieces are stored in the same K order), and the row's four UE8M0 bytes
//    go to the row's scale-factor column (four-slot ring);
//  * warps 21-23 (tile i by warp 21 + i % 3; a thread that waits on an
//    mbarrier stalls until its own MMAs drain, so three issuers keep the
//    tensor core fed) issue the tile's eight block-scaled tcgen05.mma
//    kind::mxf8f6f4 (M = 128 rows, N = 64 heads, K = 32; A = E2M1 keys with
//    their own UE8M0 scales, B = one of the query's two E4M3 pieces with its
//    UE8M0 scales per 32 elements; both pieces accumulate into the same fp32
//    accumulator slot of a five-slot tensor-memory ring), so the hardware
//    applies both sets of block scales and every row's 64 dot products come
//    out in fp32;
//  * epilogue warpgroups 2-4 (tile i: warpgroup 2 + i % 3) read a row's 64
//    accumulators back and form s = sum_h w_h * ReLU(acc_h) (one max and one
//    FMA per head); each key goes into shared memory and into a fixed
//    8,192-bucket histogram of its score bits;
//  * the rings' mbarriers are indexed by tile modulo a multiple of both the
//    ring size and the waiters' rotation, so every waiter waits on every
//    phase of its barriers;
//  * after the stream (threads 0-511) one scan of the histogram locates the CTA's 512th and
//    16th keys; one pass keeps the keys at or above the 512th key's bucket
//    (a superset of the local top-512) and collects the keys at or above the
//    16th key's bucket: the CTA's candidates, published unsorted with a
//    bound that every key it left out is below;
//  * the CTAs of a session meet at a bounded barrier (the launch is
//    cooperative, so all are resident); each then loads the session's
//    candidates at or above the largest bound and writes its own winners at
//    their ranks among them (direct counts for a few candidates, a counting
//    sort over 2048 buckets for more), so the merge runs in every CTA at
//    once instead of in the last one.  A CTA
//    whose bound beats the k-th key may hold more winners: then every such
//    CTA publishes its superset and the session's first CTA merges exactly.
//
// The bf16 query q is split per head and 32-element block into E4M3 pieces
// q = hi * 2^a + lo * 2^b, each with the block-scale rule of the cache writer
// (a the least exponent with max|q| <= 448 * 2^a, b the same for the
// remainder q - hi * 2^a).  The split is exact for every element within
// 2^-14 of its block's largest magnitude (both pieces then carry four of its
// eight significant bits); smaller elements keep their top bits.  E2M1 keys
// times E4M3 pieces are exact products; the tensor core sums them in fp32.
#include <cuda_fp16.h>

#include "ds4x_internal.cuh"
#include "tc_ptx.cuh"
#include "select512.cuh"

namespace ds4x {
namespace {

using namespace ptx;

constexpr int kTileRows = 128;
constexpr int kTileBytes = kTileRows * DS4X_IDX_ROW_BYTES;  // 8704
constexpr int kStageTiles = 2;             // tiles per bulk copy and stage: 17,408-byte copies keep
                                           // the copy engine near the HBM rate with few stages
constexpr int kStageBytes = kStageTiles * kTileBytes;
constexpr int kStages = 5;
constexpr int kConvWG = 2;                 // converter warpgroups: warps 0-7 (tile i: WG i % 2)
constexpr int kEpiWG = 3;                  // epilogue warpgroups: warps 8-19 (tile i: WG i % 3)
constexpr int kStreamThreads = 128 * (kConvWG + kEpiWG);  // 640
constexpr int kProducerWarp = kStreamThreads / 32;     // 20
constexpr int kMmaWarp = kProducerWarp + 1;            // 21: allocates tensor memory; 21-23 issue MMAs
constexpr int kMmaWarps = 3;                           // tile i is issued by warp kMmaWarp + i % 3
constexpr int kThreads = kStreamThreads + 32 * (1 + kMmaWarps);  // 768
constexpr int kASlots = 4;                 // tensor-memory A ring
constexpr int kDSlots = 5;                 // tensor-memory accumulator ring
// mbarriers indexed by tile modulo a multiple of both the ring size and the
// waiters' rotation, so each waiter waits on every phase of its barriers
constexpr int kAFullBars = 12;             // afull[i % 12]: waited by issuer i % 3
constexpr int kDFullBars = 15;             // dfull[i % 15]: waited by epilogue WG i % 3
constexpr int kChunkTiles = 64;
constexpr int kLocalK = DS4X_TOPK_MAX;     // 512
// Keys carried from one chunk to the next: every key at or above the bucket
// of the CTA's 512th, at most 1024 of them (an exact selection cuts them to
// 512 only beyond that).
constexpr int kCarry = 2 * kLocalK;         // 1024
constexpr int kKeysCap = kCarry + kChunkTiles * kTileRows;  // 9216
constexpr int kTopM = 16;                  // fewest candidates a CTA publishes
constexpr int kCandCap = kLocalK + 64;     // candidates a CTA may publish (its top M and their bucket)
constexpr int kPubCap = 1024;              // pool slots per CTA; keys a flagged CTA may publish
constexpr int kPoolPer = 8;                // pool keys each selection thread holds in registers
constexpr int kPoolCap = kPoolPer * kSelThreads;  // 4096: larger pools take the exact fallback
constexpr int kRadixBuckets = 2048;        // counting-sort buckets over the kept pool keys
constexpr int kRankStep = 8;              // candidates ranked together (lane j stores candidate j's partial)
constexpr int kDirect = 16;                // up to this many candidates a CTA ranks by direct counts
constexpr int kBuckets = 8192;             // fixed score-bit histogram (16-bit counters, 2 per word)
constexpr int kHistWords = 4096;
constexpr int kMaxCtas = 256;
constexpr int kMaxSess = 256;              // sessions one launch may score (the batched API allows
                                           // DS4X_MAX_SESSIONS; the prefill path one per CTA)
constexpr int kTmemCols = 512;
static_assert(kMaxSess >= kMaxCtas && kMaxSess >= DS4X_MAX_SESSIONS, "one session per CTA fits");
constexpr int kN = DS4X_IDX_HEADS;         // 64 heads per MMA; B rows 0-63 hold the hi pieces, 64-127 the lo pieces
constexpr uint32_t kDCol0 = 0;             // D slot j: columns [64 j, 64 j + 64)
constexpr uint32_t kACol0 = 64 * kDSlots;  // A slot a: 32 columns from kACol0 + 32 a
constexpr uint32_t kSfaCol0 = kACol0 + 32 * kASlots;  // SFA of A slot a: 4 columns from kSfaCol0 + 4 a
constexpr uint32_t kSfbCol = kSfaCol0 + 4 * kASlots;  // SFB of the hi pieces: columns +0, +1
constexpr uint32_t kSfbLoCol = kSfbCol + 4;           // SFB of the lo pieces: columns +0, +1
constexpr uint32_t kOpBytes = 128 * DS4X_IDX_DIM;  // 16384: 128 rows x 8 K chunks of 16 bytes
constexpr uint32_t kLbo = 128;             // next 16-element K chunk
constexpr uint32_t kSbo = 8 * 128;         // next 8 rows
constexpr uint32_t kIdesc = idesc_mxf8f6f4_e2m1_e4m3(kN);
constexpr unsigned long long kTimeoutNs = 500ull * 1000 * 1000;  // a bounded wait gives up after 0.5 s
constexpr uint32_t kBarStream = 2;         // named barrier of the 640 converter and epilogue threads
// An mbarrier parity wait for phase c passes early if phase c - 1 is still
// open, so each parity wait below is done by a thread (or warpgroup) that also
// waited for the slot's previous phase: the slot counts are multiples of the
// waiters' rotation.  The MMA warps' wait for a free accumulator slot (three
// issuers, four slots) uses a monotonic counter instead (drel: each epilogue
// warp adds one with release semantics once it has read its lanes).
static_assert(kStageTiles == kConvWG, "each converter warpgroup takes one tile of every stage");
static_assert(kASlots % kConvWG == 0, "an A slot's empty phases: one converter WG");
static_assert(kAFullBars % kASlots == 0 && kAFullBars % kMmaWarps == 0, "afull: one issuer per barrier");
static_assert(kDFullBars % kDSlots == 0 && kDFullBars % kEpiWG == 0, "dfull: one epilogue WG per barrier");
static_assert(kDSlots * 64 <= int(kACol0) && kACol0 + 32 * kASlots <= kSfaCol0 && kSfbLoCol + 4 <= uint32_t(kTmemCols),
              "tensor-memory map");
static_assert(kSfaCol0 % 4 == 0 && kSfbCol % 4 == 0 && kSfbLoCol % 4 == 0,
              "scale-factor columns start on a 4-column boundary");
static_assert(kSelPerThread * kSelThreads >= kKeysCap, "selection registers cover the key buffer");
static_assert(kKeysCap * 8 <= kStages * kStageBytes, "the key buffer fits the stage ring (the exact top-M copy)");
constexpr int kMaxDynSmem = 232448;         // 227 KB per CTA on sm_103

// Byte offset of (row r, K element kk) in a canonical no-swizzle K-major
// operand of 8-bit containers with 16-element chunks.
__device__ __forceinline__ uint32_t op_offset(int r, int kk) {
  return uint32_t(r >> 3) * kSbo + uint32_t(kk >> 4) * kLbo + uint32_t(r & 7) * 16 + uint32_t(kk & 15);
}

struct __align__(1024) Smem {
  uint8_t bq[kOpBytes];                       // query pieces, E4M3, canonical K-major (B)
  uint8_t stage[kStages][kStageBytes];        // raw tile ring, two tiles a stage
  unsigned long long keys[kKeysCap];          // [0, 1024): carried keys; then the chunk's keys
  unsigned long long out[kLocalK];
  unsigned long long sortbuf[2 * kLocalK];
  alignas(16) uint32_t hist[kHistWords];      // fixed histogram, or the adaptive one inside select_top
  alignas(16) float wq[DS4X_IDX_HEADS];       // head weights
  uint8_t sfb[2 * DS4X_IDX_HEADS][4];         // query-piece scale bytes per 32-element block (hi rows, lo rows)
  unsigned long long full[kStages], empty[kStages];
  unsigned long long afull[kAFullBars], aempty[kASlots], dfull[kDFullBars];
  int drel[kDSlots];                          // warps of the epilogue that released the slot so far
  unsigned long long epoch_full;               // the producer has stored `epoch`
  SelShared sel;
  unsigned long long cand[kCandCap];          // this CTA's candidates
  unsigned long long th;                      // ... and the bound on the keys it left out
  uint32_t epoch;                             // the session's exchange count at launch
  uint32_t tmem_base;
  int abort_flag;
};

// Per-session exchange words.  A launch with epoch e uses the words of
// parity e & 1; the session's first CTA clears the other parity (the next
// exchange's) before it arrives, and advances the epoch once every CTA has
// arrived, so no word is cleared while a CTA of its exchange still reads it.
struct alignas(128) SessSync {
  unsigned long long main[2];  // arrivals << 32 | candidate slots reserved
  unsigned long long fb[2];    // arrivals at the fallback barrier
  unsigned long long thm[2];   // largest bound of the session's CTAs
  uint32_t epoch;              // exchanges completed
};

struct FusedWs {
  WsHeader hdr;
  SessSync sync[kMaxSess];
  unsigned long long pool[kMaxCtas * kPubCap];  // session s: slots [cta0 * kPubCap, (cta0 + Gs) * kPubCap)
  unsigned long long lists[kMaxCtas][kPubCap];  // per CTA, when flagged: its local top-k below its bound
  int cnt[kMaxCtas];
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

// (a0, a1) = (w0 * x0 + a0, w1 * x1 + a1), each rounded once (one packed FMA).
__device__ __forceinline__ void fma_f32x2(float &a0, float &a1, float w0, float w1, float x0, float x1) {
  asm("{\n\t.reg .b64 a, w, x;\n\tmov.b64 a, {%0, %1};\n\tmov.b64 w, {%2, %3};\n\tmov.b64 x, {%4, %5};\n\t"
      "fma.rn.f32x2 a, w, x, a;\n\tmov.b64 {%0, %1}, a;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(w0), "f"(w1), "f"(x0), "f"(x1));
}

__device__ __forceinline__ void red_release_add_shared(int *p, int v) {
  asm volatile("red.release.cta.shared::cta.add.s32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_shared(const int *p) {
  int v;
  asm volatile("ld.acquire.cta.shared::cta.s32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}

// Bounded wait until the monotonic counter *p reaches target (same time-out
// and abort rules as wait_bar).
__device__ bool wait_seq(Smem &sm, const int *p, int target, WsHeader *hdr) {
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

// Bounded wait used only while shutting down after a time-out, so that no
// bulk copy or MMA is still writing into this CTA's memory when it exits.
__device__ void drain_bar(unsigned long long *bar, uint32_t parity) {
  const uint32_t b = smem_u32(bar);
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(b, parity) && globaltimer() - t0 < kTimeoutNs / 5) {
  }
}

// Two E4M3 codes (low byte: the first) -> their values, exactly (through f16x2).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two_codes) {
  uint32_t h2;
  asm("{ .reg .b16 c; cvt.u16.u32 c, %1; cvt.rn.f16x2.e4m3x2 %0, c; }" : "=r"(h2) : "r"(two_codes));
  return __half22float2(*reinterpret_cast<const __half2 *>(&h2));
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

// all converter and epilogue threads (the chunk ends)
__device__ __forceinline__ void bar_stream() { named_bar_sync(kBarStream, kStreamThreads); }

// Ranks of cand[0, nc) (this CTA's keys, all among pool[0, n)) among the n
// distinct nonzero keys of pool[0, n), all in [lo, hi]: a counting sort over
// 2048 buckets spanning [lo, hi] (bucket 0: the top), so a key's rank is the
// number of keys in higher buckets plus those of its own bucket above it.
// A candidate of rank r < k goes to out_idx[r] (and out_score[r]).
// hist[0, 2048) must be zero on entry; sorted holds n keys.
__device__ void bucket_rank(const unsigned long long *pool, int n, const unsigned long long *cand, int nc,
                            unsigned long long lo, unsigned long long hi, int k, uint32_t *hist,
                            unsigned long long *sorted, SelShared &sh, int tid, int32_t *out_idx,
                            float *out_score) {
  constexpr int kB = kRadixBuckets;
  static_assert(kB == 4 * kSelThreads, "four buckets per thread");
  const int lane = tid & 31, warp = tid >> 5;
  const unsigned long long range = hi - lo;
  const int shift = range < kB ? 0 : (64 - __clzll((long long)range)) - 11;  // range >> shift < 2048
  auto bucket = [&](unsigned long long x) { return kB - 1 - int((x - lo) >> shift); };
  for (int i = tid; i < n; i += kSelThreads) atomicAdd(&hist[bucket(pool[i])], 1u);
  bar512();
  {  // exclusive scan in place: hist[b] = keys in the buckets above b (thread t: buckets 4t .. 4t + 3)
    const uint4 c4 = reinterpret_cast<const uint4 *>(hist)[tid];
    const int local = int(c4.x + c4.y + c4.z + c4.w);
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) sh.scan[warp] = incl;
    bar512();
    int above = incl - local;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int4 sc4 = reinterpret_cast<const int4 *>(sh.scan)[j];
      above += (4 * j < warp ? sc4.x : 0) + (4 * j + 1 < warp ? sc4.y : 0) + (4 * j + 2 < warp ? sc4.z : 0) +
               (4 * j + 3 < warp ? sc4.w : 0);
    }
    const uint32_t a0 = uint32_t(above), a1 = a0 + c4.x, a2 = a1 + c4.y, a3 = a2 + c4.z;
    reinterpret_cast<uint4 *>(hist)[tid] = make_uint4(a0, a1, a2, a3);
  }
  bar512();
  for (int i = tid; i < n; i += kSelThreads) {  // counting-sort scatter: bucket by bucket, from the top
    const unsigned long long x = pool[i];
    sorted[atomicAdd(&hist[bucket(x)], 1u)] = x;
  }
  bar512();
  // hist[b] is now the end of bucket b, the start of bucket b + 1
  for (int e = tid; e < nc; e += kSelThreads) {
    const unsigned long long x = cand[e];
    const int b = bucket(x);
    const int s0 = b == 0 ? 0 : int(hist[b - 1]), s1 = int(hist[b]);
    int r = s0;
    for (int j = s0; j < s1; ++j) r += sorted[j] > x ? 1 : 0;
    if (r < k) {
      out_idx[r] = key_index(x);
      if (out_score) out_score[r] = key_score(x);
    }
  }
}

// Grid-scope release add and acquire load (the arrival and the poll of the
// session exchange).
__device__ __forceinline__ void red_release_add(unsigned long long *p, unsigned long long v) {
  asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Thread 0 of a CTA: wait (bounded) until the arrival count in bits 32-63 of
// *word reaches Gs; returns false (status DS4X_ETIMEOUT) on time-out.
__device__ bool wait_arrivals(const unsigned long long *word, unsigned int Gs, WsHeader *hdr,
                              unsigned long long *seen) {
  const unsigned long long t0 = globaltimer();
  while (true) {
    const unsigned long long wv = ld_acquire(word);
    if (uint32_t(wv >> 32) >= Gs) {
      *seen = wv;
      return true;
    }
    if (globaltimer() - t0 > kTimeoutNs) {
      atomicExch(&hdr->status, int32_t(DS4X_ETIMEOUT));
      return false;
    }
  }
}

// Cuts of the fixed histogram at the 512 and the M largest keys: the bucket
// holding the K-th key, the number of keys in higher buckets and (for K = M)
// in that bucket.  b = -1 when there are at most K keys.  Also clears the
// candidate counter.
__device__ void hist_cuts(const uint32_t *hist, SelShared &sh, int tid, int M) {
  const int lane = tid & 31, warp = tid >> 5;
  // thread t owns words [4095 - 8t - 7, 4095 - 8t] = buckets [8191 - 16t - 15, 8191 - 16t],
  // read as two 16-byte vectors (word-strided reads would conflict 8 ways)
  const uint4 lo4 = reinterpret_cast<const uint4 *>(hist)[(kHistWords - 8 - 8 * tid) / 4];
  const uint4 hi4 = reinterpret_cast<const uint4 *>(hist)[(kHistWords - 4 - 8 * tid) / 4];
  const uint32_t wd[8] = {hi4.w, hi4.z, hi4.y, hi4.x, lo4.w, lo4.z, lo4.y, lo4.x};  // word 4095 - 8t - q
  // bucket 8191 - 16t - q: the odd (higher) half of word q / 2 first
  auto count = [&](int q) { return int((q & 1) ? (wd[q >> 1] & 0xffffu) : (wd[q >> 1] >> 16)); };
  int local = 0;
#pragma unroll
  for (int q = 0; q < 8; ++q) local += int((wd[q] >> 16) + (wd[q] & 0xffffu));
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sh.scan[warp] = incl;
  if (tid == 0) {
    sh.c512_b = -1;
    sh.cM_b = -1;
    sh.cM_above = 0;
    sh.cM_cnt = 0;
    sh.fill = 0;
  }
  bar512();
  int above = incl - local, total = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int4 sc = reinterpret_cast<const int4 *>(sh.scan)[j];
    above += (4 * j < warp ? sc.x : 0) + (4 * j + 1 < warp ? sc.y : 0) + (4 * j + 2 < warp ? sc.z : 0) +
             (4 * j + 3 < warp ? sc.w : 0);
    total += sc.x + sc.y + sc.z + sc.w;
  }
  const int bhigh = kBuckets - 1 - 16 * tid;
  if (above < kLocalK && above + local >= kLocalK) {
    int acc = above;
    bool found = false;
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int cq = count(q);
      if (!found && acc + cq >= kLocalK) {
        found = true;
        sh.c512_b = bhigh - q;
        sh.c512_above = acc;
      }
      acc += cq;
    }
  }
  if (above < M && above + local >= M) {
    int acc = above;
    bool found = false;
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int cq = count(q);
      if (!found && acc + cq >= M) {
        found = true;
        sh.cM_b = bhigh - q;
        sh.cM_above = acc;
        sh.cM_cnt = cq;
      }
      acc += cq;
    }
  }
  if (tid == 0) sh.total = total;
  bar512();
}

__global__ void __launch_bounds__(kThreads, 1)
score_fused_kernel(ScoreBatch sb, FusedWs *__restrict__ ws) {
  // Launched as a programmatic dependent of the previous kernel (the append
  // of the step's new row, or the previous step's attention): its CTAs may be
  // resident early; nothing is read or written before that kernel completes.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  extern __shared__ uint8_t smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  // ---- this CTA's session and its tile range ------------------------------
  // One session: every CTA of the grid.  A batch: the CTAs are split across
  // the sessions in proportion to their tile counts, at least one each, by
  // the same arithmetic in every CTA; CTAs past the split have no work.
  int sess = 0, cta0 = 0, Gs = gridDim.x;
  const uint8_t *rows = sb.rows;
  int64_t n_rows = sb.n_rows;
  if (sb.rows_arr != nullptr) {
    int64_t total = 0;
    for (int s = 0; s < sb.n_sess; ++s) {
      const int64_t nr = sb.n_arr[s];
      total += nr > 0 ? (nr + kTileRows - 1) / kTileRows : 1;
    }
    const int64_t spare = int64_t(gridDim.x) - sb.n_sess;
    int prefix = 0;
    bool found = false;
    for (int s = 0; s < sb.n_sess; ++s) {
      const int64_t nr = sb.n_arr[s];
      const int64_t t = nr > 0 ? (nr + kTileRows - 1) / kTileRows : 1;
      const int64_t share = 1 + spare * t / total;
      const int g = int(share < t ? share : t);
      if (!found && int(blockIdx.x) < prefix + g) {
        sess = s;
        cta0 = prefix;
        Gs = g;
        found = true;
      }
      prefix += g;
    }
    if (!found) return;  // uniform across the CTA, before any barrier or allocation
    rows = sb.rows_arr[sess];
    n_rows = sb.n_arr[sess] > 0 ? sb.n_arr[sess] : 0;
  }
  const uint16_t *__restrict__ q = sb.q + size_t(sess) * DS4X_IDX_HEADS * DS4X_IDX_DIM;
  const float *__restrict__ w = sb.w + size_t(sess) * DS4X_IDX_HEADS;
  const int k = sb.k;
  int32_t *__restrict__ out_idx = sb.out_idx + size_t(sess) * k;
  float *__restrict__ out_score = sb.out_score != nullptr ? sb.out_score + size_t(sess) * k : nullptr;
  const int64_t n_tiles_total = (n_rows + kTileRows - 1) / kTileRows;
  const int64_t tile_begin = n_tiles_total * (blockIdx.x - cta0) / Gs;
  const int64_t tile_end = n_tiles_total * (blockIdx.x - cta0 + 1) / Gs;
  const int n_tiles = int(tile_end - tile_begin);
  WsHeader *hdr = &ws->hdr;

  // tiles 2j and 2j + 1 of this CTA -> stage j % kStages, one bulk copy (producer thread)
  const int n_stage_copies = (n_tiles + kStageTiles - 1) / kStageTiles;
  auto issue_stage = [&](int j) {
    const int s = j % kStages;
    const int64_t r0 = (tile_begin + int64_t(kStageTiles) * j) * kTileRows;
    const int64_t left = n_rows - r0;
    const int nr = left < kStageTiles * kTileRows ? int(left) : kStageTiles * kTileRows;
    const uint32_t bytes = uint32_t(nr) * DS4X_IDX_ROW_BYTES;
    const uint32_t bulk = bytes & ~15u;
    const uint8_t *src = rows + r0 * DS4X_IDX_ROW_BYTES;
    for (uint32_t b = bulk; b < bytes; b += 4)  // ragged tail of the last tile
      *reinterpret_cast<uint32_t *>(sm.stage[s] + b) = *reinterpret_cast<const uint32_t *>(src + b);
    mbar_arrive_expect_tx(smem_u32(&sm.full[s]), bulk);
    bulk_g2s_hint(smem_u32(sm.stage[s]), src, bulk, smem_u32(&sm.full[s]), l2_evict_first_policy());
  };

  // ---- set-up -------------------------------------------------------------
  if (tid == kProducerWarp * 32) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), kStageTiles * kTileRows);  // each converter thread, once per stage
    }
    for (int j = 0; j < kAFullBars; ++j) mbar_init(smem_u32(&sm.afull[j]), kTileRows);
    for (int j = 0; j < kASlots; ++j) mbar_init(smem_u32(&sm.aempty[j]), 1);
    for (int j = 0; j < kDFullBars; ++j) mbar_init(smem_u32(&sm.dfull[j]), 1);
    for (int j = 0; j < kDSlots; ++j) sm.drel[j] = 0;
    mbar_init(smem_u32(&sm.epoch_full), 1);
    sm.abort_flag = 0;
    fence_mbar_init();
    // the first stages go out now, under the set-up below
    for (int j = 0; j < kStages && j < n_stage_copies; ++j) issue_stage(j);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&sm.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  bool lo_nonzero = false;
  if (tid < kSelThreads) {
    // query -> two E4M3 pieces per 32-element block (B rows h and 64 + h);
    // thread t < 256 takes head t / 4, block t % 4 (32 elements, 64 bytes)
    if (tid < DS4X_IDX_HEADS * 4) {
      const int h = tid >> 2, b = tid & 3;
      const uint4 *src = reinterpret_cast<const uint4 *>(q + h * DS4X_IDX_DIM + 32 * b);
      uint4 raw[4];
#pragma unroll
      for (int v = 0; v < 4; ++v) raw[v] = src[v];
      float x[32];
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const uint32_t wv[4] = {raw[v].x, raw[v].y, raw[v].z, raw[v].w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          x[8 * v + 2 * u] = __uint_as_float(wv[u] << 16);
          x[8 * v + 2 * u + 1] = __uint_as_float(wv[u] & 0xffff0000u);
        }
      }
      float amax = 0.0f;
#pragma unroll
      for (int e = 0; e < 32; ++e) amax = fmaxf(amax, fabsf(x[e]));
      const int e_hi = block_exponent(amax, 0.875f, 9);  // 448 = 0.875 * 2^9
      const float s_hi = pow2_neg(e_hi), u_hi = pow2_neg(-e_hi);
      uint32_t hw[8];
      float rmax = 0.0f;
#pragma unroll
      for (int j = 0; j < 16; ++j) {  // elements 2j, 2j+1
        const uint32_t c2 = cvt_e4m3x2(x[2 * j + 1] * s_hi, x[2 * j] * s_hi);
        const float2 hv = e4m3x2_to_float2(c2);
        x[2 * j] -= hv.x * u_hi;  // exact remainders
        x[2 * j + 1] -= hv.y * u_hi;
        rmax = fmaxf(rmax, fmaxf(fabsf(x[2 * j]), fabsf(x[2 * j + 1])));
        if (j & 1) hw[j >> 1] |= c2 << 16; else hw[j >> 1] = c2;
      }
      const int e_lo = block_exponent(rmax, 0.875f, 9);
      const float s_lo = pow2_neg(e_lo);
      uint32_t lw[8];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t c2 = cvt_e4m3x2(x[2 * j + 1] * s_lo, x[2 * j] * s_lo);
        if (j & 1) lw[j >> 1] |= c2 << 16; else lw[j >> 1] = c2;
      }
      // elements 32 b .. 32 b + 31 are two 16-element chunks of rows h and 64 + h,
      // each group of eight in the converter's K order (even elements, then odd)
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const uint32_t a = hw[2 * g], c = hw[2 * g + 1], la = lw[2 * g], lc = lw[2 * g + 1];
        hw[2 * g] = __byte_perm(a, c, 0x6420);
        hw[2 * g + 1] = __byte_perm(a, c, 0x7531);
        lw[2 * g] = __byte_perm(la, lc, 0x6420);
        lw[2 * g + 1] = __byte_perm(la, lc, 0x7531);
      }
      *reinterpret_cast<uint4 *>(sm.bq + op_offset(h, 32 * b)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      *reinterpret_cast<uint4 *>(sm.bq + op_offset(h, 32 * b + 16)) = make_uint4(hw[4], hw[5], hw[6], hw[7]);
      *reinterpret_cast<uint4 *>(sm.bq + op_offset(DS4X_IDX_HEADS + h, 32 * b)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      *reinterpret_cast<uint4 *>(sm.bq + op_offset(DS4X_IDX_HEADS + h, 32 * b + 16)) =
          make_uint4(lw[4], lw[5], lw[6], lw[7]);
      sm.sfb[h][b] = uint8_t(e_hi + 127);
      sm.sfb[DS4X_IDX_HEADS + h][b] = uint8_t(e_lo + 127);
#pragma unroll
      for (int j = 0; j < 8; ++j) lo_nonzero |= (lw[j] & 0x7f7f7f7fu) != 0u;  // any nonzero lo code (0x80 is -0)
    }
    for (int h = tid; h < DS4X_IDX_HEADS; h += kSelThreads) sm.wq[h] = w[h];
    for (int i = tid; i < kKeysCap; i += kSelThreads) sm.keys[i] = 0ull;
    for (int i = tid; i < kHistWords; i += kSelThreads) sm.hist[i] = 0u;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  // the barrier also tells every thread whether the query has a lo piece: a
  // query that is exact in E4M3 (prefill) needs only the hi MMAs
  const bool lo_any = __syncthreads_or(lo_nonzero ? 1 : 0) != 0;
  tc_fence_after();
  const uint32_t tmem_base = sm.tmem_base;
  if (warp < 4) {
    // query-piece scale factors: column n of a 64-row B piece reads lane
    // n % 32 of every sub-partition, column base + n / 32, byte = K block
    uint32_t v[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) v[c] = *reinterpret_cast<const uint32_t *>(sm.sfb[32 * c + lane]);
    const uint32_t lanes = uint32_t(32 * warp) << 16;
    tc_st_x4(tmem_base + lanes + kSfbCol, v[0], v[1], 0u, 0u);
    tc_st_x4(tmem_base + lanes + kSfbLoCol, v[2], v[3], 0u, 0u);
    tc_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == kProducerWarp) {
    // ---- producer: bulk-copy tiles into the stage ring ---------------------
    if (lane == 0) {
      // the session's exchange count, needed only after the stream: loaded now,
      // stored once the copies are out
      uint32_t epoch;
      asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(epoch) : "l"(&ws->sync[sess].epoch) : "memory");
      int issued = min(kStages, n_stage_copies);  // issued during the set-up
      for (int j = issued; j < n_stage_copies; ++j) {
        if (!wait_bar(sm, &sm.empty[j % kStages], ((j / kStages) - 1) & 1, hdr)) break;
        issue_stage(j);
        issued = j + 1;
      }
      sm.epoch = epoch;
      mbar_arrive(smem_u32(&sm.epoch_full));
      if (*reinterpret_cast<volatile int *>(&sm.abort_flag)) {
        for (int j = max(0, issued - kStages); j < issued; ++j) drain_bar(&sm.full[j % kStages], (j / kStages) & 1);
      }
    }
  } else if (warp >= kMmaWarp) {
    // ---- MMA issuers: warp kMmaWarp + m takes tiles m, m + 3, ... ------------
    if (lane == 0) {
      const uint64_t bdesc_hi = smem_desc_noswizzle(smem_u32(sm.bq), kLbo, kSbo);
      const uint64_t bdesc_lo = smem_desc_noswizzle(smem_u32(sm.bq + op_offset(DS4X_IDX_HEADS, 0)), kLbo, kSbo);
      int issued = 0;
      for (int i = warp - kMmaWarp; i < n_tiles; i += kMmaWarps) {
        const int a = i % kASlots, d = i % kDSlots;
        if (!wait_bar(sm, &sm.afull[i % kAFullBars], (i / kAFullBars) & 1, hdr)) break;
        // slot d's earlier uses (tiles i - kDSlots, i - 2 kDSlots, ...) each end with four releases
        if (i >= kDSlots && !wait_seq(sm, &sm.drel[d], 4 * (i / kDSlots), hdr)) break;
        tc_fence_after();
        if (lo_any)
          mma_mxf8f6f4_ta_k128_2b(tmem_base + kDCol0 + uint32_t(64 * d), tmem_base + kACol0 + uint32_t(32 * a),
                                  bdesc_hi, bdesc_lo, kIdesc, tmem_base + kSfaCol0 + uint32_t(4 * a),
                                  tmem_base + kSfbCol, tmem_base + kSfbLoCol);
        else
          mma_mxf8f6f4_ta_k128_1b(tmem_base + kDCol0 + uint32_t(64 * d), tmem_base + kACol0 + uint32_t(32 * a),
                                  bdesc_hi, kIdesc, tmem_base + kSfaCol0 + uint32_t(4 * a), tmem_base + kSfbCol);
        tc_commit(smem_u32(&sm.aempty[a]));
        tc_commit(smem_u32(&sm.dfull[i % kDFullBars]));
        issued = i + 1;
      }
      if (*reinterpret_cast<volatile int *>(&sm.abort_flag) && issued > 0) {
        const int i = issued - 1;  // this thread's last commit covers all of its MMAs
        drain_bar(&sm.dfull[i % kDFullBars], (i / kDFullBars) & 1);
      }
    }
  } else if (warp < kProducerWarp) {
    const int r = tid & 127;  // row within the tile == TMEM lane
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    const bool is_conv = warp < 4 * kConvWG;
    const int role_wg = is_conv ? warp / 4 : (warp - 4 * kConvWG) / 4;
    const int n_role_wg = is_conv ? kConvWG : kEpiWG;
    int last_n_in = 0;  // keys of the last chunk, in keys[0, last_n_in) (carried ones first)
    for (int c0 = 0; c0 < n_tiles; c0 += kChunkTiles) {
      const int c1 = min(n_tiles, c0 + kChunkTiles);
      for (int i = c0 + role_wg; i < c1; i += n_role_wg) {
        if (is_conv) {
          // ---- raw row -> A slot (one code per byte) + scale-factor word -----
          const int j = i / kStageTiles, st = j % kStages, a = i % kASlots;
          wait_bar(sm, &sm.full[st], (j / kStages) & 1, hdr);
          uint32_t wd[17];
          const uint32_t *rp = reinterpret_cast<const uint32_t *>(sm.stage[st] + (i % kStageTiles) * kTileBytes +
                                                                   r * DS4X_IDX_ROW_BYTES);
#pragma unroll
          for (int t = 0; t < 17; ++t) wd[t] = rp[t];
          mbar_arrive(smem_u32(&sm.empty[st]));
          if (i >= kASlots) wait_bar(sm, &sm.aempty[a], ((i / kASlots) - 1) & 1, hdr);
          // word t holds codes 8t..8t+7 (even code in the low nibble).  Each
          // code goes to its own byte, in bits 5-2 with bits 1-0 clear (the
          // container reads bits 5-0; bits 7-6 are ignored); column 2t takes the
          // even codes 8t, 8t+2, 8t+4, 8t+6 and column 2t+1 the odd ones, so K
          // runs in that order within each group of eight (the query pieces
          // are stored in the same order; a block's 32 codes stay in its four
          // columns, so the block scales are untouched)
          uint32_t av[32];
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            av[2 * t] = (wd[t] & 0x0f0f0f0fu) << 2;
            av[2 * t + 1] = (wd[t] & 0xf0f0f0f0u) >> 2;
          }
          tc_st_x32(tmem_base + lane_base + kACol0 + uint32_t(32 * a), av);
          // row r's scales: lane r, column kSfaCol0 + 4 a + r / 32
          tc_st_x1(tmem_base + lane_base + kSfaCol0 + uint32_t(4 * a + (warp & 3)), wd[16]);
          tc_wait_st();
          tc_fence_before();
          mbar_arrive(smem_u32(&sm.afull[i % kAFullBars]));
        } else {
          // ---- epilogue: accumulators -> score -> key --------------------------
          const int d = i % kDSlots;
          const bool ok = wait_bar(sm, &sm.dfull[i % kDFullBars], (i / kDFullBars) & 1, hdr);
          tc_fence_after();
          const uint32_t d_t = tmem_base + lane_base + kDCol0 + uint32_t(64 * d);
          const float4 *w4 = reinterpret_cast<const float4 *>(sm.wq);
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t v0[16], v1[16];
            tc_ld_x16(d_t + uint32_t(32 * half), v0);
            tc_ld_x16(d_t + uint32_t(32 * half + 16), v1);
            tc_wait_ld();
            if (half == 1) {
              // this warp has read its 32 lanes of the slot: count one release
              tc_fence_before();
              __syncwarp();
              if (lane == 0) red_release_add_shared(&sm.drel[d], 1);
            }
#pragma unroll
            for (int g = 0; g < 8; ++g) {  // heads 32 half + 4 g .. + 3
              const float4 wv = w4[8 * half + g];
              const uint32_t *v = g < 4 ? v0 + 4 * g : v1 + 4 * (g - 4);
              fma_f32x2(acc[0], acc[1], wv.x, wv.y, fmaxf(__uint_as_float(v[0]), 0.0f),
                        fmaxf(__uint_as_float(v[1]), 0.0f));
              fma_f32x2(acc[2], acc[3], wv.z, wv.w, fmaxf(__uint_as_float(v[2]), 0.0f),
                        fmaxf(__uint_as_float(v[3]), 0.0f));
            }
          }
          const float s_row = (acc[0] + acc[1]) + (acc[2] + acc[3]);
          const int64_t row = (tile_begin + i) * kTileRows + r;
          unsigned long long key = 0ull;
          if (ok && row < n_rows) {
            key = make_key(s_row, uint32_t(row));
            hist_add(sm.hist, fixed_bucket(key));
          }
          sm.keys[kCarry + (i - c0) * kTileRows + r] = key;
        }
      }
      bar_stream();

      // ---- end of chunk ---------------------------------------------------------
      const int n_in = kCarry + (c1 - c0) * kTileRows;
      if (c1 == n_tiles) {  // the last chunk's keys stay in place for the exchange below
        last_n_in = n_in;
        break;
      }
      if (tid < kSelThreads) {  // threads 512-639 (the third epilogue warpgroup) wait below
        // keep a superset of the local top-512 for the next chunk
        hist_cuts(sm.hist, sm.sel, tid, kTopM);
        const int b512 = sm.sel.c512_b;  // -1: at most 512 keys, keep all
        unsigned long long v[kSelPerThread];
  #pragma unroll
        for (int qq = 0; qq < kSelPerThread; ++qq) {
          const int i = tid + qq * kSelThreads;
          v[qq] = i < n_in ? sm.keys[i] : 0ull;
        }
        if (tid == 0) sm.sel.list_cnt = 0;
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
        // the rest of the carried region is zero (the chunk region is rewritten whole)
        for (int i = n_keep + tid; i < kCarry; i += kSelThreads) sm.keys[i] = 0ull;
        bar512();
        if (n_keep > kCarry) {  // a very wide boundary bucket: reduce exactly to 512
          const int m = select_top(sm.keys, n_keep, kLocalK, sm.out, sm.hist, sm.sortbuf, sm.sel, tid);
          for (int i = tid; i < kCarry; i += kSelThreads) sm.keys[i] = i < m ? sm.out[i] : 0ull;
          bar512();
          n_keep = m;
        }
        // histogram of the carried keys for the next chunk
        for (int i = tid; i < kHistWords; i += kSelThreads) sm.hist[i] = 0u;
        bar512();
        for (int i = tid; i < n_keep; i += kSelThreads) hist_add(sm.hist, fixed_bucket(sm.keys[i]));
        bar512();
      }
      bar_stream();
    }

    if (tid < kSelThreads) {  // the exchange: threads 0-511
      // The next kernel in the stream (the attention, launched as a programmatic
      // dependent) may take an SM as soon as this grid's CTAs leave; it waits
      // for the whole grid before it reads the indices.
      if (tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

      // ---- this CTA's candidates ------------------------------------------------
      // The CTA publishes its keys down to the bucket of its M-th key (all of
      // them when it has few) with a bound th that every key it leaves out is
      // below.  M covers about k / Gs winners per CTA with a wide margin; any M
      // gives the exact result, a small one only makes the fallback likelier.
      if (tid == 0) sm.sel.ok = wait_bar(sm, &sm.epoch_full, 0, hdr) && !*reinterpret_cast<volatile int *>(&sm.abort_flag);
      const int n_in = last_n_in;
      const float lam = float(k) / float(Gs);
      const int M = min(k, max(kTopM, int(ceilf(lam + 4.0f * sqrtf(lam) + 4.0f))));
      hist_cuts(sm.hist, sm.sel, tid, M);
      if (sm.sel.ok) {
        const int total = sm.sel.total, bM = sm.sel.cM_b;
        // 0: every key; 1: the keys in buckets >= bM; 2: more than kCandCap of those, the exact top M
        const int mode =
            total <= M + 32 ? 0 : (sm.sel.cM_above + sm.sel.cM_cnt <= kCandCap ? 1 : 2);
        const int ncand = mode == 0 ? total : (mode == 1 ? sm.sel.cM_above + sm.sel.cM_cnt : M);
        SessSync &ss = ws->sync[sess];
        const uint32_t par = sm.epoch & 1u;
        unsigned long long reserved = 0ull;
        if (tid == 0 && Gs > 1) reserved = atomicAdd(&ss.main[par], static_cast<unsigned long long>(ncand));
        if (mode != 2) {
          // every key at or above the bucket's floor (mode 0: every key); few
          // qualify, so a warp appends only when one of its lanes has one
          const unsigned long long thr =
              (mode == 0 || bM == 0) ? 1ull : static_cast<unsigned long long>(uint32_t(bM + kBuckets) << 18) << 32;
          const ulonglong2 *k2 = reinterpret_cast<const ulonglong2 *>(sm.keys);
          for (int j = tid; 2 * j < n_in; j += kSelThreads) {
            const ulonglong2 kv = k2[j];  // n_in is even
            const bool c0 = kv.x >= thr, c1 = kv.y >= thr;
            if (__any_sync(__activemask(), c0 || c1)) {
              const unsigned act = __activemask();
              const unsigned m0 = __ballot_sync(act, c0), m1 = __ballot_sync(act, c1);
              const int leader = __ffs(act) - 1;
              int base = 0;
              if (lane == leader) base = atomicAdd(&sm.sel.fill, __popc(m0) + __popc(m1));
              base = __shfl_sync(act, base, leader);
              const unsigned lt = (1u << lane) - 1u;
              const int p0 = base + __popc(m0 & lt), p1 = base + __popc(m0) + __popc(m1 & lt);
              if (c0 && p0 < kCandCap) sm.cand[p0] = kv.x;
              if (c1 && p1 < kCandCap) sm.cand[p1] = kv.y;
            }
          }
          // the bucket's floor (bucket 0 also holds everything below it: nothing is left out)
          if (tid == 0)
            sm.th = (mode == 0 || bM == 0) ? 0ull
                                           : static_cast<unsigned long long>(uint32_t(bM + kBuckets) << 18) << 32;
        } else {
          unsigned long long *scratch = reinterpret_cast<unsigned long long *>(&sm.stage[0][0]);
          for (int i = tid; i < n_in; i += kSelThreads) scratch[i] = sm.keys[i];
          bar512();
          select_top(scratch, n_in, M, sm.cand, sm.hist, sm.sortbuf, sm.sel, tid);
          if (warp == 0) {
            unsigned long long t = ~0ull;
            for (int i = lane; i < M; i += 32) t = min(t, sm.cand[i]);
            for (int o = 16; o > 0; o >>= 1) t = min(t, __shfl_xor_sync(0xffffffffu, t, o));
            if (lane == 0) sm.th = t;
          }
        }
        if (tid == 0) sm.sel.base = uint32_t(reserved);
        bar512();

        // ---- exchange: publish, meet, load the session's candidates ------------------
        const unsigned long long th = sm.th;
        unsigned long long *pool_g = ws->pool + size_t(cta0) * kPubCap;
        if (Gs > 1) {
          const uint32_t base = sm.sel.base;
          for (int i = tid; i < ncand; i += kSelThreads) pool_g[base + i] = sm.cand[i];
          if (tid == 0) atomicMax(&ss.thm[par], th);
        }
        reinterpret_cast<uint4 *>(sm.hist)[tid] = make_uint4(0u, 0u, 0u, 0u);  // the counting sort's 2048 buckets
        if (tid == 0) {
          sm.sel.ncol = 0;
          sm.sel.nhi = 0;
          sm.sel.nge = 0;
          sm.sel.wcnt = 0;
          sm.sel.pub_cnt = 0;
        }
        bar512();
        int n_all = ncand;
        unsigned long long thmax = th;
        if (Gs > 1) {
          if (tid == 0) {
            if (int(blockIdx.x) == cta0) {  // the next exchange's words: nothing in this launch uses them
              ss.main[par ^ 1u] = 0ull;
              ss.fb[par ^ 1u] = 0ull;
              ss.thm[par ^ 1u] = 0ull;
            }
            red_release_add(&ss.main[par], 1ull << 32);
            unsigned long long seen = 0ull;
            const unsigned extra = __ldcg(&hdr->wait_extra);
            const bool ok = wait_arrivals(&ss.main[par], unsigned(Gs) + extra, hdr, &seen);
            if (ok && int(blockIdx.x) == cta0) ss.epoch = sm.epoch + 1u;
            sm.sel.n_all = int(uint32_t(seen));
            sm.sel.ok = ok ? 1 : 0;
          }
          bar512();
          n_all = sm.sel.n_all;
          thmax = ld_cg(&ss.thm[par]);
        }
        const bool overflow = n_all > kPoolCap;
        if (sm.sel.ok) {
          // The pool keys at or above the largest bound, compacted into pool_s
          // (the stage ring is free now): no key below it can be above a
          // winner, and when none of the CTAs is flagged the winners are among
          // them.  Their count decides whether any CTA is flagged.
          unsigned long long *pool_s = reinterpret_cast<unsigned long long *>(&sm.stage[0][0]);
          static_assert(kPoolCap * 8 <= kStages * kStageBytes, "the pool fits in the stage ring");
          {
            unsigned long long v[kPoolPer];
  #pragma unroll
            for (int q = 0; q < kPoolPer; ++q) {
              const int i = tid + q * kSelThreads;
              v[q] = (!overflow && i < n_all) ? (Gs > 1 ? ld_cg(pool_g + i) : sm.cand[i]) : 0ull;
            }
            unsigned keep = 0u, mn = ~0u, mx = 0u;
            int cnt = 0;
  #pragma unroll
            for (int q = 0; q < kPoolPer; ++q) {
              const bool kq = v[q] != 0ull && v[q] >= thmax;
              keep |= kq ? (1u << q) : 0u;
              cnt += __popc(__ballot_sync(0xffffffffu, kq));
              if (kq) {
                const uint32_t h = uint32_t(v[q] >> 32);
                mn = min(mn, h);
                mx = max(mx, h);
              }
            }
            int base = 0;
            if (lane == 0 && cnt > 0) base = atomicAdd(&sm.sel.nge, cnt);
            base = __shfl_sync(0xffffffffu, base, 0);
            const unsigned lt = (1u << lane) - 1u;
  #pragma unroll
            for (int q = 0; q < kPoolPer; ++q) {
              const bool kq = (keep >> q) & 1u;
              const unsigned mk = __ballot_sync(0xffffffffu, kq);
              if (kq) pool_s[base + __popc(mk & lt)] = v[q];
              base += __popc(mk);
            }
            mn = __reduce_min_sync(0xffffffffu, mn);
            mx = __reduce_max_sync(0xffffffffu, mx);
            if (lane == 0) {
              sm.sel.red_lo[warp] = mn;
              sm.sel.red_hi[warp] = mx;
            }
          }
          // this CTA's candidates at or above the largest bound, into sortbuf
          for (int e0 = 0; e0 < ncand; e0 += kSelThreads) {
            const int e = e0 + tid;
            const unsigned long long x = e < ncand ? sm.cand[e] : 0ull;
            const bool h = x != 0ull && x >= thmax;
            const int p = warp_append(&sm.sel.nhi, h);
            if (h) sm.sortbuf[p] = x;
          }
          bar512();
          const int n_ge = sm.sel.nge;
          // No CTA left out a key above the k-th candidate: the pool holds the
          // session's top-k.  (One CTA: its candidates always do.)
          const bool fast = !overflow && (Gs == 1 || (n_all < k ? thmax == 0ull : n_ge >= k));
          if (fast) {
            // Every winner is one of some CTA's candidates at or above the
            // largest bound, and a candidate wins iff fewer than k pool keys
            // are above it; its rank is that count.
            const int nhi = sm.sel.nhi;
            const int nwin = min(n_all, k);
            if (nhi <= kDirect) {
              // per-warp partial counts, in the histogram's words (unused on this path)
              int *rank_part = reinterpret_cast<int *>(sm.hist);
              static_assert((kSelThreads / 32) * kDirect <= kHistWords, "rank partials fit the histogram words");
              for (int e0 = 0; e0 < nhi; e0 += kRankStep) {
                unsigned long long x[kRankStep];
                unsigned r[kRankStep];
  #pragma unroll
                for (int j = 0; j < kRankStep; ++j) {
                  x[j] = e0 + j < nhi ? sm.sortbuf[e0 + j] : ~0ull;
                  r[j] = 0u;
                }
  #pragma unroll
                for (int q = 0; q < kPoolPer; ++q) {
                  if (q * kSelThreads >= n_ge) break;
                  const int i = q * kSelThreads + tid;
                  const unsigned long long pv = i < n_ge ? pool_s[i] : 0ull;
  #pragma unroll
                  for (int j = 0; j < kRankStep; ++j) r[j] += pv > x[j] ? 1u : 0u;
                }
  #pragma unroll
                for (int j = 0; j < kRankStep; ++j) r[j] = __reduce_add_sync(0xffffffffu, r[j]);
                unsigned mine = 0u;
  #pragma unroll
                for (int j = 0; j < kRankStep; ++j) mine = lane == j ? r[j] : mine;
                if (lane < kRankStep && e0 + lane < nhi) rank_part[warp * kDirect + e0 + lane] = int(mine);
              }
              bar512();
              for (int e = tid; e < nhi; e += kSelThreads) {
                int r = 0;
  #pragma unroll
                for (int w = 0; w < kSelThreads / 32; ++w) r += rank_part[w * kDirect + e];
                if (r < k) {
                  const unsigned long long x = sm.sortbuf[e];
                  out_idx[r] = key_index(x);
                  if (out_score) out_score[r] = key_score(x);
                }
              }
            } else {
              // more candidates: a counting sort of the kept pool keys ranks them all at once
              uint32_t mn = ~0u, mx = 0u;
              for (int w = 0; w < kSelThreads / 32; ++w) {
                mn = min(mn, sm.sel.red_lo[w]);
                mx = max(mx, sm.sel.red_hi[w]);
              }
              const unsigned long long lo = static_cast<unsigned long long>(mn) << 32;
              const unsigned long long hi = (static_cast<unsigned long long>(mx) << 32) | 0xffffffffull;
              static_assert(2 * kPoolCap * 8 <= kStages * kStageBytes, "the pool and its sorted copy fit the stage ring");
              bucket_rank(pool_s, n_ge, sm.sortbuf, nhi, lo, hi, k, sm.hist, pool_s + kPoolCap, sm.sel, tid, out_idx,
                          out_score);
            }
            if (int(blockIdx.x) == cta0) {
              for (int e = nwin + tid; e < k; e += kSelThreads) {
                out_idx[e] = -1;
                if (out_score) out_score[e] = __uint_as_float(0x7fc00000u);
              }
            }
          } else {
            // ---- exact fallback -----------------------------------------------------
            // A CTA whose bound is above the k-th candidate may hold winners it
            // did not publish: it publishes its local top-k below its bound, and
            // the session's first CTA merges them with the pool.
            bool flagged;
            if (overflow || n_all < k) {
              flagged = th != 0ull;
            } else {
              unsigned c = 0u;
  #pragma unroll
              for (int q = 0; q < kPoolPer; ++q) {  // the whole pool again (pool_s keeps only the top part)
                const int i = tid + q * kSelThreads;
                const unsigned long long pv = i < n_all ? (Gs > 1 ? ld_cg(pool_g + i) : sm.cand[i]) : 0ull;
                c += (pv != 0ull && pv >= th) ? 1u : 0u;
              }
              c = __reduce_add_sync(0xffffffffu, c);
              bar512();
              if (lane == 0) sm.sel.red_cnt[warp] = int(c);
              bar512();
              int s = 0;
              for (int w = 0; w < kSelThreads / 32; ++w) s += sm.sel.red_cnt[w];
              flagged = s < k;
            }
            int npub = 0;
            if (flagged) {
              const int m = select_top(sm.keys, n_in, k, sm.out, sm.hist, sm.sortbuf, sm.sel, tid);
              for (int i0 = 0; i0 < m; i0 += kSelThreads) {
                const int i = i0 + tid;
                const unsigned long long x = i < m ? sm.out[i] : 0ull;
                const bool pub = x != 0ull && x < th;
                const int p = warp_append(&sm.sel.pub_cnt, pub);
                if (pub && p < kPubCap) ws->lists[blockIdx.x][p] = x;
              }
              bar512();
              npub = min(sm.sel.pub_cnt, kPubCap);
            }
            if (tid == 0) ws->cnt[blockIdx.x] = npub;
            bar512();
            if (tid == 0) red_release_add(&ss.fb[par], 1ull << 32);
            if (int(blockIdx.x) == cta0) {
              if (tid == 0) {
                unsigned long long seen = 0ull;
                sm.sel.ok = wait_arrivals(&ss.fb[par], unsigned(Gs), hdr, &seen) ? 1 : 0;
                atomicAdd(&hdr->fallback, 1u);
              }
              bar512();
              if (sm.sel.ok) {
                // the pool and every flagged CTA's list, reduced to the exact top-k
                int fill = 0;
                for (int src_i = -1; src_i < Gs; ++src_i) {
                  const unsigned long long *src = src_i < 0 ? pool_g : ws->lists[cta0 + src_i];
                  const int len = src_i < 0 ? (Gs > 1 ? n_all : 0) : min(__ldcg(&ws->cnt[cta0 + src_i]), kPubCap);
                  for (int off = 0; off < len; off += kPubCap) {
                    const int cl = min(kPubCap, len - off);
                    if (fill + cl > kKeysCap) {
                      const int m = select_top(sm.keys, fill, k, sm.out, sm.hist, sm.sortbuf, sm.sel, tid);
                      for (int i = tid; i < m; i += kSelThreads) sm.keys[i] = sm.out[i];
                      bar512();
                      fill = m;
                    }
                    for (int i = tid; i < cl; i += kSelThreads) sm.keys[fill + i] = ld_cg(src + off + i);
                    fill += cl;
                    bar512();
                  }
                }
                const int m = select_top(sm.keys, fill, k, sm.out, sm.hist, sm.sortbuf, sm.sel, tid);
                const unsigned long long srt = block_sort512_desc(tid < m ? sm.out[tid] : 0ull, sm.sortbuf, tid);
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
            }
          }
        }
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

}  // namespace

size_t score_fused_ws_bytes() { return sizeof(FusedWs); }

int score_fused_max_ctas() { return kMaxCtas; }

cudaError_t launch_score_batch(const ScoreBatch &sb, int64_t tiles_hint, void *ws, cudaStream_t stream) {
  static std::atomic<uint64_t> smem_set{0};
  static_assert(sizeof(Smem) + 1024 <= size_t(kMaxDynSmem), "shared memory budget");
  const int smem_bytes = int(sizeof(Smem)) + 1024;
  cudaError_t e = set_max_smem_once(score_fused_kernel, smem_bytes, smem_set);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int cap = sms < kMaxCtas ? sms : kMaxCtas;
  // one session: no more CTAs than tiles; a batch: every SM (the kernel splits them)
  const int grid = (tiles_hint > 0 && tiles_hint < cap) ? int(tiles_hint) : cap;
  if (sb.rows_arr != nullptr && grid < sb.n_sess) return cudaErrorInvalidConfiguration;
  // cooperative: the CTAs of a session meet at a barrier, so all must be
  // resident; programmatic stream serialisation: they may be dispatched while
  // the previous kernel finishes (each waits for it before touching memory)
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = size_t(smem_bytes);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, score_fused_kernel, sb, static_cast<FusedWs *>(ws));
}

cudaError_t launch_score_fused(const uint8_t *idx_rows, int64_t n_rows, const uint16_t *q, const float *w,
                               int32_t k, int32_t *out_idx, float *out_score, void *ws, cudaStream_t stream) {
  ScoreBatch sb{};
  sb.rows = idx_rows;
  sb.n_rows = n_rows;
  sb.n_sess = 1;
  sb.q = q;
  sb.w = w;
  sb.k = k;
  sb.out_idx = out_idx;
  sb.out_score = out_score;
  return launch_score_batch(sb, (n_rows + kTileRows - 1) / kTileRows, ws, stream);
}

}  // namespace ds4x
