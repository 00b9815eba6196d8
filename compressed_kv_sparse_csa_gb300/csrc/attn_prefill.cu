// Prefill sparse attention on the tensor cores (DS4X README, "Packed prefill
// implementation": each query token of a prefill chunk attends over its own
// top-k packed KV rows; "Packed cache ABI" for the 583-byte row).
//
// Per query token (64 heads, up to 512 selected rows; the rows are both keys
// and values):
//
//   l_hj = scale * (q_h . v_j),  o_h = sum_j softmax_j(l_h)_j v_j,
//   lse_h = log sum_j e^(l_hj)
//
// The same kernel runs the dense (HCA) attention over every row of an array
// (DS4X README, "Optimization details", the HCA bullet): there an item is a
// run of consecutive rows rather than a query token, every item reads the one
// query, and its normalised output goes out in fp32 with its LSE for the
// split-KV combine over the items.
//
// One persistent CTA per SM takes query tokens blockIdx.x, + gridDim.x, ...
// and runs each query's rows in tiles of 128 through two tcgen05.mma
// (kind::f16, fp16 operands, fp32 accumulators in tensor memory):
//
//   S^T[128 rows][64 heads] = V'[128 rows][512] . Q'[64 heads][512]^T
//   O^T[512 dims][64 heads] += V'^T[512][128 rows] . P^T[128 rows][64 heads]
//
// V' is the tile's rows widened to fp16 once, in shared memory, as eight
// 128-byte-swizzled panels of 64 dims (row r of a panel: 128 bytes, its
// 16-byte chunk c at position c ^ (r % 8)).  The first MMA reads the panels
// K-major (rows = M, a K step 32 bytes further into a panel), the second
// reads the same bytes MN-major (dims = M: two panels per 128-dim M tile),
// so each row is widened once and read twice.  Q' and P^T use the same
// swizzle.
//
// Exact operands.  Before a query's first tile its S_b (b < 7) = the largest
// scale byte of non-RoPE block b over the query's selected rows is found.
// Row j's block-b value code * 2^(s_jb - 127) is then stored as the fp16
// code * 2^(s_jb - S_b), exact while s_jb >= S_b - 15 (smaller rows round at
// 2^-24 of the block's largest scale); RoPE values are fp16 already.  The
// query's dim d of block b is q_hd * 2^(S_b - 127 + c_h) in fp16, c_h putting
// head h's largest such value in [2^14, 2^15) (every bf16 value down to
// 2^-17 of that is exact).  So S^T is 2^c_h times the exact dot products up
// to fp32 accumulation, and the output's block b is scaled back by
// 2^(S_b - 127) at the end.
//
// Softmax: online over the tiles in the log2 domain with a lazy maximum: a
// head's reference maximum moves (and its O^T column and running sum are
// rescaled) only when a tile's maximum exceeds it by more than 8, so
// p = 2^(l - m) stays below 2^8.  p goes to the second MMA as fp16 hi + lo
// (22 significant bits); the running sums are fp32.
//
// Roles: all 16 warps widen (warp w: rows 8 w .. 8 w + 7 of each tile, one
// row per step, lane L converting the row's 4-byte words L + 32 i:
// coalesced loads, conflict-free swizzled stores), then read S^T (warp w:
// lanes 32 (w % 4) .., heads 16 (w / 4) ..), run the softmax and write P^T;
// lane 0 of warps 0 and 1 issue each tile's MMAs once a barrier shows every
// warp's operands written, each half of them (S^T as two K halves into two
// accumulators that the softmax adds; O^T two of its four M tiles each), and
// each commits to the tile's barriers (two arrivals a phase): one thread
// alone issues at about half the tensor core's rate for these shapes.  A
// tile's steps run in sequence: widen -> S^T ->
// softmax -> O^T; the next tile's row words are requested as soon as this
// tile's second MMA is issued, so they arrive while it runs.
//
// Named barriers: 1 = vote (bar.red.or of a failed wait, so that all threads
// leave together), 2 = the tile maxima.
//
// Every wait is bounded (0.5 s); a time-out sets DS4X_ETIMEOUT in the
// workspace status and every thread leaves at its next vote.
#include <cuda_fp16.h>

#include "ds4x_internal.cuh"
#include "tc_ptx.cuh"

namespace ds4x {
namespace {

using namespace ptx;

constexpr int kHeads = 64;
constexpr int kDim = DS4X_KV_DIM;                          // 512
constexpr int kNopeBlocks = DS4X_KV_NOPE / DS4X_KV_BLOCK;  // 7
constexpr int kTile = 128;                                 // rows per tile
constexpr int kThreads = 512;
constexpr int kTmemCols = 512;
constexpr uint32_t kOCol = 0;    // O^T: dims 128 i .. as columns 64 i .. 64 i + 63
constexpr uint32_t kSCol = 256;  // S^T in two K halves: columns 256 .. 319 (dims 0-255), 320 .. 383
constexpr int kIssuers = 2;      // lane 0 of warps 0 and 1 issue the MMAs
constexpr unsigned long long kTimeoutNs = 500ull * 1000 * 1000;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazy = 8.0f;    // a head's reference maximum moves by more than this only
constexpr int kCodeWords = DS4X_KV_NOPE / 4;                      // 112 words of E4M3 codes
constexpr int kRowWords = (DS4X_KV_NOPE + 2 * DS4X_KV_ROPE) / 4;  // 144 words of codes + RoPE

// Byte offsets in the swizzled operands: V' (row r, 8-dim chunk C), Q' (head
// h, chunk C), P^T (row r, 8-head chunk hc).  A panel holds 64 dims (heads)
// of every row (head): 128 bytes a row, chunk c at position c ^ (row % 8).
__device__ __forceinline__ uint32_t v_off(int r, int C) {
  return uint32_t(C >> 3) * 16384u + uint32_t(r) * 128u + (uint32_t((C & 7) ^ (r & 7)) << 4);
}
__device__ __forceinline__ uint32_t q_off(int h, int C) {
  return uint32_t(C >> 3) * 8192u + uint32_t(h) * 128u + (uint32_t((C & 7) ^ (h & 7)) << 4);
}
__device__ __forceinline__ uint32_t p_off(int r, int hc) { return uint32_t(r) * 128u + (uint32_t(hc ^ (r & 7)) << 4); }

// Shared-memory descriptor, 128-byte swizzle.  K-major: sbo = distance of
// 8-row groups (a K step moves the start 32 bytes inside the panel).
// MN-major: lbo = distance of 64-wide panels along M (N), sbo = distance of
// 8-row groups along K.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return uint64_t((saddr & 0x3FFFFu) >> 4) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
         (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

struct __align__(1024) ASmem {
  uint8_t qs[kHeads * kDim * 2];     // Q' (B of the first MMA, K-major): 8 panels of 8 KB
  uint8_t kv[kTile * kDim * 2];      // V' (A of both MMAs): 8 panels of 16 KB
  uint8_t p_hi[kTile * kHeads * 2];  // P^T hi / lo (B of the second MMA, MN-major): one panel each
  uint8_t p_lo[kTile * kHeads * 2];
  float red[4][kHeads];              // per-quadrant maxima (each tile), then sums (each query)
  float qscale[kHeads];              // scale * log2(e) * 2^-c_h
  float hinv[kHeads];                // a query's 1 / (sum of p) per head, for its output
  float tmax[kHeads];                // a tile's maximum per head (log2 units)
  int sb[2][8];                      // S_b (UE8M0 bytes; [7] = 127 for the RoPE part), by query parity
  uint8_t rvalid[kTile];             // the tile's row j is a selected, in-range row
  unsigned long long s_full, pv_done;
  uint32_t tmem_base;
  int abort_flag;
};

// the dynamic shared memory, rounded up to a 1024-byte boundary inside it, fits
// the 227 KB a CTA may have
static_assert(sizeof(ASmem) + 1024 - 16 <= 232448, "shared-memory budget");

// Item qi (a query token, or a dense tile) attends over k rows: idx[qi][0..k),
// or with idx null the consecutive rows qi k .. qi k + k - 1 (those below
// n_rows).  Its query is q + qi q_stride (q_stride 0: one query shared by
// every item); its normalised output goes to out as bf16 or, with out_f32 set,
// to out_f32 in fp32 (the split-KV partials of the dense attention).
struct PrefillAttnArgs {
  const uint8_t *kv;
  int64_t n_rows;
  const int32_t *idx;  // [T][k], or null (dense items)
  int32_t T, k;
  float scale;
  const uint16_t *q;   // bf16 [64][512] per item, q_stride elements apart
  int64_t q_stride;
  uint16_t *out;       // bf16 [T][64][512] (unused when out_f32 is set)
  float *out_f32;      // fp32 [T][64][512] or null
  float *lse;          // [T][64] or null
};

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ bool wait_bar(ASmem &sm, unsigned long long *bar, uint32_t parity, WsHeader *hdr) {
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

// Used only while shutting down after a time-out: no MMA may still write
// this CTA's memory when it exits.
__device__ void drain_bar(unsigned long long *bar, uint32_t parity) {
  const uint32_t b = smem_u32(bar);
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(b, parity) && globaltimer() - t0 < kTimeoutNs / 5) {
  }
}

// 2^e as fp16 bits for e <= 0 (0 below the smallest subnormal 2^-24).
__device__ __forceinline__ uint32_t pow2_half_bits(int e) {
  if (e >= -14) return uint32_t(e + 15) << 10;
  if (e >= -24) return 1u << (e + 24);
  return 0u;
}

__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }  // e in [-126, 127]

__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ float ex2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// A float as a signed integer with the same order (for redux max); -inf is
// the least value a logit takes here.
__device__ __forceinline__ int ordered_int(float f) {
  const int i = __float_as_int(f);
  return i >= 0 ? i : (i ^ 0x7fffffff);
}
__device__ __forceinline__ float ordered_float(int i) { return __int_as_float(i >= 0 ? i : (i ^ 0x7fffffff)); }

__device__ __forceinline__ int redux_max(int v) {
  int r;
  asm volatile("redux.sync.max.s32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
  return r;
}
__device__ __forceinline__ uint32_t redux_max_u(uint32_t v) {
  uint32_t r;
  asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
  return r;
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
  return r;
}

__device__ __forceinline__ bool row_ok(const PrefillAttnArgs &a, int32_t row) {
  return row >= 0 && int64_t(row) < a.n_rows;
}

// The 8 rows of a warp's share of tile t (row k's index in lane 8 t + k of
// `rows`): lane L loads each row's 4-byte aligned words L + 32 i, i < 5, up
// to word 144 (which ends at row byte 580 at most, so every word read lies
// inside its row).  A skipped row, or a tile past the last, reads nothing and
// gives zeros.
__device__ __forceinline__ void load_tile_words(const PrefillAttnArgs &a, int32_t rows, int t, int n_tiles, int lane,
                                               uint32_t (&w)[8][5]) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int32_t row = __shfl_sync(0xffffffffu, rows, (8 * t + k) & 31);
    if (t < n_tiles && row_ok(a, row)) {  // warp-uniform
      const int64_t o = int64_t(row) * DS4X_KV_ROW_BYTES;
      const uint32_t *wp = reinterpret_cast<const uint32_t *>(a.kv + (o & ~int64_t(3)));
#pragma unroll
      for (int i = 0; i < 5; ++i) w[k][i] = 32 * i + lane <= kRowWords ? __ldg(wp + 32 * i + lane) : 0u;
    } else {
#pragma unroll
      for (int i = 0; i < 5; ++i) w[k][i] = 0u;
    }
  }
}

// Lane L's row of query qi: row 8 warp + L % 8 of tile L / 8 (-1 past k).
__device__ __forceinline__ int32_t query_row(const PrefillAttnArgs &a, int qi, int warp, int lane) {
  const int pos = kTile * (lane >> 3) + 8 * warp + (lane & 7);
  if (pos >= a.k) return -1;
  if (a.idx == nullptr) {  // dense item: the array's rows qi k + pos (n_rows < 2^31)
    const int64_t r = int64_t(qi) * a.k + pos;
    return r < a.n_rows ? int32_t(r) : -1;
  }
  return __ldg(a.idx + int64_t(qi) * a.k + pos);
}

// The row's 7 scale bytes (a skipped row reads row 0's, dropped by pack_scales).
__device__ __forceinline__ void load_scale_bytes(const PrefillAttnArgs &a, int32_t row, uint32_t (&b)[kNopeBlocks]) {
  const uint8_t *sp =
      a.kv + (row_ok(a, row) ? int64_t(row) * DS4X_KV_ROW_BYTES : 0) + DS4X_KV_NOPE + 2 * DS4X_KV_ROPE;
#pragma unroll
  for (int i = 0; i < kNopeBlocks; ++i) b[i] = __ldg(sp + i);
}
// ... as scale bytes 0-3 / 4-6 (zeros for a skipped row).
__device__ __forceinline__ void pack_scales(const PrefillAttnArgs &a, int32_t row, const uint32_t (&b)[kNopeBlocks],
                                            uint32_t &sc0, uint32_t &sc1) {
  const bool v = row_ok(a, row);
  sc0 = v ? b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24) : 0u;
  sc1 = v ? b[4] | (b[5] << 8) | (b[6] << 16) : 0u;
}

// This thread's 64 query values (head qh, block qb) of query qi, copied raw
// (cp.async, 16 bytes a copy) to their Q' places; the thread waits for its
// own copies before it converts them.
__device__ __forceinline__ void copy_query_async(ASmem &sm, const PrefillAttnArgs &a, int qi, int qh, int qb) {
  const uint16_t *src = a.q + int64_t(qi) * a.q_stride + int64_t(qh) * kDim + 64 * qb;
#pragma unroll
  for (int c = 0; c < 8; ++c)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(sm.qs + q_off(qh, 8 * qb + c))),
                 "l"(src + 8 * c)
                 : "memory");
  asm volatile("cp.async.commit_group;" ::: "memory");
}

__global__ void __launch_bounds__(kThreads, 1) attn_prefill_kernel(PrefillAttnArgs a, WsHeader *__restrict__ hdr) {
  extern __shared__ uint8_t smem_raw[];
  ASmem &sm = *reinterpret_cast<ASmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_tiles = (a.k + kTile - 1) / kTile;

  if (tid == 0) {
    mbar_init(smem_u32(&sm.s_full), kIssuers);  // one commit from each issuer
    mbar_init(smem_u32(&sm.pv_done), kIssuers);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (tid < 16) sm.sb[tid >> 3][tid & 7] = (tid & 7) < kNopeBlocks ? 0 : 127;
  if (warp == 0) {
    tmem_alloc(smem_u32(&sm.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  const uint32_t kv_a = smem_u32(sm.kv), q_a = smem_u32(sm.qs);
  const uint32_t ph_a = smem_u32(sm.p_hi), pl_a = smem_u32(sm.p_lo);
  constexpr uint32_t kIdS = idesc_f16(128, kHeads, 0, 0);  // V' K-major, Q' K-major
  constexpr uint32_t kIdO = idesc_f16(128, kHeads, 1, 1);  // V'^T MN-major, P^T MN-major
  // the operands' descriptors at their first K step (later steps add to the address field)
  const uint64_t dS_a = desc_sw128(kv_a, 16, 1024), dS_b = desc_sw128(q_a, 16, 1024);
  const uint64_t dO_a = desc_sw128(kv_a, 16384, 1024);
  const uint64_t dO_bh = desc_sw128(ph_a, 8192, 1024), dO_bl = desc_sw128(pl_a, 8192, 1024);

  const int qd = warp & 3, hg = warp >> 2;  // softmax: tile rows 32 qd + lane, heads 16 hg .. 16 hg + 15
  const int r_sm = 32 * qd + lane;
  const uint32_t lane_base = uint32_t(32 * qd) << 16;
  // the row sums: after the butterfly each lane holds head hl of its warp's group
  const int hl = 8 * ((lane >> 4) & 1) + 4 * ((lane >> 3) & 1) + 2 * ((lane >> 2) & 1) + ((lane >> 1) & 1);
  const int qh = tid >> 3, qb = tid & 7;  // Q': head tid / 8, block tid % 8
  uint32_t g = 0;   // tiles so far (the phase of s_full and pv_done)
  // the MMA issuers: lane 0 of warps 0 and 1 (issuer ih = warp)
  const bool issuer = lane == 0 && warp < kIssuers;
  const int ih = warp;
  int pending = 0;  // an issuer: 1 = s_full of the current tile committed last, 2 = pv_done of the last tile
  bool ok = true, aborted = false;
  int qn = 0;       // queries so far: sb[qn & 1] is this query's
  // this query's inputs: lane L's row (row 8 warp + L % 8 of tile L / 8) and its
  // scale bytes 0-3 / 4-6 (the raw query values are copied to Q''s places)
  int32_t rowm = -1;
  uint32_t sc0 = 0, sc1 = 0;
  // Launched as a programmatic dependent: nothing above touches global memory;
  // wait here for the previous kernel.  Kernels launched as dependents of this
  // one may be scheduled from now on (they too wait for its completion).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (int(blockIdx.x) < a.T) {  // the first query's inputs (later queries' arrive during the previous epilogue)
    copy_query_async(sm, a, blockIdx.x, qh, qb);
    rowm = query_row(a, blockIdx.x, warp, lane);
    // the first tile's rows toward L2 while the scale bytes are awaited (lanes 0-7
    // hold the tile's rows 8 warp + 0..7; lane L < 6 takes the row's L-th 128-byte
    // line, every address inside the row)
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int32_t row = __shfl_sync(0xffffffffu, rowm, k);
      if (lane < 6 && row_ok(a, row)) {
        const int64_t o = int64_t(row) * DS4X_KV_ROW_BYTES;
        const int64_t line = (o & ~int64_t(127)) + 128 * lane;
        const int64_t at = line > o ? line : o;
        if (at < o + DS4X_KV_ROW_BYTES) asm volatile("prefetch.global.L2 [%0];" ::"l"(a.kv + at));
      }
    }
    uint32_t b[kNopeBlocks];
    load_scale_bytes(a, rowm, b);
    pack_scales(a, rowm, b, sc0, sc1);
  }
  for (int qi = blockIdx.x; qi < a.T && !aborted; qi += gridDim.x, ++qn) {
    int *sbq = sm.sb[qn & 1];
    uint32_t raw[8][5];  // the words of the warp's 8 rows of the next tile to widen (tile 0's
    load_tile_words(a, rowm, 0, n_tiles, lane, raw);  // arrive while S_b is found and Q' converted)
    if (named_bar_or(1, kThreads, !ok)) break;  // the previous query's readers of Q', sb[(qn + 1) & 1] are done
    if (tid < 8) sm.sb[(qn + 1) & 1][tid] = tid < kNopeBlocks ? 0 : 127;  // for the next query
    if (!row_ok(a, rowm) && rowm != -1) atomicExch(&hdr->status, int32_t(DS4X_EDEVICE));
#pragma unroll
    for (int b = 0; b < kNopeBlocks; ++b) {  // S_b
      const uint32_t m = redux_max_u(((b < 4 ? sc0 >> (8 * b) : sc1 >> (8 * (b - 4)))) & 0xffu);
      if (lane == 0 && m > 0) atomicMax(&sbq[b], int(m));
    }
    if (named_bar_or(1, kThreads, !ok)) break;
    // the lane's row's fp16 factors 2^(s_b - S_b): blocks 2 i (low half) and 2 i + 1 of fac[i]
    uint32_t fac[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int b0 = 2 * i, b1 = 2 * i + 1;
      const uint32_t s_0 = (b0 < 4 ? sc0 >> (8 * b0) : sc1 >> (8 * (b0 - 4))) & 0xffu;
      const uint32_t s_1 = b1 < kNopeBlocks ? (b1 < 4 ? sc0 >> (8 * b1) : sc1 >> (8 * (b1 - 4))) & 0xffu : 0u;
      fac[i] = pow2_half_bits(int(s_0) - sbq[b0]) |
               (b1 < kNopeBlocks ? pow2_half_bits(int(s_1) - sbq[b1]) << 16 : 0u);
    }
    // ---- Q' in place: this thread's 64 values times 2^(S_b - 127 + c_h), to fp16 ----------
    {
      asm volatile("cp.async.wait_all;" ::: "memory");  // this thread's raw query values
      uint4 qv[8];
      int emax = -1;  // the largest bf16 exponent field among the normal values
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        qv[c] = *reinterpret_cast<const uint4 *>(sm.qs + q_off(qh, 8 * qb + c));
        const uint32_t w4[4] = {qv[c].x, qv[c].y, qv[c].z, qv[c].w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int e0 = int((w4[u] >> 7) & 0xff), e1 = int((w4[u] >> 23) & 0xff);
          if (e0 != 0) emax = max(emax, e0);
          if (e1 != 0) emax = max(emax, e1);
        }
      }
      const int sh_b = sbq[qb] - 127;
      int eh = emax < 0 ? -100000 : emax - 127 + sh_b;
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) eh = max(eh, __shfl_xor_sync(0xffffffffu, eh, o));
      const int c_h = eh == -100000 ? 0 : 14 - eh;
      // x * 2^(sh_b + c_h) as two exact power-of-two products (each factor a normal float)
      const int s1 = max(-126, min(127, sh_b + c_h)), s2 = max(-126, min(127, sh_b + c_h - s1));
      const float f1 = pow2f(s1), f2 = pow2f(s2);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint4 *qp = reinterpret_cast<uint4 *>(sm.qs + q_off(qh, 8 * qb + c));
        const uint32_t w4[4] = {qv[c].x, qv[c].y, qv[c].z, qv[c].w};
        uint32_t o4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float x0 = __uint_as_float(w4[u] << 16) * f1 * f2;
          const float x1 = __uint_as_float(w4[u] & 0xffff0000u) * f1 * f2;
          const __half2 hv = __floats2half2_rn(x0, x1);
          o4[u] = *reinterpret_cast<const uint32_t *>(&hv);
        }
        *qp = make_uint4(o4[0], o4[1], o4[2], o4[3]);
      }
      if (qb == 0) {
        const int e1 = max(-126, min(127, -c_h)), e2 = max(-126, min(127, -c_h - e1));
        sm.qscale[qh] = a.scale * kLog2e * pow2f(e1) * pow2f(e2);
      }
    }
    fence_proxy_async_smem();

    int32_t rowm_next = -1;  // the next query's rows (requested in the last tile)
    float m_ref[16];  // head 16 hg + i's reference maximum (log2 units), the same in every lane
    float m_lane = -INFINITY, wsum = 0.0f;  // head 16 hg + hl: the same maximum, the warp's rows' sum
#pragma unroll
    for (int i = 0; i < 16; ++i) m_ref[i] = -INFINITY;
    for (int t = 0; t < n_tiles; ++t, ++g) {
      // ---- widen tile t into V' (after the previous tile's second MMA) ----------
      if (g > 0 && !wait_bar(sm, &sm.pv_done, (g - 1) & 1, hdr)) ok = false;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int r = 8 * warp + k, src = 8 * t + k;
        const int32_t row = __shfl_sync(0xffffffffu, rowm, src);
        if (lane == 0) sm.rvalid[r] = row_ok(a, row) ? 1 : 0;
        // a skipped row's words are zeros, so it widens to zeros with any shift and factor
        const uint32_t sh = 8u * (uint32_t(row) * uint32_t(DS4X_KV_ROW_BYTES) & 3u);
        uint32_t nx[5];  // word m + 1: from lane L + 1 (lane 31: lane 0's next stretch)
#pragma unroll
        for (int i = 0; i < 5; ++i) nx[i] = __shfl_sync(0xffffffffu, raw[k][i], (lane + 1) & 31);
#pragma unroll
        for (int i = 0; i < 5; ++i) {
          const int m = 32 * i + lane;  // the row's 4-byte word m (bytes 4 m .. 4 m + 3)
          const uint32_t wv = __funnelshift_r(raw[k][i], lane == 31 ? (i < 4 ? nx[i + 1] : 0u) : nx[i], sh);
          // (every lane takes part in the shuffle, before the branch)
          const uint32_t fw = i < 4 ? __shfl_sync(0xffffffffu, fac[i < 4 ? i : 0], src) : 0u;
          if (i < 3 || (i == 3 && lane < 16)) {  // four E4M3 codes of block m / 16 = 2 i + lane / 16
            const uint32_t f = ((lane & 16) ? fw >> 16 : fw & 0xffffu) * 0x10001u;
            uint32_t h0, h1;
            asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
                "cvt.rn.f16x2.e4m3x2 %0, lo;\n\tcvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
                : "=r"(h0), "=r"(h1)
                : "r"(wv));
            *reinterpret_cast<uint2 *>(sm.kv + v_off(r, m >> 1) + (m & 1) * 8) =
                make_uint2(hmul2_bits(h0, f), hmul2_bits(h1, f));
          } else if (i == 3 || lane < 16) {  // two FP16 RoPE values
            const int rm = m - kCodeWords;
            *reinterpret_cast<uint32_t *>(sm.kv + v_off(r, DS4X_KV_NOPE / 8 + (rm >> 2)) + (rm & 3) * 4) = wv;
          }
        }
      }
      fence_proxy_async_smem();
      if (named_bar_or(1, kThreads, !ok)) {  // every warp's V' (and Q', rvalid) written
        aborted = true;
        break;
      }
      if (issuer) {
        tc_fence_after();
        // issuer ih: K steps 16 ih .. 16 ih + 15 (dims 256 ih ..) into its own accumulator,
        // columns kSCol + 64 ih; K step ks: 32 bytes into panel ks / 4 (the descriptors'
        // address field counts 16 bytes)
#pragma unroll
        for (int kk = 0; kk < kDim / 16 / kIssuers; ++kk) {
          const int ks = (kDim / 16 / kIssuers) * ih + kk;
          mma_f16_ss(tmem + kSCol + 64u * uint32_t(ih), dS_a + uint64_t(1024 * (ks >> 2) + 2 * (ks & 3)),
                     dS_b + uint64_t(512 * (ks >> 2) + 2 * (ks & 3)), kIdS, kk > 0 ? 1u : 0u);
        }
        tc_commit(smem_u32(&sm.s_full));
        pending = 1;
      }

      // ---- softmax of tile t ------------------------------------------------------
      if (!wait_bar(sm, &sm.s_full, g & 1, hdr)) ok = false;
      tc_fence_after();
      float l[16];
      {
        uint32_t sv[16];
        tc_ld_x16(tmem + lane_base + kSCol + 16u * hg, sv);
        tc_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) l[i] = __uint_as_float(sv[i]);
        tc_ld_x16(tmem + lane_base + kSCol + 64u + 16u * hg, sv);
        tc_wait_ld();
        const bool rv0 = sm.rvalid[r_sm] != 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) l[i] = rv0 ? (l[i] + __uint_as_float(sv[i])) * sm.qscale[16 * hg + i] : -INFINITY;
      }
      float *red = &sm.red[0][0];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int mx = redux_max(ordered_int(l[i]));
        if (lane == i) red[qd * kHeads + 16 * hg + i] = ordered_float(mx);
      }
      named_bar_sync(2, kThreads);
      // each head's tile maximum once, over the four quadrants (lanes 0-15 of the first
      // quadrant's warps: head 16 hg + lane), then read by every thread
      if (qd == 0 && lane < 16) {
        const int hh = 16 * hg + lane;
        sm.tmax[hh] = fmaxf(fmaxf(red[hh], red[kHeads + hh]), fmaxf(red[2 * kHeads + hh], red[3 * kHeads + hh]));
      }
      named_bar_sync(2, kThreads);
      bool rescale = false;
      float alpha[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float mt = sm.tmax[16 * hg + i];
        alpha[i] = 1.0f;
        if (mt > m_ref[i] + kLazy) {
          alpha[i] = m_ref[i] == -INFINITY ? 0.0f : ex2(m_ref[i] - mt);
          m_ref[i] = mt;
          rescale = true;
        }
      }
      {  // the same decision for this lane's head of the sum
        const float mt = sm.tmax[16 * hg + hl];
        if (mt > m_lane + kLazy) {
          wsum *= m_lane == -INFINITY ? 0.0f : ex2(m_lane - mt);
          m_lane = mt;
        }
      }
      if (rescale && t > 0) {  // warp-uniform: every lane of a warp holds the same maxima
#pragma unroll 1
        for (int mi = 0; mi < kDim / 128; ++mi) {
          uint32_t ov[16];
          const uint32_t ta = tmem + lane_base + kOCol + 64u * mi + 16u * hg;
          tc_ld_x16(ta, ov);
          tc_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha[i]);
          tc_st_x16(ta, ov);
        }
        tc_wait_st();
      }
      {
        const bool rv = sm.rvalid[r_sm] != 0;
        uint32_t ph[8], pl[8];
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          const float p0 = rv ? ex2(l[i] - m_ref[i]) : 0.0f;
          const float p1 = rv ? ex2(l[i + 1] - m_ref[i + 1]) : 0.0f;
          l[i] = p0;
          l[i + 1] = p1;
          const __half2 hi = __floats2half2_rn(p0, p1);
          const float2 hf = __half22float2(hi);
          const __half2 lo = __floats2half2_rn(p0 - hf.x, p1 - hf.y);
          ph[i / 2] = *reinterpret_cast<const uint32_t *>(&hi);
          pl[i / 2] = *reinterpret_cast<const uint32_t *>(&lo);
        }
        *reinterpret_cast<uint4 *>(sm.p_hi + p_off(r_sm, 2 * hg)) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
        *reinterpret_cast<uint4 *>(sm.p_hi + p_off(r_sm, 2 * hg + 1)) = make_uint4(ph[4], ph[5], ph[6], ph[7]);
        *reinterpret_cast<uint4 *>(sm.p_lo + p_off(r_sm, 2 * hg)) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
        *reinterpret_cast<uint4 *>(sm.p_lo + p_off(r_sm, 2 * hg + 1)) = make_uint4(pl[4], pl[5], pl[6], pl[7]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      if (named_bar_or(1, kThreads, !ok)) {  // every warp's P^T (and O^T rescale) written
        aborted = true;
        break;
      }
      if (issuer) {
        tc_fence_after();
        // M tile mi: panels 2 mi, 2 mi + 1 (32 KB on); K step ks: 16 rows (2 KB) on.  The four
        // M tiles' accumulators are independent: issuer ih takes M tiles 2 ih and 2 ih + 1,
        // their MMAs interleaved
        const uint32_t acc0 = t > 0 ? 1u : 0u;
#pragma unroll
        for (int ks = 0; ks < kTile / 16; ++ks) {
#pragma unroll
          for (int mj = 0; mj < kDim / 128 / kIssuers; ++mj) {
            const int mi = (kDim / 128 / kIssuers) * ih + mj;
            const uint64_t ad = dO_a + uint64_t(2048 * mi + 128 * ks);
            mma_f16_ss(tmem + kOCol + 64u * mi, ad, dO_bh + uint64_t(128 * ks), kIdO, ks > 0 ? 1u : acc0);
            mma_f16_ss(tmem + kOCol + 64u * mi, ad, dO_bl + uint64_t(128 * ks), kIdO, 1u);
          }
        }
        tc_commit(smem_u32(&sm.pv_done));
        pending = 2;
      }
      // the next tile's words arrive while this tile's second MMA runs (requested
      // after the proxy fence above, which would otherwise wait for them)
      load_tile_words(a, rowm, t + 1, n_tiles, lane, raw);
      if (t + 1 == n_tiles) rowm_next = qi + int(gridDim.x) < a.T ? query_row(a, qi + int(gridDim.x), warp, lane) : -1;
      // this tile's p summed over the warp's 32 rows, head by head (a butterfly:
      // after it lane L holds head hl(L)), added to the lane's running sum
      {
        float w8[8], w4[4], w2[2];
        const bool b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1, b2 = (lane >> 2) & 1, b1 = (lane >> 1) & 1;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float send = b4 ? l[k] : l[k + 8], keep = b4 ? l[k + 8] : l[k];
          w8[k] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float send = b3 ? w8[k] : w8[k + 4], keep = b3 ? w8[k + 4] : w8[k];
          w4[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const float send = b2 ? w4[k] : w4[k + 2], keep = b2 ? w4[k + 2] : w4[k];
          w2[k] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
        }
        const float send = b1 ? w2[0] : w2[1], keep = b1 ? w2[1] : w2[0];
        float w1 = keep + __shfl_xor_sync(0xffffffffu, send, 2);
        w1 += __shfl_xor_sync(0xffffffffu, w1, 1);
        wsum += w1;
      }
    }
    if (aborted) break;

    // ---- the query's output: O^T / sum, block scales put back ---------------------------
    if (!wait_bar(sm, &sm.pv_done, (g - 1) & 1, hdr)) ok = false;
    tc_fence_after();
    // the next query's scale bytes and values are requested now and used after the output
    const bool more = qi + int(gridDim.x) < a.T;
    uint32_t scb_next[kNopeBlocks];  // packed after the output (their loads are in flight meanwhile)
    if (more) load_scale_bytes(a, rowm_next, scb_next);
    if (more) copy_query_async(sm, a, qi + int(gridDim.x), qh, qb);  // Q''s buffer is free: the last first MMA is done
    float *red = &sm.red[0][0];
    if ((lane & 1) == 0) red[qd * kHeads + 16 * hg + hl] = wsum;
    if (named_bar_or(1, kThreads, !ok)) break;
    // each head's sum once, by the even lanes of the first quadrant's warps (lane L:
    // head 16 hg + hl; m_lane is that head's reference maximum, the same value as
    // m_ref[hl]): its reciprocal for every thread, and its LSE
    if (qd == 0 && (lane & 1) == 0) {
      const int hh = 16 * hg + hl;
      const float tot = (red[hh] + red[kHeads + hh]) + (red[2 * kHeads + hh] + red[3 * kHeads + hh]);
      sm.hinv[hh] = tot > 0.0f ? __frcp_rn(tot) : 0.0f;  // = 1 / tot, correctly rounded
      if (a.lse != nullptr)
        a.lse[int64_t(qi) * kHeads + hh] = tot > 0.0f ? (m_lane + log2f(tot)) * 0.6931471805599453f : -INFINITY;
    }
    named_bar_sync(2, kThreads);
    float inv[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) inv[i] = sm.hinv[16 * hg + i];
    if (a.out_f32 != nullptr) {
      // fp32 [head][dim] straight from the accumulator: a warp's store is 32
      // consecutive dims of one head
      float *of = a.out_f32 + int64_t(qi) * kHeads * kDim;
#pragma unroll 1
      for (int mi = 0; mi < kDim / 128; ++mi) {
        uint32_t ov[16];
        tc_ld_x16(tmem + lane_base + kOCol + 64u * mi + 16u * hg, ov);
        tc_wait_ld();
        const int d = 128 * mi + 32 * qd + lane;
        const float fb = ldexpf(1.0f, sbq[d >> 6] - 127);
#pragma unroll
        for (int i = 0; i < 16; ++i) of[(16 * hg + i) * kDim + d] = (__uint_as_float(ov[i]) * inv[i]) * fb;
      }
      tc_fence_before();
    } else {
      // o as bf16 [head][dim] in V''s space (free once the last second MMA is done),
      // then out with 16-byte stores
      uint16_t *os = reinterpret_cast<uint16_t *>(sm.kv);
#pragma unroll 1
      for (int mi = 0; mi < kDim / 128; ++mi) {
        uint32_t ov[16];
        tc_ld_x16(tmem + lane_base + kOCol + 64u * mi + 16u * hg, ov);
        tc_wait_ld();
        const int d = 128 * mi + 32 * qd + lane;
        const float fb = ldexpf(1.0f, sbq[d >> 6] - 127);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          os[(16 * hg + i) * kDim + d] = f32_to_bf16_rn((__uint_as_float(ov[i]) * inv[i]) * fb);
      }
      tc_fence_before();
      named_bar_sync(2, kThreads);
      const uint4 *s4 = reinterpret_cast<const uint4 *>(sm.kv);
      uint4 *o4 = reinterpret_cast<uint4 *>(a.out + int64_t(qi) * kHeads * kDim);
#pragma unroll
      for (int c = 0; c < kHeads * kDim * 2 / 16 / kThreads; ++c) o4[tid + c * kThreads] = s4[tid + c * kThreads];
    }
    if (more) pack_scales(a, rowm_next, scb_next, sc0, sc1);
    rowm = rowm_next;
  }
  if (aborted || !ok) {  // the issuers: no MMA may still write this CTA's memory when it exits
    if (issuer && pending == 1) drain_bar(&sm.s_full, (g - 1 + (aborted ? 1 : 0)) & 1);
    if (issuer && pending == 2) drain_bar(&sm.pv_done, (g - 1) & 1);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

size_t attn_prefill_ws_bytes() { return kWsHeaderBytes; }

namespace {

cudaError_t launch_items(const PrefillAttnArgs &a, void *ws, cudaStream_t stream) {
  static std::atomic<uint64_t> smem_set{0};
  // the dynamic shared memory is at least 16-byte aligned: room to round it up to 1024
  const int smem = int(sizeof(ASmem)) + 1024 - 16;
  cudaError_t e = set_max_smem_once(attn_prefill_kernel, smem, smem_set);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // programmatic stream serialisation: the CTAs may be scheduled while the
  // previous kernel finishes; they wait for it before touching global memory
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(unsigned(a.T < sms ? a.T : sms));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = size_t(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_prefill_kernel, a, reinterpret_cast<WsHeader *>(ws));
}

}  // namespace

cudaError_t launch_attn_prefill(const uint8_t *kv_rows, int64_t n_rows, const int32_t *idx, int32_t n_queries,
                                int32_t k, const uint16_t *q, float scale, uint16_t *out, float *lse, void *ws,
                                cudaStream_t stream) {
  const PrefillAttnArgs a{kv_rows, n_rows, idx, n_queries, k, scale, q, int64_t(kHeads) * kDim, out, nullptr, lse};
  return launch_items(a, ws, stream);
}

cudaError_t launch_attn_dense_items(const uint8_t *kv_rows, int64_t n_rows, int32_t rows_per_item, int32_t items,
                                    const uint16_t *q, float scale, float *out_f32, float *lse, void *ws,
                                    cudaStream_t stream) {
  if (rows_per_item < 1 || rows_per_item > DS4X_TOPK_MAX || items < 1 || n_rows > int64_t(INT32_MAX))
    return cudaErrorInvalidValue;
  const PrefillAttnArgs a{kv_rows, n_rows, nullptr, items, rows_per_item, scale, q, 0, nullptr, out_f32, lse};
  return launch_items(a, ws, stream);
}

}  // namespace ds4x
