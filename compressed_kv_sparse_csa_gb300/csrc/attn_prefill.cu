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
// One persistent CTA per SM takes query tokens blockIdx.x, + gridDim.x, ...
// and runs each query's rows in tiles of 128 through two tcgen05.mma
// (kind::f16, fp16 operands, fp32 accumulators in tensor memory):
//
//   S^T[128 rows][64 heads] = V'[128 rows][512] . Q'[64 heads][512]^T
//   O^T[512 dims][64 heads] += V'^T[512][128 rows] . P^T[128 rows][64 heads]
//
// V' is the tile's rows widened to fp16 once, in shared memory, in the
// canonical no-swizzle layout (core matrices of 8 rows x 8 dims); the first
// MMA reads it K-major (rows = M), the second reads the same bytes MN-major
// (dims = M), so each row is widened once and read twice.
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
// Roles: all 16 warps widen each tile's rows (two passes of 64 rows, eight
// threads per row: seven 8-dim non-RoPE chunks and one RoPE chunk each,
// straight from global memory with 4-byte loads), then read S^T (warp w:
// lanes 32 (w % 4) .., heads 16 (w / 4) ..), run the softmax and write P^T;
// thread 0 issues each tile's MMAs once a barrier shows every warp's
// operands written.  One tile's steps run in sequence: widen -> S^T ->
// softmax -> O^T, the next tile's widening waiting for the previous tile's
// second MMA to release V' and P^T.
//
// Named barriers: 1 = vote (bar.red.or of a failed wait, so that all threads
// leave together), 2 = the tile maxima, 3 = the S_b reset.
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
constexpr int kDim = DS4X_KV_DIM;                     // 512
constexpr int kNopeBlocks = DS4X_KV_NOPE / DS4X_KV_BLOCK;  // 7
constexpr int kTile = 128;                            // rows per tile
constexpr int kWorkers = 512;                         // warps 0-15
constexpr int kThreads = kWorkers;
constexpr int kTmemCols = 512;
constexpr uint32_t kOCol = 0;                         // O^T: dims 128 i .. as columns 64 i .. 64 i + 63
constexpr uint32_t kSCol = 256;                       // S^T: columns 256 .. 319
constexpr unsigned long long kTimeoutNs = 500ull * 1000 * 1000;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazy = 8.0f;                         // a head's reference maximum moves by more than this only

// Shared-memory byte offsets of element (row, dim) of V' / (head, dim) of Q' /
// (row, head) of P^T: core matrices of 8 x 8 fp16 values (16-byte rows).
__device__ __forceinline__ uint32_t kv_off(int r, int chunk) { return uint32_t(r >> 3) * 8192u + uint32_t(chunk) * 128u + uint32_t(r & 7) * 16u; }
__device__ __forceinline__ uint32_t q_off(int h, int chunk) { return uint32_t(h >> 3) * 8192u + uint32_t(chunk) * 128u + uint32_t(h & 7) * 16u; }
__device__ __forceinline__ uint32_t p_off(int r, int hchunk) { return uint32_t(r >> 3) * 1024u + uint32_t(hchunk) * 128u + uint32_t(r & 7) * 16u; }

struct __align__(128) ASmem {
  uint8_t qs[kHeads * kDim * 2];   // Q' (B of the first MMA, K-major)
  uint8_t kv[kTile * kDim * 2];    // V' (A of both MMAs)
  uint8_t p_hi[kTile * kHeads * 2];  // P^T hi / lo (B of the second MMA, MN-major)
  uint8_t p_lo[kTile * kHeads * 2];
  float red[2][4][kHeads];         // per-quadrant maxima / sums, double-buffered by use
  float qscale[kHeads];            // scale * log2(e) * 2^-c_h
  int sb[8];                       // S_b (UE8M0 bytes); sb[7] = 127 (RoPE)
  uint8_t rvalid[kTile];           // the tile's row j is a selected, in-range row
  unsigned long long s_full, pv_done;
  uint32_t tmem_base;
  int abort_flag;
};

struct PrefillAttnArgs {
  const uint8_t *kv;
  int64_t n_rows;
  const int32_t *idx;  // [T][k]
  int32_t T, k;
  float scale;
  const uint16_t *q;   // bf16 [T][64][512]
  uint16_t *out;       // bf16 [T][64][512]
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

// Two E4M3 codes (bits 0-7 and 8-15) -> fp16x2 (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v) {
  uint32_t r;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(r) : "r"(v));
  return r;
}

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

__global__ void __launch_bounds__(kThreads, 1) attn_prefill_kernel(PrefillAttnArgs a, WsHeader *__restrict__ hdr) {
  extern __shared__ uint8_t smem_raw[];
  ASmem &sm = *reinterpret_cast<ASmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_tiles = (a.k + kTile - 1) / kTile;

  if (tid == 0) {
    mbar_init(smem_u32(&sm.s_full), 1);
    mbar_init(smem_u32(&sm.pv_done), 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
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

  const int qd = warp & 3, hg = warp >> 2;  // softmax: tile rows 32 qd + lane, heads 16 hg .. 16 hg + 15
  const int r_sm = 32 * qd + lane;
  const uint32_t lane_base = uint32_t(32 * qd) << 16;
  uint32_t g = 0;   // tiles so far (the phase of s_full and pv_done)
  int rp = 0;       // uses of red so far
  int pending = 0;  // thread 0: 1 = s_full of tile g - 1 committed last, 2 = its pv_done
  bool ok = true, aborted = false;
  for (int qi = blockIdx.x; qi < a.T && !aborted; qi += gridDim.x) {
    const int32_t *idxq = a.idx + int64_t(qi) * a.k;
    // ---- S_b: the largest scale byte of each non-RoPE block over the selected rows
    if (named_bar_or(1, kThreads, !ok)) break;  // the previous query's readers of sb are done
    if (tid < 8) sm.sb[tid] = tid < kNopeBlocks ? 0 : 127;
    named_bar_sync(3, kThreads);
    {
      uint32_t sc[kNopeBlocks];
#pragma unroll
      for (int b = 0; b < kNopeBlocks; ++b) sc[b] = 0;
      if (tid < a.k) {
        const int32_t row = idxq[tid];
        if (row >= 0 && int64_t(row) < a.n_rows) {
          const uint8_t *sp = a.kv + int64_t(row) * DS4X_KV_ROW_BYTES + DS4X_KV_NOPE + 2 * DS4X_KV_ROPE;
#pragma unroll
          for (int b = 0; b < kNopeBlocks; ++b) sc[b] = sp[b];
        } else if (row != -1) {
          atomicExch(&hdr->status, int32_t(DS4X_EDEVICE));
        }
      }
#pragma unroll
      for (int b = 0; b < kNopeBlocks; ++b) {
        const uint32_t m = redux_max_u(sc[b]);
        if (lane == 0 && m > 0) atomicMax(&sm.sb[b], int(m));
      }
    }
    if (named_bar_or(1, kThreads, !ok)) break;
    // ---- Q': thread (head tid / 8, block tid % 8) ----------------------------------
    {
      const int h = tid >> 3, b = tid & 7;
      const int sh_b = sm.sb[b] - 127;
      const uint4 *src = reinterpret_cast<const uint4 *>(a.q + (int64_t(qi) * kHeads + h) * kDim + 64 * b);
      uint4 v[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) v[c] = src[c];
      int emax = -1;  // largest bf16 exponent field among the normal values
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint32_t w4[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int e0 = int((w4[u] >> 7) & 0xff), e1 = int((w4[u] >> 23) & 0xff);
          if (e0 != 0) emax = max(emax, e0);
          if (e1 != 0) emax = max(emax, e1);
        }
      }
      int eh = emax < 0 ? -100000 : emax - 127 + sh_b;
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) eh = max(eh, __shfl_xor_sync(0xffffffffu, eh, o));
      const int c_h = eh == -100000 ? 0 : 14 - eh;
      const int shift = sh_b + c_h;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint32_t w4[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
        uint32_t o4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float x0 = ldexpf(__uint_as_float(w4[u] << 16), shift);
          const float x1 = ldexpf(__uint_as_float(w4[u] & 0xffff0000u), shift);
          const __half2 hv = __floats2half2_rn(x0, x1);
          o4[u] = *reinterpret_cast<const uint32_t *>(&hv);
        }
        *reinterpret_cast<uint4 *>(sm.qs + q_off(h, 8 * b + c)) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
      }
      if (b == 0) sm.qscale[h] = ldexpf(a.scale * kLog2e, -c_h);
    }
    fence_proxy_async_smem();

    float m_ref[16], sums[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      m_ref[i] = -INFINITY;
      sums[i] = 0.0f;
    }
    for (int t = 0; t < n_tiles; ++t, ++g) {
      // ---- widen tile t into V' (after the previous tile's second MMA) ----------
      if (g > 0 && !wait_bar(sm, &sm.pv_done, (g - 1) & 1, hdr)) ok = false;
#pragma unroll 1
      for (int ps = 0; ps < 2; ++ps) {
        const int rr = 64 * ps + 8 * (warp >> 1) + (lane & 7);
        const int j = 4 * (warp & 1) + (lane >> 3);
        const int pos = kTile * t + rr;
        const int32_t row = pos < a.k ? idxq[pos] : -1;
        const bool valid = row >= 0 && int64_t(row) < a.n_rows;
        if (j == 0) sm.rvalid[rr] = valid ? 1 : 0;
        uint4 oc[8];
        if (valid) {
          const uint8_t *rowp = a.kv + int64_t(row) * DS4X_KV_ROW_BYTES;
          const uint32_t o3 = uint32_t(reinterpret_cast<uintptr_t>(rowp)) & 3u;
          const uint32_t *wn = reinterpret_cast<const uint32_t *>(rowp + 56 * j - o3);
          const uint32_t *wr = reinterpret_cast<const uint32_t *>(rowp + DS4X_KV_NOPE + 16 * j - o3);
          uint32_t raw[15], rw[5];
#pragma unroll
          for (int i = 0; i < 15; ++i) raw[i] = __ldg(wn + i);
#pragma unroll
          for (int i = 0; i < 5; ++i) rw[i] = __ldg(wr + i);
          const int blo = (7 * j) >> 3, bhi = (7 * j + 6) >> 3;
          const uint8_t *scp = rowp + DS4X_KV_NOPE + 2 * DS4X_KV_ROPE;
          const uint32_t flo = pow2_half_bits(int(__ldg(scp + blo)) - sm.sb[blo]) * 0x10001u;
          const uint32_t fhi = pow2_half_bits(int(__ldg(scp + bhi)) - sm.sb[bhi]) * 0x10001u;
          const uint32_t sh = 8u * o3;
#pragma unroll
          for (int i = 0; i < 7; ++i) {
            const uint32_t f = ((7 * j + i) >> 3) == blo ? flo : fhi;
            const uint32_t u0 = __funnelshift_r(raw[2 * i], raw[2 * i + 1], sh);
            const uint32_t u1 = __funnelshift_r(raw[2 * i + 1], raw[2 * i + 2], sh);
            oc[i] = make_uint4(hmul2_bits(e4m3x2_to_f16x2(u0 & 0xffffu), f), hmul2_bits(e4m3x2_to_f16x2(u0 >> 16), f),
                               hmul2_bits(e4m3x2_to_f16x2(u1 & 0xffffu), f), hmul2_bits(e4m3x2_to_f16x2(u1 >> 16), f));
          }
          oc[7] = make_uint4(__funnelshift_r(rw[0], rw[1], sh), __funnelshift_r(rw[1], rw[2], sh),
                             __funnelshift_r(rw[2], rw[3], sh), __funnelshift_r(rw[3], rw[4], sh));
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) oc[i] = make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int i = 0; i < 7; ++i) *reinterpret_cast<uint4 *>(sm.kv + kv_off(rr, 7 * j + i)) = oc[i];
        *reinterpret_cast<uint4 *>(sm.kv + kv_off(rr, 56 + j)) = oc[7];
      }
      fence_proxy_async_smem();
      if (named_bar_or(1, kThreads, !ok)) {  // every warp's V' (and Q', rvalid) written
        aborted = true;
        break;
      }
      if (tid == 0) {
        tc_fence_after();
#pragma unroll 4
        for (int ks = 0; ks < kDim / 16; ++ks)
          mma_f16_ss(tmem + kSCol, smem_desc_noswizzle(kv_a + 256u * ks, 128, 8192),
                     smem_desc_noswizzle(q_a + 256u * ks, 128, 8192), kIdS, ks > 0 ? 1u : 0u);
        tc_commit(smem_u32(&sm.s_full));
        pending = 1;
      }

      // ---- softmax of tile t ------------------------------------------------------
      if (!wait_bar(sm, &sm.s_full, g & 1, hdr)) ok = false;
      tc_fence_after();
      uint32_t sv[16];
      tc_ld_x16(tmem + lane_base + kSCol + 16u * hg, sv);
      tc_wait_ld();
      const bool rv = sm.rvalid[r_sm] != 0;
      float l[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) l[i] = rv ? __uint_as_float(sv[i]) * sm.qscale[16 * hg + i] : -INFINITY;
      float *red = &sm.red[rp & 1][0][0];
      ++rp;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int mx = redux_max(ordered_int(l[i]));
        if (lane == i) red[qd * kHeads + 16 * hg + i] = ordered_float(mx);
      }
      named_bar_sync(2, kThreads);
      bool rescale = false;
      float alpha[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int hh = 16 * hg + i;
        const float mt = fmaxf(fmaxf(red[hh], red[kHeads + hh]), fmaxf(red[2 * kHeads + hh], red[3 * kHeads + hh]));
        alpha[i] = 1.0f;
        if (mt > m_ref[i] + kLazy) {
          alpha[i] = m_ref[i] == -INFINITY ? 0.0f : ex2(m_ref[i] - mt);
          m_ref[i] = mt;
          sums[i] *= alpha[i];
          rescale = true;
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
      uint32_t ph[8], pl[8];
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        const float p0 = rv ? ex2(l[i] - m_ref[i]) : 0.0f;
        const float p1 = rv ? ex2(l[i + 1] - m_ref[i + 1]) : 0.0f;
        sums[i] += p0;
        sums[i + 1] += p1;
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
      fence_proxy_async_smem();
      tc_fence_before();
      if (named_bar_or(1, kThreads, !ok)) {  // every warp's P^T (and O^T rescale) written
        aborted = true;
        break;
      }
      if (tid == 0) {
        tc_fence_after();
#pragma unroll 1
        for (int mi = 0; mi < kDim / 128; ++mi) {
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks) {
            const uint64_t ad = smem_desc_noswizzle(kv_a + 2048u * mi + 16384u * ks, 8192, 128);
            mma_f16_ss(tmem + kOCol + 64u * mi, ad, smem_desc_noswizzle(ph_a + 2048u * ks, 1024, 128), kIdO,
                       (t > 0 || ks > 0) ? 1u : 0u);
            mma_f16_ss(tmem + kOCol + 64u * mi, ad, smem_desc_noswizzle(pl_a + 2048u * ks, 1024, 128), kIdO, 1u);
          }
        }
        tc_commit(smem_u32(&sm.pv_done));
        pending = 2;
      }
    }
    if (aborted) break;

    // ---- the query's output: O^T / sum, block scales put back ---------------------------
    if (!wait_bar(sm, &sm.pv_done, (g - 1) & 1, hdr)) ok = false;
    tc_fence_after();
    float *red = &sm.red[rp & 1][0][0];
    ++rp;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float s = sums[i];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == i) red[qd * kHeads + 16 * hg + i] = s;
    }
    if (named_bar_or(1, kThreads, !ok)) break;
    float inv[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int hh = 16 * hg + i;
      const float tot = (red[hh] + red[kHeads + hh]) + (red[2 * kHeads + hh] + red[3 * kHeads + hh]);
      inv[i] = tot > 0.0f ? 1.0f / tot : 0.0f;
      if (a.lse != nullptr && qd == 0 && lane == i)
        a.lse[int64_t(qi) * kHeads + hh] = tot > 0.0f ? (m_ref[i] + log2f(tot)) * 0.6931471805599453f : -INFINITY;
    }
    uint16_t *outq = a.out + int64_t(qi) * kHeads * kDim;
#pragma unroll 1
    for (int mi = 0; mi < kDim / 128; ++mi) {
      uint32_t ov[16];
      tc_ld_x16(tmem + lane_base + kOCol + 64u * mi + 16u * hg, ov);
      tc_wait_ld();
      const int d = 128 * mi + 32 * qd + lane;
      const float fb = ldexpf(1.0f, sm.sb[d >> 6] - 127);
#pragma unroll
      for (int i = 0; i < 16; ++i)
        outq[(16 * hg + i) * kDim + d] = f32_to_bf16_rn((__uint_as_float(ov[i]) * inv[i]) * fb);
    }
    tc_fence_before();
  }
  if (aborted || !ok) {  // thread 0: no MMA may still write this CTA's memory when it exits
    if (tid == 0 && pending == 1) drain_bar(&sm.s_full, (g - 1 + (aborted ? 1 : 0)) & 1);
    if (tid == 0 && pending == 2) drain_bar(&sm.pv_done, (g - 1) & 1);
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

cudaError_t launch_attn_prefill(const uint8_t *kv_rows, int64_t n_rows, const int32_t *idx, int32_t n_queries,
                                int32_t k, const uint16_t *q, float scale, uint16_t *out, float *lse, void *ws,
                                cudaStream_t stream) {
  static std::atomic<uint64_t> smem_set{0};
  const int smem = int(sizeof(ASmem)) + 128;
  cudaError_t e = set_max_smem_once(attn_prefill_kernel, smem, smem_set);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  PrefillAttnArgs a{kv_rows, n_rows, idx, n_queries, k, scale, q, out, lse};
  const int grid = n_queries < sms ? n_queries : sms;
  attn_prefill_kernel<<<grid, kThreads, smem, stream>>>(a, reinterpret_cast<WsHeader *>(ws));
  return cudaGetLastError();
}

}  // namespace ds4x
