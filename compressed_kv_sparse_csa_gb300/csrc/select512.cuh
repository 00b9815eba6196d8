// Exact selection and sorting of 64-bit (score, index) keys by the 512
// threads 0-511 of a CTA (named barrier 1): shared by the fused decode scorer
// and the prefill top-k.  Keys are sortable (score, index) keys as built by
// make_key; a zero key is padding.
#pragma once

#include <stdint.h>

#include "tc_ptx.cuh"

namespace ds4x {
namespace {

constexpr int kSelThreads = 512;   // threads 0-511 run the selection
constexpr int kSelPerThread = 18;  // keys a selection thread holds: 18 * 512 = 9216 per pass
constexpr int kSelCap = kSelThreads * kSelPerThread;
constexpr uint32_t kBarSel = 1;    // named barrier of the 512 selection threads

struct SelShared {
  unsigned long long red_min[16], red_max[16];
  int red_cnt[16];
  alignas(16) int scan[16];
  uint32_t red_lo[16], red_hi[16];
  int bstar, above, bcnt, out_cnt, list_cnt;
  int c512_b, c512_above, cM_b, cM_above, cM_cnt, total;
  int fill, ncol, wcnt, pub_cnt, n_all, ok, nhi, nge;
  uint32_t base;
  unsigned long long cut;
};

__device__ __forceinline__ void bar512() { ptx::named_bar_sync(kBarSel, kSelThreads); }

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
  for (int size = 2; size <= kSelThreads; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      unsigned long long o;
      if (stride >= 32) {
        buf[pb * kSelThreads + tid] = v;
        bar512();
        o = buf[pb * kSelThreads + (tid ^ stride)];
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
      const int i = tid + q * kSelThreads;
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
    for (int b = tid; b < kAdaptBuckets; b += kSelThreads) hist[b] = 0;
    bar512();
    unsigned long long kmin = ~0ull, kmax = 0;
    int nz = 0;
    for (int w = 0; w < kSelThreads / 32; ++w) {
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
      for (int i = tid; i < bcnt; i += kSelThreads) out[base + i] = list[i];
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
    if (bcnt <= kSelThreads) {
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

}  // namespace
}  // namespace ds4x
