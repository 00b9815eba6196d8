// Thin inline-PTX wrappers for the sm_103a features the tensor-core kernels
// use: mbarriers, 1-D bulk (TMA) copies, tensor memory (tcgen05.alloc/ld/st),
// block-scaled tcgen05.mma with the A operand in tensor memory, fp16
// tcgen05.mma with both operands in shared memory, and named barriers.
#pragma once

#include <stdint.h>

namespace ds4x {
namespace ptx {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier --------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, but the thread may sleep in hardware up to `hint_ns`
// (returning early when the phase completes) instead of re-polling.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// ---- bulk copy global -> shared, completion counted on an mbarrier ----------
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// An L2 policy for data read once (evicted first, so it does not push out
// what later phases reuse), and the bulk copy that takes it.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// ---- tensor memory -----------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 consecutive 32-bit columns: this thread's lane, columns taddr..taddr+31.
__device__ __forceinline__ void tc_st_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tc_ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// Instruction descriptor, kind::mxf8f6f4 with block scaling (UE8M0 scale
// factors, one per 32 K-elements): A type E2M1 (5), B type E4M3 (0), both
// K-major, fp32 D, M = 128; the scale-factor byte ids of A (bits 29-30) and
// B (bits 4-5) are OR-ed in per K step.
__host__ __device__ constexpr uint32_t idesc_mxf8f6f4_e2m1_e4m3(uint32_t N) {
  return (5u << 7) | (0u << 10) | ((N >> 3) << 17) | (1u << 23) | (1u << 27);
}

// One 128-row tile against the whole 128-element K extent and two B operands
// (N = 64 each) summed into one accumulator: K step s (32 elements) issues
// D (+)= (A_s * SFA_s)(B1_s * SFB1_s)^T and D += (A_s * SFA_s)(B2_s * SFB2_s)^T,
// block-scaled.  A is in tensor memory (one E2M1 code per byte, in bits 5-2;
// 8 columns per step), B1 and B2 in shared memory (descriptors + 16 = 256
// bytes per step); step s reads byte s of every scale-factor word (ids s).
// The first MMA overwrites D.  Scale-factor columns start on 4-column
// boundaries.
__device__ __forceinline__ void mma_mxf8f6f4_ta_k128_2b(uint32_t d_tmem, uint32_t a_tmem, uint64_t b1_desc0,
                                                        uint64_t b2_desc0, uint32_t idesc, uint32_t sfa_tmem,
                                                        uint32_t sfb1_tmem, uint32_t sfb2_tmem) {
  asm volatile(
      "{\n\t.reg .pred pf, pt;\n\t.reg .b32 a, id;\n\t.reg .b64 b1, b2;\n\t"
      "setp.ne.b32 pf, %4, %4;\n\tsetp.eq.b32 pt, %4, %4;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], [%1], %2, %4, [%5], [%6], pf;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], [%1], %3, %4, [%5], [%7], pt;\n\t"
      "add.u32 a, %1, 8;\n\tadd.s64 b1, %2, 16;\n\tadd.s64 b2, %3, 16;\n\tor.b32 id, %4, 0x20000010;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], [a], b1, id, [%5], [%6], pt;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], [a], b2, id, [%5], [%7], pt;\n\t"
      "add.u32 a, a, 8;\n\tadd.s64 b1, b1, 16;\n\tadd.s64 b2, b2, 16;\n\tor.b32 id, %4, 0x40000020;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], [a], b1, id, [%5], [%6], pt;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], [a], b2, id, [%5], [%7], pt;\n\t"
      "add.u32 a, a, 8;\n\tadd.s64 b1, b1, 16;\n\tadd.s64 b2, b2, 16;\n\tor.b32 id, %4, 0x60000030;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], [a], b1, id, [%5], [%6], pt;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], [a], b2, id, [%5], [%7], pt;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b1_desc0), "l"(b2_desc0), "r"(idesc), "r"(sfa_tmem), "r"(sfb1_tmem),
        "r"(sfb2_tmem)
      : "memory");
}

// The same with one B operand (the query's lo piece is all zero): four MMAs,
// K step s reading scale-factor byte s.
__device__ __forceinline__ void mma_mxf8f6f4_ta_k128_1b(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc0,
                                                        uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem) {
  asm volatile(
      "{\n\t.reg .pred pf, pt;\n\t.reg .b32 a, id;\n\t.reg .b64 b;\n\t"
      "setp.ne.b32 pf, %3, %3;\n\tsetp.eq.b32 pt, %3, %3;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], [%1], %2, %3, [%4], [%5], pf;\n\t"
      "add.u32 a, %1, 8;\n\tadd.s64 b, %2, 16;\n\tor.b32 id, %3, 0x20000010;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], [a], b, id, [%4], [%5], pt;\n\t"
      "add.u32 a, a, 8;\n\tadd.s64 b, b, 16;\n\tor.b32 id, %3, 0x40000020;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], [a], b, id, [%4], [%5], pt;\n\t"
      "add.u32 a, a, 8;\n\tadd.s64 b, b, 16;\n\tor.b32 id, %3, 0x60000030;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], [a], b, id, [%4], [%5], pt;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc0), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// tcgen05.st of one / four 32-bit columns (32 lanes x 32 bits each).
__device__ __forceinline__ void tc_st_x1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}
__device__ __forceinline__ void tc_st_x4(uint32_t taddr, uint32_t v0, uint32_t v1, uint32_t v2, uint32_t v3) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(v0), "r"(v1),
               "r"(v2), "r"(v3)
               : "memory");
}

// Arrive (once) on an mbarrier when every tcgen05 op this thread issued so far completes.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// Shared-memory matrix descriptor, no swizzle, K-major: core matrices of
// 8 rows x 16 bytes; lbo = byte distance between core matrices along K,
// sbo = along M/N.
__device__ __forceinline__ uint64_t smem_desc_noswizzle(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return uint64_t((saddr & 0x3FFFFu) >> 4) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
         (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46);
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also ORs a predicate over its nthreads participants:
// every participant gets the same result.
__device__ __forceinline__ bool named_bar_or(uint32_t id, uint32_t nthreads, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %3, 0;\n\tbar.red.or.pred q, %1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(id), "r"(nthreads), "r"(uint32_t(v))
      : "memory");
  return r != 0;
}

// ---- kind::f16 (fp16 operands, fp32 accumulate) --------------------------------
// Instruction descriptor: D f32 (bits 4-5 = 1), A and B fp16 (type 0), A / B
// K-major (0) or MN-major (1) in bits 15 / 16, N >> 3 in bits 17-22, M >> 4 in
// bits 24-28.
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t M, uint32_t N, uint32_t a_mn, uint32_t b_mn) {
  return (1u << 4) | (a_mn << 15) | (b_mn << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// D (+)= A * B with A and B in shared memory (descriptors); accumulate when acc != 0.
// With no swizzle the descriptor's leading byte offset is the distance between
// core matrices adjacent along K and the stride byte offset the distance along
// M (or N), for K-major and MN-major operands alike.
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc)
      : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns: this thread's lane, columns taddr..taddr+15.
__device__ __forceinline__ void tc_st_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

}  // namespace ptx
}  // namespace ds4x
