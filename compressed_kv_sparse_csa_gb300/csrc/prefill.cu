// Chunked-prefill query quantiser (DS4X README, "Packed prefill
// implementation": the batch score/top-k over the packed indexer rows for a
// chunk of query tokens; the scorer itself is in prefill_score.cu).
//
// quantize_query_kernel: each 128-value query vector (one token, one head)
// becomes E4M3 codes with one UE8M0 scale per 32 values, with the block scale
// rule of the cache writer (least e with amax <= 448 * 2^e) and the hardware
// round-to-nearest-even E4M3 converter; one warp per vector.  The codes and
// scales are exactly the block-scaled B operand the prefill scorer's MMA
// reads.
#include "ds4x_internal.cuh"

namespace ds4x {
namespace {

constexpr int kQBlock = 32;

__global__ void __launch_bounds__(256) quantize_query_kernel(const float *__restrict__ q, int64_t n_vec,
                                                             uint8_t *__restrict__ codes,
                                                             uint8_t *__restrict__ scales) {
  // launched as a programmatic dependent: the previous kernel is complete and
  // visible past this wait; the next kernel's CTAs may be scheduled from now on
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int64_t v = int64_t(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (v >= n_vec) return;
  // lane owns elements 4 lane .. 4 lane + 3; block b = lane / 8
  const float4 x = reinterpret_cast<const float4 *>(q + v * DS4X_IDX_DIM)[lane];
  float amax = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const int e = block_exponent(amax, 0.875f, 9);  // 448 = 0.875 * 2^9
  const float s = pow2_neg(e);
  const uint32_t lo = cvt_e4m3x2(x.y * s, x.x * s), hi = cvt_e4m3x2(x.w * s, x.z * s);
  reinterpret_cast<uint32_t *>(codes + v * DS4X_IDX_DIM)[lane] = lo | (hi << 16);
  if ((lane & 7) == 0) scales[v * (DS4X_IDX_DIM / kQBlock) + (lane >> 3)] = uint8_t(e + 127);
}

}  // namespace

cudaError_t launch_quantize_query(const float *q, int64_t n_vec, uint8_t *codes, uint8_t *scales,
                                  cudaStream_t stream) {
  const int warps = 8;
  const int64_t blocks = (n_vec + warps - 1) / warps;
  return launch_pdl(quantize_query_kernel, unsigned(blocks), warps * 32, 0, stream, q, n_vec, codes, scales);
}

}  // namespace ds4x
