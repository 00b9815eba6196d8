// Kernel-side copy between device memory and page-locked host memory (or
// within either): each thread moves 16-byte words, the tail byte by byte.  A
// decode loop whose inputs and results live in pinned host memory can move
// them with this kernel inside its CUDA graph instead of copy-engine copies,
// whose hand-over to and from the kernels costs several microseconds each.
// Launched as a programmatic dependent of the previous kernel (it waits for it
// before touching memory), and lets its own dependents be scheduled at once.
#include "ds4x_internal.cuh"

namespace ds4x {
namespace {

constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads) copy16_kernel(uint4 *__restrict__ dst, const uint4 *__restrict__ src,
                                                              size_t n16, uint8_t *__restrict__ dst_tail,
                                                              const uint8_t *__restrict__ src_tail, uint32_t tail) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const size_t stride = size_t(gridDim.x) * blockDim.x;
  for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride) dst[i] = src[i];
  if (blockIdx.x == 0 && threadIdx.x < tail) dst_tail[threadIdx.x] = src_tail[threadIdx.x];
}

}  // namespace

cudaError_t launch_copy(void *dst, const void *src, size_t bytes, cudaStream_t stream) {
  const size_t n16 = bytes / 16;
  const uint32_t tail = uint32_t(bytes - 16 * n16);
  const size_t want = (n16 + kCopyThreads - 1) / kCopyThreads;
  const int grid = int(want < 1 ? 1 : (want > 1024 ? 1024 : want));
  return launch_pdl(copy16_kernel, unsigned(grid), kCopyThreads, 0, stream, static_cast<uint4 *>(dst),
                    static_cast<const uint4 *>(src), n16, static_cast<uint8_t *>(dst) + 16 * n16,
                    static_cast<const uint8_t *>(src) + 16 * n16, tail);
}

}  // namespace ds4x
