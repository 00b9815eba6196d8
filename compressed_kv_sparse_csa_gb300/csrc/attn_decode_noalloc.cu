// ds4x_sparse_attn_decode_noalloc: the sparse decode attention for callers
// that cannot allocate device memory.
//
// Some hosts cannot hand this library a workspace: an engine whose device
// memory is carved up once at start-up and never grows, or a plugin living
// inside a runtime that offers it no allocator and where a cudaMalloc in the
// middle of a decode step would synchronise the whole device.  This entry
// point needs no workspace: the kernel keeps its split partials in shared
// memory, and the workspace header it writes its status to is one
// file-scope device array, which every GPU that loads the library keeps for
// the life of the process.  It launches exactly the kernel
// ds4x_sparse_attn_decode launches.
#include <atomic>

#include "ds4x_internal.cuh"

namespace {

// The workspace ds4x_sparse_attn_decode needs for any k: the 256-byte header.
constexpr size_t kNoAllocScratchBytes = ds4x::kWsHeaderBytes;

static __device__ __align__(256) unsigned char g_attn_scratch[kNoAllocScratchBytes];

// Device address of g_attn_scratch, looked up once per device.  In host code
// the array's name only stands in for the symbol; its device address must
// come from cudaGetSymbolAddress with that device current.
std::atomic<void *> g_scratch_addr[64];

int scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DS4X_ECUDA;
  if (dev < 0 || dev >= 64) return DS4X_EINVAL;
  void *p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || p == nullptr) return DS4X_ECUDA;
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return DS4X_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int require_gb300() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    return DS4X_ECUDA;
  }
  return (major == 10 && minor == 3) ? DS4X_OK : DS4X_EARCH;
}

}  // namespace

extern "C" int ds4x_sparse_attn_decode_noalloc(const uint8_t *kv_rows, int64_t n_rows, const int32_t *idx,
                                               int32_t k, const uint16_t *q_bf16, float softmax_scale,
                                               uint16_t *out_bf16, float *lse, ds4x_stream_t stream) {
  if (kv_rows == nullptr || idx == nullptr || q_bf16 == nullptr || out_bf16 == nullptr) return DS4X_EINVAL;
  if (!aligned16(kv_rows) || !aligned16(idx) || !aligned16(q_bf16) || !aligned16(out_bf16) ||
      (lse != nullptr && !aligned16(lse)))
    return DS4X_EINVAL;
  if (n_rows < 1 || k < 1 || k > DS4X_TOPK_MAX) return DS4X_EINVAL;
  if (ds4x::attn_decode_ws_bytes(k) > kNoAllocScratchBytes) return DS4X_EWORKSPACE;
  int st = require_gb300();
  if (st != DS4X_OK) return st;
  void *scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != DS4X_OK) return st;
  const cudaError_t e = ds4x::launch_attn_decode(kv_rows, n_rows, idx, k, q_bf16, softmax_scale, out_bf16, lse,
                                                 scratch, stream);
  return e == cudaSuccess ? DS4X_OK : DS4X_ECUDA;
}
