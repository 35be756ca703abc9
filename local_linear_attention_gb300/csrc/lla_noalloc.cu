// lla_forward_noalloc: the causal LLA forward for callers that cannot allocate device memory.
//
// Some callers are not allowed to allocate GPU memory themselves: a plugin that a host
// application only hands input and output buffers, or a latency-critical loop that must not call
// the allocator once it is running (an allocation can block on the device or fail under memory
// pressure at an unpredictable moment). lla_forward allocates its scratch and lla_forward_ws
// needs the caller to supply it; this entry point needs neither. Its scratch is one fixed-size
// array in device memory that belongs to the library: every GPU that loads this part of the
// library holds it (kNoAllocScratchBytes) until the process exits.
//
// The array's name is only a stand-in in host code, not a device address, so the host side looks
// up the real address once per device (cudaGetSymbolAddress, with that device current) and passes
// it on like any other workspace pointer. The computation is exactly lla_forward_ws's.
#include <mutex>

#include "lla_internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)LLA_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device; looked up on the first call per
// device and cached.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (err != cudaSuccess) return err;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int lla_forward_noalloc(const void* q, const void* k, const void* v, void* out, int B,
                                   int H, int T, int d, int dv, float h, float lambda, int dtype,
                                   void* stream) {
  const size_t need = lla_workspace_size(B, H, T, d, dv, dtype);
  if (need > kNoAllocScratchBytes) return LLA_ERR_UNSUPPORTED;
  if (need == 0)  // invalid sizes or an empty problem: lla_forward_ws reports it, touching nothing
    return lla_forward_ws(q, k, v, out, B, H, T, d, dv, h, lambda, dtype, nullptr, 0, stream);
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return LLA_ERR_CUDA;
  // Every stage writes the part of the scratch it later reads before reading it, so nothing left
  // over from an earlier call needs clearing.
  return lla_forward_ws(q, k, v, out, B, H, T, d, dv, h, lambda, dtype, scratch,
                        kNoAllocScratchBytes, stream);
}
