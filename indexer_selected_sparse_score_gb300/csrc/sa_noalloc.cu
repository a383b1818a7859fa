// sa_fused_decode_noalloc: the fused step for callers that cannot allocate
// device memory.  It runs the same kernels as sa_fused_decode, but its scratch
// (index scores, top-k indices when the caller passes none, split-KV partials)
// lives in one fixed, library-owned device array instead of a caller
// workspace.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

// Bytes of the library-owned scratch array (see SA_NOALLOC_SCRATCH_BYTES).
constexpr size_t kNoAllocScratchBytes = SA_NOALLOC_SCRATCH_BYTES;

// The scratch itself.  Every GPU that loads this library holds it until the
// process exits; every call of sa_fused_decode_noalloc on a device shares it.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device.  In host code
// the symbol's name is only a host-side handle; the device address comes from
// cudaGetSymbolAddress, looked up once per device with that device current.
cudaError_t scratch_address(void **ptr) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *ptr = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" sa_status sa_fused_decode_noalloc(const sa_index_args *ia, const sa_attn_args *aa,
                                             int32_t K, int32_t *idx_out, void *out,
                                             uint32_t *device_status, sa_stream_t stream) {
  if (!ia || !aa) return sa::set_error(SA_ERR_INVALID_ARG, "index or attention args pointer is NULL");
  if (K < 0) return sa::set_error(SA_ERR_INVALID_ARG, "K must be >= 0");
  if ((reinterpret_cast<uintptr_t>(device_status) & 3u) != 0)
    return sa::set_error(SA_ERR_INVALID_ARG, "device_status must be 4-byte aligned");
  const size_t need = sa_workspace_size(ia, aa, K);
  if (need == 0) return sa::set_error(SA_ERR_INVALID_ARG, "arguments rejected (see the other entry points' checks)");
  if (need > kNoAllocScratchBytes)
    return sa::set_error(SA_ERR_UNSUPPORTED,
                         "problem needs %zu bytes of scratch; sa_fused_decode_noalloc has %zu "
                         "(use sa_fused_decode with a caller workspace)",
                         need, kNoAllocScratchBytes);
  void *scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess)
    return sa::set_error(SA_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
  // No part of the scratch has to start at zero: every scratch element a
  // kernel reads was written earlier in the same call.  The status word the
  // kernels flag into is the caller's device_status (or none).
  return sa::fused_with_scratch(ia, aa, K, idx_out, out, scratch, need, device_status,
                                reinterpret_cast<cudaStream_t>(stream));
}
