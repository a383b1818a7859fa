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

// Device addresses of g_noalloc_scratch, one per CUDA context that has
// called in (a device's primary context in the usual case).  In host code the
// symbol's name is only a host-side handle; the device address comes from
// cudaGetSymbolAddress, looked up once per context with that context current.
// Keying on the context rather than the device ordinal keeps the address
// right after cudaDeviceReset or in a context other than the primary one,
// where the module is loaded anew and the array may move.
constexpr int kMaxContexts = 64;
std::mutex g_setup_mutex;
CUcontext g_ctx[kMaxContexts] = {};
void *g_scratch_addr[kMaxContexts] = {};
int g_n_ctx = 0;

using CtxGetCurrent = CUresult (*)(CUcontext *);

CtxGetCurrent ctx_get_current() {
  static CtxGetCurrent fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrent>(p);
  });
  return fn;
}

cudaError_t scratch_address(void **ptr) {
  CtxGetCurrent get = ctx_get_current();
  if (!get) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  if (!ctx) {  // no context current on this thread yet: the runtime makes the device's primary one current
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaSetDevice(dev);
    if (e != cudaSuccess) return e;
    if (get(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorDeviceUninitialized;
  }
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  for (int i = 0; i < g_n_ctx; ++i)
    if (g_ctx[i] == ctx) {
      *ptr = g_scratch_addr[i];
      return cudaSuccess;
    }
  void *p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  if (g_n_ctx < kMaxContexts) {
    g_ctx[g_n_ctx] = ctx;
    g_scratch_addr[g_n_ctx] = p;
    ++g_n_ctx;
  }
  *ptr = p;
  return cudaSuccess;
}

}  // namespace

extern "C" size_t sa_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

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
