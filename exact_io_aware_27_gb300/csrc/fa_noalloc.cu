// fa_backward_noalloc: the backward pass for callers that cannot allocate
// device memory (see include/fa.h). Its workspace is the file-scope array
// below instead of a caller buffer; everything else is fa_backward's path.
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_internal.h"

namespace fa {
namespace {

// Shared by every call on a device; allocated when the library's device code
// is loaded on that device and held until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_workspace[FA_NOALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
void* g_workspace_addr[kMaxDevices];  // device address of the array, per device
std::mutex g_mu;

// Looks up (once per device, with that device current) the device address of
// the array. Host code cannot use the array's name as a device pointer.
int noalloc_workspace(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_workspace_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_workspace) != cudaSuccess || !p) return FA_ERR_CUDA;
    g_workspace_addr[dev] = p;
  }
  *out = g_workspace_addr[dev];
  return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" int fa_backward_noalloc(const void* Q, const void* K, const void* V, const void* O,
                                   const float* L, const void* dO, int B, int H, int n, int m,
                                   int d, int causal, float scale, void* dQ, void* dK, void* dV,
                                   void* stream) {
  const size_t need = fa_backward_workspace_size(B, H, n, m, d);
  if (need == 0) {
    // invalid sizes: let fa_backward's own checks name the error
    return fa_backward(Q, K, V, O, L, dO, B, H, n, m, d, causal, scale, dQ, dK, dV, nullptr, 0,
                       stream);
  }
  if (need > (size_t)FA_NOALLOC_WORKSPACE_BYTES) return FA_ERR_WORKSPACE_TOO_SMALL;
  // Argument checks that need no device first, so bad calls touch no CUDA state
  // (fa_backward repeats them, with the overlap checks, once the workspace is known).
  if (!Q || !K || !V || !O || !L || !dO || !dQ || !dK || !dV) return FA_ERR_INVALID_ARG;
  for (const void* p : {Q, K, V, O, dO, static_cast<const void*>(dQ),
                        static_cast<const void*>(dK), static_cast<const void*>(dV)})
    if (reinterpret_cast<uintptr_t>(p) & 15u) return FA_ERR_MISALIGNED;
  if (reinterpret_cast<uintptr_t>(L) & 3u) return FA_ERR_MISALIGNED;
  void* ws = nullptr;
  const int rc = fa::noalloc_workspace(&ws);
  if (rc != FA_OK) return rc;
  return fa_backward(Q, K, V, O, L, dO, B, H, n, m, d, causal, scale, dQ, dK, dV, ws,
                     (size_t)FA_NOALLOC_WORKSPACE_BYTES, stream);
}
