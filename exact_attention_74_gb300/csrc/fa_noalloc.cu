// fa_noalloc.cu -- fa_bwd_noalloc: the backward pass with its workspace taken
// from memory the library reserves when it is loaded, for callers that
// cannot allocate device memory themselves.
//
// The scratch is one file-scope device array.  Host code never uses the
// array's name as an address (on the host it is only a stand-in symbol); the
// first call on each device, with that device current, resolves the real
// device address with cudaGetSymbolAddress and keeps it for later calls.
#include <mutex>

#include "fa.h"
#include "fa_internal.h"

namespace fa {
namespace {

// Workspace of fa_bwd_noalloc, shared by every call on a device.  Each call
// clears and rewrites what it uses (fa_bwd's first kernel zeroes the dQ
// accumulator and writes both row vectors), so leftover contents from an
// earlier call do not matter; calls that overlap on the GPU would race on it.
static __device__ __align__(256) unsigned char g_bwd_scratch[FA_BWD_NOALLOC_MAX_WORKSPACE];

constexpr int kMaxDevices = 128;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_bwd_scratch on the current device (set up once).
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return FA_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" int fa_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                              const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int N_q, int N_kv,
                              int d, int causal, float scale, fa_stream_t stream) {
  // Argument checks: fa_bwd with no workspace checks every other argument
  // first and returns FA_ERR_WORKSPACE only when they are all valid; it
  // launches nothing and makes no CUDA call on that path.
  const int st = fa_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N_q, N_kv, d, causal, scale, nullptr, 0, stream);
  if (st != FA_ERR_WORKSPACE) return st;
  const size_t need = fa_bwd_workspace_bytes(B, H, N_q, N_kv, d);
  if (need > FA_BWD_NOALLOC_MAX_WORKSPACE) return FA_ERR_WORKSPACE;   // problem too large for the scratch
  void* ws = nullptr;
  const int sa = fa::scratch_address(&ws);
  if (sa != FA_OK) return sa;
  return fa_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N_q, N_kv, d, causal, scale, ws,
                FA_BWD_NOALLOC_MAX_WORKSPACE, stream);
}
