// fa_noalloc.cu -- fa_bwd_noalloc: the backward pass with its workspace taken
// from memory the library reserves when it is loaded, for callers that
// cannot allocate device memory themselves.
//
// The scratch is one file-scope device array.  Host code never uses the
// array's name as an address (on the host it is only a stand-in symbol);
// every call, with the caller's device current, looks up the array's device
// address on that device with cudaGetSymbolAddress.  The lookup allocates
// nothing, and doing it on every call keeps the address right even after the
// device's context has been torn down and re-created (cudaDeviceReset reloads
// the module, and the array may then sit elsewhere).
#include "fa.h"
#include "fa_internal.h"

namespace fa {
namespace {

// Workspace of fa_bwd_noalloc, shared by every call on a device.  Each call
// clears and rewrites what it uses (the backward's first kernel writes both
// row vectors and the counters and clears the dQ accumulator), so leftover
// contents from an earlier call do not matter; calls that overlap on the GPU
// would race on it.
static __device__ __align__(256) unsigned char g_bwd_scratch[FA_BWD_NOALLOC_MAX_WORKSPACE];

// Device address of g_bwd_scratch on the current device.
int scratch_address(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  *out = p;
  return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" int fa_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                              const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int N_q, int N_kv,
                              int d, int causal, float scale, fa_stream_t stream) {
  // Argument checks: the backward with no workspace checks every other argument
  // first and returns FA_ERR_WORKSPACE only when they are all valid; it
  // launches nothing and makes no CUDA call on that path.
  const int st = fa::bwd_entry(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N_q, N_kv, d, causal, scale, 0, false, nullptr, 0,
                               false, static_cast<cudaStream_t>(stream));
  if (st != FA_ERR_WORKSPACE) return st;
  const size_t need = fa_bwd_workspace_bytes(B, H, N_q, N_kv, d);
  if (need > FA_BWD_NOALLOC_MAX_WORKSPACE) return FA_ERR_WORKSPACE;   // problem too large for the scratch
  void* ws = nullptr;
  const int sa = fa::scratch_address(&ws);
  if (sa != FA_OK) return sa;
  return fa::bwd_entry(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N_q, N_kv, d, causal, scale, 0, false, ws,
                       FA_BWD_NOALLOC_MAX_WORKSPACE, true, static_cast<cudaStream_t>(stream));
}
