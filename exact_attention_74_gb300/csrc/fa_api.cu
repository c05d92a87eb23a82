// fa_api.cu -- the C-ABI entry points of include/fa.h: argument checks, TMA
// tensor maps, device checks and the device status word.  No entry point
// allocates device memory; argument errors are returned before any CUDA call.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <initializer_list>
#include <mutex>

#include "fa.h"
#include "fa_internal.h"

namespace fa {

// Device status word of the library (one per device that loads the module).
// Kernels OR kStatusTimeout into it; fa_get_last_device_status reads and
// clears it.
__device__ unsigned g_status_word;

namespace {

std::atomic<unsigned long long> g_timeout_ns{1000000000ull};

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

struct DevState {
  bool checked = false;
  bool supported = false;
  int n_sms = 0;
};

bool misaligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) != 0; }

// True when p lies in memory the current device addresses directly: a device
// allocation of this device (or one it has peer access to) or managed
// memory.  Host memory, pinned or not, and unknown addresses are refused, so
// no tensor map or kernel is ever built on them.
bool is_device_memory(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (at.type == cudaMemoryTypeManaged) return true;
  return at.type == cudaMemoryTypeDevice && at.devicePointer != nullptr;
}

int check_device_memory(std::initializer_list<const void*> ptrs) {
  for (const void* p : ptrs)
    if (!is_device_memory(p)) return FA_ERR_INVALID;
  return FA_OK;
}

int check_sizes(int B, int H, int N_q, int N_kv, int d, int causal, float scale) {
  if (B < 1 || H < 1 || N_q < 1 || N_kv < 1) return FA_ERR_INVALID;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID;
  if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H > 0x7fffffffLL) return FA_ERR_INVALID;
  return FA_OK;
}

// Workspace of fa_fwd_fp8: e4m3 copies of Q, K and V (rows padded to 128),
// then the fp32 multipliers of Q and K, the largest |V| of each key block and
// of each (batch, head); each part rounded up to 256 B.
struct Fp8Layout {
  size_t q8, k8, v8, qinv, kinv, vbmax, vamax, total;
};

Fp8Layout fp8_layout(int B, int H, int N_q, int N_kv, int d) {
  auto r256 = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t BH = static_cast<size_t>(B) * H;
  const size_t nqp = (static_cast<size_t>(N_q) + 127) / 128 * 128, nkp = (static_cast<size_t>(N_kv) + 127) / 128 * 128;
  Fp8Layout L;
  L.q8 = 0;
  const size_t dd = static_cast<size_t>(d);
  L.k8 = L.q8 + r256(BH * nqp * dd);
  L.v8 = L.k8 + r256(BH * nkp * dd);
  L.qinv = L.v8 + r256(BH * nkp * dd);
  L.kinv = L.qinv + r256(BH * (nqp / 128) * sizeof(float));
  L.vbmax = L.kinv + r256(BH * (nkp / 128) * sizeof(float));
  L.vamax = L.vbmax + r256(BH * (nkp / 128) * sizeof(float));
  L.total = L.vamax + r256(BH * sizeof(float));
  return L;
}

}  // namespace

// Resolve the current device: must be compute capability 10.3 (sm_103a code
// only); returns the watchdog handle for its kernels and, if asked, its
// multiprocessor count.
int device_ctl(DevCtl* ctl, int* n_sms) {
  static std::mutex mu;
  static DevState states[128];
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  if (dev < 0 || dev >= 128) return FA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> g(mu);
  DevState& s = states[dev];
  if (!s.checked) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      cudaGetLastError();
      return FA_ERR_CUDA;
    }
    s.supported = (major == 10 && minor == 3);
    if (cudaDeviceGetAttribute(&s.n_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return FA_ERR_CUDA;
    }
    s.checked = true;
  }
  if (!s.supported) return FA_ERR_UNSUPPORTED;
  // The status word's device address is looked up on every call (a host-side
  // query): a context torn down and re-created (cudaDeviceReset) reloads the
  // module, and the word may then live elsewhere.
  void* word = nullptr;
  if (cudaGetSymbolAddress(&word, g_status_word) != cudaSuccess || word == nullptr) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  ctl->status = static_cast<unsigned*>(word);
  ctl->timeout_ns = g_timeout_ns.load();
  if (n_sms) *n_sms = s.n_sms;
  return FA_OK;
}

// 3-D map over a contiguous bf16 [BH, N, d] tensor: box 64 (d) x box_rows
// x 1, 128-byte swizzle, out-of-range rows read as zero.
int make_map_bf16(CUtensorMap* m, const void* ptr, int d, int N, int BH, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return FA_ERR_CUDA;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N) * d * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// The same bf16 tensor in boxes of 32 columns (64 bytes) x box_rows x 1 with
// 64-byte swizzle: one half of a d = 64 row per box.
int make_map_bf16_sw64(CUtensorMap* m, const void* ptr, int d, int N, int BH, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return FA_ERR_CUDA;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N) * d * 2};
  cuuint32_t box[3] = {32, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// 3-D map over a contiguous u8 [BH, rows, inner] tensor (inner a multiple of
// 128): 128 x 128 x 1 boxes, 128-byte swizzle.
int make_map_u8(CUtensorMap* m, const void* ptr, int inner, int rows, int BH) {
  auto fn = encode_fn();
  if (!fn) return FA_ERR_CUDA;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows) * inner};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// 3-D map over a contiguous fp32 [BH, N, d] tensor: box box_cols x box_rows
// x 1 with 128-byte swizzle (box_cols * 4 must be 128); rows past N are
// skipped by stores and reductions.
int make_map_f32(CUtensorMap* m, const void* ptr, int d, int N, int BH, int box_cols, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return FA_ERR_CUDA;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(N) * d * 4};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

constexpr int kDefaultEmuPer32 = 0;
constexpr float kDefaultTau = 8.0f;

}  // namespace fa

using namespace fa;

extern "C" {

int fa_fwd_ex(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N_q,
              int N_kv, int d, int causal, float scale, float tau, int emu_per_32, fa_stream_t stream) {
  if (!Q || !K || !V || !O || !LSE) return FA_ERR_INVALID;
  int st = check_sizes(B, H, N_q, N_kv, d, causal, scale);
  if (st != FA_OK) return st;
  if (!(tau >= 0.f && tau <= 16.f)) return FA_ERR_INVALID;
  if (emu_per_32 == -1) emu_per_32 = kDefaultEmuPer32;
  if (emu_per_32 != 0 && emu_per_32 != 8 && emu_per_32 != 16) return FA_ERR_INVALID;
  if (misaligned(Q, 16) || misaligned(K, 16) || misaligned(V, 16) || misaligned(O, 16) ||
      misaligned(LSE, 4))
    return FA_ERR_ALIGN;
  FwdLaunch a;
  st = device_ctl(&a.ctl);
  if (st != FA_OK) return st;
  if ((st = check_device_memory({Q, K, V, O, LSE})) != FA_OK) return st;
  const int BH = B * H;
  if ((st = make_map_bf16(&a.tmQ, Q, d, N_q, BH)) != FA_OK) return st;
  // rows per K box: at d = 256 each CTA of a pair loads 64 keys of a step
  if ((st = make_map_bf16(&a.tmK, K, d, N_kv, BH, d == 256 ? 64 : 128)) != FA_OK) return st;
  if ((st = make_map_bf16(&a.tmV, V, d, N_kv, BH, 128)) != FA_OK) return st;
  if ((st = make_map_bf16(&a.tmO, O, d, N_q, BH, 32)) != FA_OK) return st;
  a.o = O;
  a.lse = LSE;
  a.BH = BH;
  a.N_q = N_q;
  a.N_kv = N_kv;
  a.d = d;
  a.causal = causal;
  a.scale = scale;
  a.tau = tau;
  a.emu_per_32 = emu_per_32;
  a.stream = static_cast<cudaStream_t>(stream);
  const cudaError_t e = (d == 64) ? launch_fwd_d64(a) : (d == 128) ? launch_fwd_d128(a) : launch_fwd_d256(a);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

int fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N_q,
           int N_kv, int d, int causal, float scale, fa_stream_t stream) {
  return fa_fwd_ex(Q, K, V, O, LSE, B, H, N_q, N_kv, d, causal, scale, kDefaultTau, -1, stream);
}

size_t fa_fwd_fp8_workspace_bytes(int B, int H, int N_q, int N_kv, int d) {
  if (check_sizes(B, H, N_q, N_kv, d, 0, 1.0f) != FA_OK || (d != 128 && d != 256)) return 0;
  return fp8_layout(B, H, N_q, N_kv, d).total;
}

int fa_fwd_fp8(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N_q,
               int N_kv, int d, int causal, float scale, const unsigned* signs, void* workspace,
               size_t workspace_bytes, fa_stream_t stream) {
  if (!Q || !K || !V || !O || !LSE) return FA_ERR_INVALID;
  int st = check_sizes(B, H, N_q, N_kv, d, causal, scale);
  if (st != FA_OK) return st;
  if (d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  if (misaligned(Q, 16) || misaligned(K, 16) || misaligned(V, 16) || misaligned(O, 16) ||
      misaligned(LSE, 4))
    return FA_ERR_ALIGN;
  const Fp8Layout L = fp8_layout(B, H, N_q, N_kv, d);
  if (!workspace || workspace_bytes < L.total) return FA_ERR_WORKSPACE;
  if (misaligned(workspace, 256)) return FA_ERR_ALIGN;
  Fp8Launch a;
  st = device_ctl(&a.ctl);
  if (st != FA_OK) return st;
  if ((st = check_device_memory({Q, K, V, O, LSE, workspace})) != FA_OK) return st;
  const int BH = B * H;
  const int nqp = (N_q + 127) / 128 * 128, nkp = (N_kv + 127) / 128 * 128;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.q8 = ws + L.q8;
  a.k8 = ws + L.k8;
  a.v8 = ws + L.v8;
  a.qinv = reinterpret_cast<float*>(ws + L.qinv);
  a.kinv = reinterpret_cast<float*>(ws + L.kinv);
  a.vbmax = reinterpret_cast<float*>(ws + L.vbmax);
  a.vamax = reinterpret_cast<float*>(ws + L.vamax);
  if ((st = make_map_u8(&a.tmQ8, a.q8, d, nqp, BH)) != FA_OK) return st;
  if ((st = make_map_u8(&a.tmK8, a.k8, d, nkp, BH)) != FA_OK) return st;
  if ((st = make_map_u8(&a.tmV8, a.v8, d, nkp, BH)) != FA_OK) return st;
  a.q = Q;
  a.k = K;
  a.v = V;
  a.o = O;
  a.lse = LSE;
  a.BH = BH;
  a.N_q = N_q;
  a.N_kv = N_kv;
  a.causal = causal;
  a.d = d;
  a.hadamard = signs != nullptr;
  for (int i = 0; i < 8; ++i) a.signs[i] = signs && i < d / 32 ? signs[i] : 0u;
  a.scale = scale;
  a.tau = kDefaultTau;
  a.stream = static_cast<cudaStream_t>(stream);
  const cudaError_t e = launch_fwd_fp8(a);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

size_t fa_bwd_workspace_bytes(int B, int H, int N_q, int N_kv, int d) {
  if (check_sizes(B, H, N_q, N_kv, d, 0, 1.0f) != FA_OK || d == 256) return 0;
  const size_t rows = static_cast<size_t>(B) * H * N_q;
  const size_t rows_pad = static_cast<size_t>(B) * H * ((static_cast<size_t>(N_q) + 127) / 128 * 128);
  const size_t acc = (rows * d * sizeof(float) + 255) / 256 * 256;
  const size_t vec = (rows_pad * sizeof(float) + 255) / 256 * 256;
  const size_t cnt = (rows_pad / 128 * sizeof(unsigned) + 255) / 256 * 256;
  return acc + 2 * vec + cnt + 256;   // + the CTA ticket word
}

}  // extern "C"

namespace fa {

// fa_bwd_ex's work; `internal_workspace` marks the library's own scratch
// (fa_bwd_noalloc), whose address is not a caller's allocation and is not
// checked as one.
int bwd_entry(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE,
              void* dQ, void* dK, void* dV, int B, int H, int N_q, int N_kv, int d, int causal, float scale,
              int deterministic, bool pair, void* workspace, size_t workspace_bytes, bool internal_workspace,
              cudaStream_t stream) {
  if (!Q || !K || !V || !O || !dO || !LSE || !dQ || !dK || !dV) return FA_ERR_INVALID;
  int st = check_sizes(B, H, N_q, N_kv, d, causal, scale);
  if (st != FA_OK) return st;
  if (d == 256) return FA_ERR_UNSUPPORTED;   // the backward kernel covers d = 64 and 128
  if (pair && d != 64) return FA_ERR_UNSUPPORTED;   // the pair kernel covers d = 64
  if (deterministic != 0 && deterministic != 1) return FA_ERR_INVALID;
  if (misaligned(Q, 16) || misaligned(K, 16) || misaligned(V, 16) || misaligned(O, 16) ||
      misaligned(dO, 16) || misaligned(dQ, 16) || misaligned(dK, 16) || misaligned(dV, 16) ||
      misaligned(LSE, 4))
    return FA_ERR_ALIGN;
  const size_t need = fa_bwd_workspace_bytes(B, H, N_q, N_kv, d);
  if (!workspace || workspace_bytes < need) return FA_ERR_WORKSPACE;
  if (misaligned(workspace, 256)) return FA_ERR_ALIGN;
  BwdLaunch a;
  st = device_ctl(&a.ctl, &a.n_sms);
  if (st != FA_OK) return st;
  if ((st = check_device_memory({Q, K, V, O, dO, LSE, dQ, dK, dV})) != FA_OK) return st;
  if (!internal_workspace && (st = check_device_memory({workspace})) != FA_OK) return st;
  const int BH = B * H;
  if ((st = make_map_bf16(&a.tmQ, Q, d, N_q, BH)) != FA_OK) return st;
  if ((st = make_map_bf16(&a.tmK, K, d, N_kv, BH)) != FA_OK) return st;
  if ((st = make_map_bf16(&a.tmV, V, d, N_kv, BH)) != FA_OK) return st;
  if ((st = make_map_bf16(&a.tmdO, dO, d, N_q, BH)) != FA_OK) return st;
  if ((st = make_map_f32(&a.tmDQ, workspace, d, N_q, BH, 32, 32)) != FA_OK) return st;
  if (pair) {
    if ((st = make_map_bf16(&a.tmQh, Q, d, N_q, BH, 64)) != FA_OK) return st;
    if ((st = make_map_bf16(&a.tmdOh, dO, d, N_q, BH, 64)) != FA_OK) return st;
    if ((st = make_map_bf16_sw64(&a.tmQc, Q, d, N_q, BH, 128)) != FA_OK) return st;
    if ((st = make_map_bf16_sw64(&a.tmdOc, dO, d, N_q, BH, 128)) != FA_OK) return st;
    if ((st = make_map_bf16_sw64(&a.tmKc, K, d, N_kv, BH, 128)) != FA_OK) return st;
  }
  const size_t rows = static_cast<size_t>(BH) * N_q;
  a.o = O;
  a.dO = dO;
  a.lse = LSE;
  a.dq = dQ;
  a.dk = dK;
  a.dv = dV;
  const size_t rows_pad = static_cast<size_t>(BH) * ((static_cast<size_t>(N_q) + 127) / 128 * 128);
  a.dq_acc = static_cast<float*>(workspace);
  a.delta = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                     (rows * d * sizeof(float) + 255) / 256 * 256);
  a.counters = reinterpret_cast<unsigned*>(reinterpret_cast<char*>(a.delta) +
                                           2 * ((rows_pad * sizeof(float) + 255) / 256 * 256));
  a.ticket = reinterpret_cast<unsigned*>(reinterpret_cast<char*>(a.counters) +
                                         (rows_pad / 128 * sizeof(unsigned) + 255) / 256 * 256);
  a.deterministic = deterministic;
  a.BH = BH;
  a.N_q = N_q;
  a.N_kv = N_kv;
  a.d = d;
  a.causal = causal;
  a.scale = scale;
  a.stream = stream;
  const cudaError_t e = pair ? launch_bwd_pair(a) : launch_bwd(a);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

}  // namespace fa

extern "C" {

int fa_bwd_ex(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE,
              void* dQ, void* dK, void* dV, int B, int H, int N_q, int N_kv, int d, int causal, float scale,
              int deterministic, void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  return bwd_entry(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N_q, N_kv, d, causal, scale, deterministic, false,
                   workspace, workspace_bytes, false, static_cast<cudaStream_t>(stream));
}

int fa_bwd_pair(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE,
                void* dQ, void* dK, void* dV, int B, int H, int N_q, int N_kv, int d, int causal, float scale,
                void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  return bwd_entry(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N_q, N_kv, d, causal, scale, 0, true, workspace,
                   workspace_bytes, false, static_cast<cudaStream_t>(stream));
}

int fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE,
           void* dQ, void* dK, void* dV, int B, int H, int N_q, int N_kv, int d, int causal, float scale,
           void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  return fa_bwd_ex(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N_q, N_kv, d, causal, scale, 0, workspace,
                   workspace_bytes, stream);
}

int fa_get_last_device_status(fa_stream_t stream) {
  DevCtl ctl;
  const int st = device_ctl(&ctl);
  if (st != FA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned v = 0;
  if (cudaMemcpyAsync(&v, ctl.status, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemsetAsync(ctl.status, 0, sizeof(unsigned), s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  if (v & kStatusTimeout) return FA_ERR_TIMEOUT;
  if (v & kStatusLaunchConfig) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

int fa_set_wait_timeout_ns(unsigned long long ns) {
  if (ns < 1000ull || ns > 100000000000ull) return FA_ERR_INVALID;
  g_timeout_ns.store(ns);
  return FA_OK;
}

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported head dimension or device";
    case FA_ERR_ALIGN: return "pointer misaligned";
    case FA_ERR_WORKSPACE: return "workspace missing or too small";
    case FA_ERR_CUDA: return "CUDA call or kernel launch failed";
    case FA_ERR_TIMEOUT: return "a bounded in-kernel wait ran out";
    default: return "unknown status";
  }
}

}  // extern "C"
