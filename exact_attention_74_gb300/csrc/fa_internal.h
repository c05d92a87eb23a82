// fa_internal.h -- host-side interface between the C-ABI layer (fa_api.cu)
// and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace fa {

struct FwdLaunch {
  CUtensorMap tmQ, tmK, tmV;   // 3-D maps (d, N, B*H), 64 x 128 x 1 boxes (K, V: 64 x 64 at d = 256),
                               // 128 B swizzle
  CUtensorMap tmO;             // O (d, N_q, B*H), 64 x 32 x 1 boxes, 128 B swizzle (d = 64, 128 stores)
  void* o;
  float* lse;
  int BH, N_q, N_kv, d, causal;
  float scale;
  float tau;                   // log2 units
  int emu_per_32;              // 0, 8 or 16
  DevCtl ctl;
  cudaStream_t stream;
};

cudaError_t launch_fwd_d64(const FwdLaunch& a);
cudaError_t launch_fwd_d128(const FwdLaunch& a);
cudaError_t launch_fwd_d256(const FwdLaunch& a);   // 64-row K boxes, pairs of CTAs

struct BwdLaunch {
  CUtensorMap tmQ, tmK, tmV, tmdO;   // same map shape as the forward's
  CUtensorMap tmDQ;                  // fp32 dQ accumulator (d, N_q, B*H), 32 x 32 x 1 boxes
  // pair kernel only (d = 64): Q and dO in 64-row boxes (128-byte swizzle),
  // Q, dO and K in 32-column boxes of 128 rows (64-byte swizzle)
  CUtensorMap tmQh, tmdOh, tmQc, tmdOc, tmKc;
  const void* o;
  const void* dO;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  float* dq_acc;      // workspace: fp32 [B*H, N_q, d]
  float* delta;       // workspace: fp32 [B*H, N_q rounded up to 128], then LSE*log2e, same shape
  unsigned* counters; // workspace: [B*H, N_q / 128 rounded up] dQ contributions applied (deterministic mode)
  unsigned* ticket;   // workspace: one word, the next CTA ticket
  int deterministic;
  int BH, N_q, N_kv, d, causal;
  int n_sms;          // multiprocessor count of the device
  float scale;
  DevCtl ctl;
  cudaStream_t stream;
};

cudaError_t launch_bwd(const BwdLaunch& a);
// The backward at d = 64 on pairs of CTAs sharing 256-key products.
cudaError_t launch_bwd_pair(const BwdLaunch& a);

// The 8-bit forward (d = 128): quantisation into the workspace, then the
// attention kernel on the e4m3 copies.
struct Fp8Launch {
  CUtensorMap tmQ8, tmK8, tmV8;     // u8 maps, 128 x 128 x 1 boxes, 128 B swizzle
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  uint8_t* q8;        // [B*H, N_q padded to 128, d]
  uint8_t* k8;        // [B*H, N_kv padded to 128, d]
  uint8_t* v8;        // [B*H, N_kv padded to 128, d]
  float* qinv;        // [B*H, N_q blocks]
  float* kinv;        // [B*H, N_kv blocks]
  float* vbmax;       // [B*H, N_kv blocks] largest |V| of each block
  float* vamax;       // [B*H] largest |V| of each (batch, head)
  int BH, N_q, N_kv, d, causal, hadamard;   // d: 128 or 256
  unsigned signs[8];                         // d / 32 words used
  float scale, tau;
  DevCtl ctl;
  cudaStream_t stream;
};

cudaError_t launch_fwd_fp8(const Fp8Launch& a);

// Defined in fa_api.cu.
int device_ctl(DevCtl* ctl, int* n_sms = nullptr);
// The backward entry point's checks and launches; pair = the kernel on pairs
// of CTAs (d = 64 only); internal_workspace = the library's own scratch array
// (not checked as a caller allocation).
int bwd_entry(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE,
              void* dQ, void* dK, void* dV, int B, int H, int N_q, int N_kv, int d, int causal, float scale,
              int deterministic, bool pair, void* workspace, size_t workspace_bytes, bool internal_workspace,
              cudaStream_t stream);
int make_map_bf16(CUtensorMap* m, const void* ptr, int d, int N, int BH, int box_rows = 128);
// Same tensor, 32-column x box_rows boxes with 64-byte swizzle.
int make_map_bf16_sw64(CUtensorMap* m, const void* ptr, int d, int N, int BH, int box_rows);
int make_map_f32(CUtensorMap* m, const void* ptr, int d, int N, int BH, int box_cols, int box_rows);
// 3-D map over a contiguous u8 [BH, rows, inner] tensor, 128 x 128 x 1 boxes, 128-byte swizzle.
int make_map_u8(CUtensorMap* m, const void* ptr, int inner, int rows, int BH);

}  // namespace fa
