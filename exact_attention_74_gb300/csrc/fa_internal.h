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
cudaError_t launch_fwd_d256(const FwdLaunch& a);   // 64-row K/V boxes

struct BwdLaunch {
  CUtensorMap tmQ, tmK, tmV, tmdO;   // same map shape as the forward's
  CUtensorMap tmDQ;                  // fp32 dQ accumulator (d, N_q, B*H), 32 x 32 x 1 boxes
  const void* o;
  const void* dO;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  float* dq_acc;      // workspace: fp32 [B*H, N_q, d]
  float* delta;       // workspace: fp32 [B*H, N_q rounded up to 128], then LSE*log2e, same shape
  unsigned* counters; // workspace: [B*H, N_q / 128 rounded up] dQ contributions applied (deterministic mode)
  int deterministic;
  int BH, N_q, N_kv, d, causal;
  int n_sms;          // multiprocessor count of the device
  float scale;
  DevCtl ctl;
  cudaStream_t stream;
};

cudaError_t launch_bwd(const BwdLaunch& a);

// Defined in fa_api.cu.
int device_ctl(DevCtl* ctl, int* n_sms = nullptr);
int make_map_bf16(CUtensorMap* m, const void* ptr, int d, int N, int BH, int box_rows = 128);
int make_map_f32(CUtensorMap* m, const void* ptr, int d, int N, int BH, int box_cols, int box_rows);

}  // namespace fa
