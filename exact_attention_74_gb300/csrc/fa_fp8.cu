// The 8-bit forward: quantisation kernels and the attention kernel launch.
#include "fa_fwd8_kernel.cuh"

namespace fa {

cudaError_t launch_fwd_fp8(const Fp8Launch& a) {
  using namespace fwd8;
  const int nqb = (a.N_q + kBM - 1) / kBM, nkb = (a.N_kv + kBN - 1) / kBN;
  if (nqb > 65535 || nkb > 65535) return cudaErrorInvalidValue;
  const uint4 signs = make_uint4(a.signs[0], a.signs[1], a.signs[2], a.signs[3]);
  quant_qk_kernel<<<dim3(a.BH, nqb > nkb ? nqb : nkb, 3), kQThreads, 0, a.stream>>>(
      static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k),
      static_cast<const __nv_bfloat16*>(a.v), a.q8, a.k8, a.qinv, a.kinv, a.vbmax, a.N_q, a.N_kv, a.hadamard,
      signs);
  quant_v_kernel<<<dim3(a.BH, nkb), kQThreads, 0, a.stream>>>(static_cast<const __nv_bfloat16*>(a.v), a.vbmax,
                                                              a.vamax, a.v8, a.N_kv);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  Params p;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.qinv = a.qinv;
  p.kinv = a.kinv;
  p.vamax = a.vamax;
  p.BH = a.BH;
  p.N_q = a.N_q;
  p.N_kv = a.N_kv;
  p.causal = a.causal;
  p.n_qpairs = (a.N_q + 2 * kBM - 1) / (2 * kBM);
  p.n_qblk = nqb;
  p.n_kv_tiles = nkb;
  p.c0 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634 / (a.hadamard ? D : 1));
  p.tau = a.tau;
  p.ctl = a.ctl;
  e = cudaFuncSetAttribute(fwd8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(p.n_qpairs) * p.BH;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  fwd8_kernel<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, a.stream>>>(a.tmQ8, a.tmK8, a.tmV8, p);
  return cudaGetLastError();
}

}  // namespace fa
