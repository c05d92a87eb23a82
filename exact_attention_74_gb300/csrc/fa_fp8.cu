// The 8-bit forward: quantisation kernels and the attention kernel launch.
#include "fa_fwd8_256_kernel.cuh"

namespace fa {

namespace {

template <int DQ>
cudaError_t launch_quant(const Fp8Launch& a, int nqb, int nkb) {
  using namespace fwd8;
  SignWords signs;
  for (int i = 0; i < 8; ++i) signs.w[i] = a.signs[i];
  constexpr int nt = QuantCfg<DQ>::kThreads;
  quant_qk_kernel<DQ><<<dim3(a.BH, nqb > nkb ? nqb : nkb, 3), nt, 0, a.stream>>>(
      static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k),
      static_cast<const __nv_bfloat16*>(a.v), a.q8, a.k8, a.qinv, a.kinv, a.vbmax, a.N_q, a.N_kv, a.hadamard,
      signs);
  quant_v_kernel<DQ><<<dim3(a.BH, nkb), nt, 0, a.stream>>>(static_cast<const __nv_bfloat16*>(a.v), a.vbmax,
                                                          a.vamax, a.v8, a.N_kv);
  return cudaGetLastError();
}

cudaError_t launch_attention_d128(const Fp8Launch& a, int nqb, int nkb) {
  using namespace fwd8;
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
  cudaError_t e = cudaFuncSetAttribute(fwd8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(p.n_qpairs) * p.BH;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  fwd8_kernel<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, a.stream>>>(a.tmQ8, a.tmK8, a.tmV8, p);
  return cudaGetLastError();
}

cudaError_t launch_attention_d256(const Fp8Launch& a, int nqb, int nkb) {
  using namespace fwd8_256;
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
  p.n_qtiles = nqb;
  p.n_steps = nkb;
  p.c0 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634 / (a.hadamard ? D : 1));
  p.tau = a.tau;
  p.ctl = a.ctl;
  cudaError_t e = cudaFuncSetAttribute(fwd8_256_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(p.n_qtiles) * p.BH;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  fwd8_256_kernel<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, a.stream>>>(a.tmQ8, a.tmK8, a.tmV8, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_fp8(const Fp8Launch& a) {
  const int nqb = (a.N_q + 127) / 128, nkb = (a.N_kv + 127) / 128;
  if (nqb > 65535 || nkb > 65535) return cudaErrorInvalidValue;
  if (a.d != 128 && a.d != 256) return cudaErrorInvalidValue;
  cudaError_t e = a.d == 128 ? launch_quant<128>(a, nqb, nkb) : launch_quant<256>(a, nqb, nkb);
  if (e != cudaSuccess) return e;
  return a.d == 128 ? launch_attention_d128(a, nqb, nkb) : launch_attention_d256(a, nqb, nkb);
}

}  // namespace fa
