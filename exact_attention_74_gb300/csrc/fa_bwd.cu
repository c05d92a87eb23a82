// Backward kernel instances: head dimensions 64 and 128 on single CTAs (at
// d = 64 the unordered mode has a kernel of its own), and 64 on pairs of CTAs.
#include "fa_bwd_kernel.cuh"
#include "fa_bwd64_kernel.cuh"
#include "fa_bwd_pair_kernel.cuh"

namespace fa {

namespace {

// d = 64, unordered dQ reduction: prep (clearing the accumulator), the main
// pass with every intermediate in its own tensor-memory columns, convert.
cudaError_t launch_bwd64(const BwdLaunch& a) {
  constexpr int D = bwd64::D;
  const int nq_pad = (a.N_q + bwd64::kBN - 1) / bwd64::kBN * bwd64::kBN;
  float* lse2 = a.delta + static_cast<size_t>(a.BH) * nq_pad;
  {
    const long long rows = static_cast<long long>(a.BH) * nq_pad;
    const long long blocks = (rows + 8 * 4 * (256 / D) - 1) / (8 * 4 * (256 / D));
    bwd::prep_kernel<D><<<static_cast<unsigned>(blocks < 65535 * 8 ? blocks : 65535 * 8), 256, 0, a.stream>>>(
        static_cast<const __nv_bfloat16*>(a.o), static_cast<const __nv_bfloat16*>(a.dO), a.lse, lse2, a.delta,
        a.dq_acc, a.counters, a.ticket, 1, a.BH, a.N_q, nq_pad);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  bwd::Params p{};
  p.dq_acc = a.dq_acc;
  p.ticket = a.ticket;
  p.dk = static_cast<__nv_bfloat16*>(a.dk);
  p.dv = static_cast<__nv_bfloat16*>(a.dv);
  p.lse2 = lse2;
  p.delta = a.delta;
  p.counters = a.counters;
  p.deterministic = 0;
  p.BH = a.BH;
  p.N_q = a.N_q;
  p.N_kv = a.N_kv;
  p.nq_pad = nq_pad;
  p.causal = a.causal;
  p.n_q_tiles = nq_pad / bwd64::kBN;
  p.n_kv_tiles = (a.N_kv + bwd64::kBM - 1) / bwd64::kBM;
  p.c = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  p.scale = a.scale;
  p.ctl = a.ctl;
  p.n_sms = a.n_sms;
  cudaError_t e = cudaFuncSetAttribute(bwd64::main64_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       bwd64::kSmem);
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(p.n_kv_tiles) * p.BH;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  bwd64::main64_kernel<<<static_cast<unsigned>(grid), bwd64::kThreads, bwd64::kSmem, a.stream>>>(
      a.tmQ, a.tmK, a.tmV, a.tmdO, a.tmDQ, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long n8 = static_cast<long long>(a.BH) * a.N_q * D / 8;
  const long long blocks = (n8 + 255) / 256;
  bwd::convert_kernel<<<static_cast<unsigned>(blocks < 8192 ? blocks : 8192), 256, 0, a.stream>>>(
      a.dq_acc, static_cast<__nv_bfloat16*>(a.dq), n8, a.scale);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const BwdLaunch& a) {
  if (a.d == 64) return a.deterministic ? bwd::launch<64>(a) : launch_bwd64(a);
  return bwd::launch<128>(a);
}

cudaError_t launch_bwd_pair(const BwdLaunch& a) {
  constexpr int D = bwd_pair::D;
  const int nq_pad = (a.N_q + bwd_pair::kBN - 1) / bwd_pair::kBN * bwd_pair::kBN;
  float* lse2 = a.delta + static_cast<size_t>(a.BH) * nq_pad;
  {
    const long long rows = static_cast<long long>(a.BH) * nq_pad;
    const long long blocks = (rows + 8 * 4 * (256 / D) - 1) / (8 * 4 * (256 / D));
    bwd::prep_kernel<D><<<static_cast<unsigned>(blocks < 65535 * 8 ? blocks : 65535 * 8), 256, 0, a.stream>>>(
        static_cast<const __nv_bfloat16*>(a.o), static_cast<const __nv_bfloat16*>(a.dO), a.lse, lse2, a.delta,
        a.dq_acc, a.counters, a.ticket, 1, a.BH, a.N_q, nq_pad);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  bwd::Params p{};
  p.dq_acc = a.dq_acc;
  p.ticket = a.ticket;
  p.dk = static_cast<__nv_bfloat16*>(a.dk);
  p.dv = static_cast<__nv_bfloat16*>(a.dv);
  p.lse2 = lse2;
  p.delta = a.delta;
  p.counters = a.counters;
  p.deterministic = 0;
  p.BH = a.BH;
  p.N_q = a.N_q;
  p.N_kv = a.N_kv;
  p.nq_pad = nq_pad;
  p.causal = a.causal;
  p.n_q_tiles = nq_pad / bwd_pair::kBN;
  p.n_kv_tiles = (a.N_kv + bwd_pair::kBM - 1) / bwd_pair::kBM;
  p.c = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  p.scale = a.scale;
  p.ctl = a.ctl;
  p.n_sms = a.n_sms;
  cudaError_t e = cudaFuncSetAttribute(bwd_pair::pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       bwd_pair::kSmem);
  if (e != cudaSuccess) return e;
  // two CTAs (one cluster) per 256 keys of every (batch, head)
  const long long grid = 2LL * ((p.n_kv_tiles + 1) / 2) * p.BH;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  bwd_pair::pair_kernel<<<static_cast<unsigned>(grid), bwd_pair::kThreads, bwd_pair::kSmem, a.stream>>>(
      a.tmK, a.tmV, a.tmKc, a.tmQh, a.tmQc, a.tmdOh, a.tmdOc, a.tmDQ, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long n8 = static_cast<long long>(a.BH) * a.N_q * D / 8;
  const long long blocks = (n8 + 255) / 256;
  bwd::convert_kernel<<<static_cast<unsigned>(blocks < 8192 ? blocks : 8192), 256, 0, a.stream>>>(
      a.dq_acc, static_cast<__nv_bfloat16*>(a.dq), n8, a.scale);
  return cudaGetLastError();
}

}  // namespace fa
