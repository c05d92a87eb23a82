// fa_fwd8_kernel.cuh -- the 8-bit forward (d = 128): quantisation kernels and
// the attention kernel on e4m3 operands.
//
// "FlashAttention-3: Fast and Accurate Attention with Asynchrony and
// Low-precision" 技術 3: Q, K and V are held in 8-bit floating point with one
// scale per block, and Q and K are first multiplied by one random orthogonal
// matrix D H (D random signs, H the Hadamard matrix), which leaves Q K^T
// unchanged and spreads outlier channels ("incoherent processing").  Here:
//
//   quant_qk_kernel  one 128-row block of Q or K per CTA (d / 32 threads per
//                    row): negate the channels whose sign bit is set, the
//                    Hadamard butterfly (stages 1, 2, ..., d / 2, fp32,
//                    unnormalised, so the logit scale is divided by d), the
//                    block's largest magnitude amax, multiplier
//                    inv = 448 / amax, codes e4m3(x * inv) (nearest even,
//                    saturating); in the same launch, each block of V's
//                    largest |V|
//   quant_v_kernel   V's codes with its (batch, head)'s multiplier, rows in
//                    place ([B*H, keys, d]: the MN-major operand of P V)
//   fwd8_kernel      the d = 128 forward of fa_fwd_kernel.cuh on e4m3 tiles
//                    (16 KB each): kind::f8f6f4 products, S scaled by
//                    c = scale log2(e) / (inv_q inv_k) per key tile, P rounded
//                    to e4m3 (P <= 2^tau <= 448) into tensor memory (four per
//                    column), O divided by inv_v at the end
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "exp2.cuh"
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace fwd8 {

constexpr int D = 128;
constexpr int kBM = 128;               // query rows per tile
constexpr int kBN = 128;               // keys per tile
constexpr int kThreads = 320;          // 10 warps
constexpr int kTileBytes = 128 * 128;  // one 128-row x 128-byte swizzle panel
constexpr int kSlots = 8;
constexpr int kQOff = 0;
constexpr int kKVOff = 2 * kTileBytes;
constexpr int kBarOff = kKVOff + kSlots * kTileBytes;
// barrier indices
constexpr int kQFull = 0;              // 2
constexpr int kKVFull = 2;             // kSlots
constexpr int kKVEmpty = 2 + kSlots;   // kSlots
constexpr int kSFull = 2 + 2 * kSlots; // 2
constexpr int kPFull = 4 + 2 * kSlots; // 2
constexpr int kOFull = 6 + 2 * kSlots; // 2
constexpr int kNumBars = 8 + 2 * kSlots;
constexpr int kMiscOff = kBarOff + 8 * kNumBars;
constexpr int kSmemBytes = kMiscOff + 16 + 1024;
__device__ constexpr uint32_t col_S(int t) { return 128u * t; }
__device__ constexpr uint32_t col_O(int t) { return 256u + 128u * t; }
constexpr uint32_t kTmemCols = 512;

// ------------------------------------------------------------ quantisation
//
// One CTA per 128-row block, d / 32 threads per row: thread (row r, group q)
// holds channels 32q .. 32q + 31, so a warp loads and stores whole rows.  The
// Hadamard stages h = 1 .. 16 stay inside a thread; h = 32, 64, 128 pair a
// thread with lane ^ 1, ^ 2, ^ 4 (the threads of one row are adjacent lanes).
constexpr int kQCh = 32;               // channels per thread

template <int DQ>
struct QuantCfg {
  static constexpr int kPerRow = DQ / kQCh;          // threads per row
  static constexpr int kThreads = kBM * kPerRow;     // 512 at d = 128, 1024 at d = 256
};

// Sign bits of the incoherent processing: bit c % 32 of word c / 32 negates
// channel c (d / 32 words used).
struct SignWords {
  uint32_t w[8];
};

// Largest value of v over the NT threads of the block (all threads get it).
template <int NT>
__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  v = red[0];
#pragma unroll
  for (int w = 1; w < NT / 32; ++w) v = fmaxf(v, red[w]);
  __syncthreads();
  return v;
}

__device__ __forceinline__ float e4m3_multiplier(float amax) {
  return amax > 0.f ? __fdiv_rn(448.f, amax) : 1.f;
}

// This thread's 32 channels of a row as fp32 (zeros when !valid).
__device__ __forceinline__ void load_group(const __nv_bfloat16* row, bool valid, float (&x)[kQCh]) {
#pragma unroll
  for (int i = 0; i < kQCh / 8; ++i) {
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (valid) w = reinterpret_cast<const uint4*>(row)[i];
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[8 * i + 2 * e] = __uint_as_float(ws[e] << 16);
      x[8 * i + 2 * e + 1] = __uint_as_float(ws[e] & 0xffff0000u);
    }
  }
}

__device__ __forceinline__ float max_abs(const float (&x)[kQCh]) {
  float m0 = 0.f, m1 = 0.f;
#pragma unroll
  for (int c = 0; c < kQCh; c += 4) {
    m0 = max3(m0, fabsf(x[c]), fabsf(x[c + 1]));
    m1 = max3(m1, fabsf(x[c + 2]), fabsf(x[c + 3]));
  }
  return fmaxf(m0, m1);
}

// Codes of x * inv (each product rounded once, as __fmul_rn), stored as 32
// bytes at dst (16-byte aligned).
__device__ __forceinline__ void store_codes(uint8_t* dst, const float (&x)[kQCh], float inv, bool valid) {
  uint32_t w[kQCh / 4];
  const float2 inv2 = make_float2(inv, inv);
#pragma unroll
  for (int i = 0; i < kQCh / 4; ++i) {
    const float2 a = mul2(make_float2(x[4 * i], x[4 * i + 1]), inv2);
    const float2 b = mul2(make_float2(x[4 * i + 2], x[4 * i + 3]), inv2);
    w[i] = valid ? pack_e4m3x4(a.x, a.y, b.x, b.y) : 0u;     // rows past N: +0 codes
  }
  uint4* d = reinterpret_cast<uint4*>(dst);
  d[0] = make_uint4(w[0], w[1], w[2], w[3]);
  d[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// grid (B*H, blocks, 3): z = 0 quantises a block of Q, z = 1 of K (after
// the sign flips and the Hadamard transform when hadamard != 0); z = 2
// writes the largest |V| of a block of V to vbmax.  Rows past N count as
// zeros.
template <int DQ>
__global__ void __launch_bounds__(QuantCfg<DQ>::kThreads)
quant_qk_kernel(const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ K,
                const __nv_bfloat16* __restrict__ V, uint8_t* __restrict__ Q8, uint8_t* __restrict__ K8,
                float* __restrict__ qinv, float* __restrict__ kinv, float* __restrict__ vbmax, int N_q,
                int N_kv, int hadamard, SignWords signs) {
  using QC = QuantCfg<DQ>;
  __shared__ float red[QC::kThreads / 32];
  const int z = blockIdx.z;
  const int N = z == 0 ? N_q : N_kv;
  const int nblk = (N + kBM - 1) / kBM;
  const int blk = blockIdx.y;
  if (blk >= nblk) return;                              // uniform over the block
  const int bh = blockIdx.x;
  const int q = threadIdx.x % QC::kPerRow;
  const int r = blk * kBM + threadIdx.x / QC::kPerRow;
  const bool valid = r < N;
  const __nv_bfloat16* src = z == 0 ? Q : z == 1 ? K : V;
  float x[kQCh];
  load_group(src + (static_cast<size_t>(bh) * N + r) * DQ + kQCh * q, valid, x);
  if (z == 2) {
    const float m = block_max<QC::kThreads>(max_abs(x), red);
    if (threadIdx.x == 0) vbmax[static_cast<size_t>(bh) * nblk + blk] = m;
    return;
  }
  if (hadamard) {
    const uint32_t sw = signs.w[q];
#pragma unroll
    for (int c = 0; c < kQCh; ++c)
      if ((sw >> c) & 1u) x[c] = -x[c];
    // stage h = 1: (a, b) -> (a + b, a - b), each rounded once
#pragma unroll
    for (int i = 0; i < kQCh; i += 2) {
      const float a = x[i], b = x[i + 1];
      x[i] = __fadd_rn(a, b);
      x[i + 1] = __fsub_rn(a, b);
    }
    // stages h = 2 .. 16: two neighbouring butterflies per packed pair of
    // operations; fma(-1, b, a) is a - b rounded once
    const float2 neg1 = make_float2(-1.f, -1.f);
#pragma unroll
    for (int h = 2; h < kQCh; h *= 2) {
#pragma unroll
      for (int i = 0; i < kQCh; i += 2) {
        if (i & h) continue;
        const float2 a = make_float2(x[i], x[i + 1]), b = make_float2(x[i + h], x[i + h + 1]);
        const float2 sum = add2(a, b), dif = fma2(neg1, b, a);
        x[i] = sum.x;
        x[i + 1] = sum.y;
        x[i + h] = dif.x;
        x[i + h + 1] = dif.y;
      }
    }
    // stages h = 32 s across lanes: the lower thread of a pair keeps x + y,
    // the upper y - x, both as fma(+-1, x, y) rounded once
#pragma unroll
    for (int s = 1; s < QC::kPerRow; s <<= 1) {
      const float sg = (q & s) == 0 ? 1.f : -1.f;
      const float2 sg2 = make_float2(sg, sg);
#pragma unroll
      for (int c = 0; c < kQCh; c += 2) {
        const float2 y = make_float2(__shfl_xor_sync(0xffffffffu, x[c], s),
                                     __shfl_xor_sync(0xffffffffu, x[c + 1], s));
        const float2 r = fma2(sg2, make_float2(x[c], x[c + 1]), y);
        x[c] = r.x;
        x[c + 1] = r.y;
      }
    }
  }
  const float inv = e4m3_multiplier(block_max<QC::kThreads>(max_abs(x), red));
  const size_t npad = static_cast<size_t>(nblk) * kBM;
  store_codes((z == 1 ? K8 : Q8) + (static_cast<size_t>(bh) * npad + r) * DQ + kQCh * q, x, inv, valid);
  if (threadIdx.x == 0) (z == 1 ? kinv : qinv)[static_cast<size_t>(bh) * nblk + blk] = inv;
}

// grid (B*H, key blocks): V's codes with its head's multiplier 448 / max|V|
// (the maximum of the head's block maxima), rows in place ([B*H, keys padded
// to 128, d]); block 0 also stores that maximum in vamax for the epilogue.
template <int DQ>
__global__ void __launch_bounds__(QuantCfg<DQ>::kThreads)
quant_v_kernel(const __nv_bfloat16* __restrict__ V, const float* __restrict__ vbmax,
               float* __restrict__ vamax, uint8_t* __restrict__ V8, int N_kv) {
  using QC = QuantCfg<DQ>;
  __shared__ float red[QC::kThreads / 32];
  const int bh = blockIdx.x;
  const int nblk = gridDim.y;
  float m = 0.f;
  for (int i = threadIdx.x; i < nblk; i += QC::kThreads) m = fmaxf(m, vbmax[static_cast<size_t>(bh) * nblk + i]);
  m = block_max<QC::kThreads>(m, red);
  if (blockIdx.y == 0 && threadIdx.x == 0) vamax[bh] = m;
  const int q = threadIdx.x % QC::kPerRow;
  const int r = blockIdx.y * kBN + threadIdx.x / QC::kPerRow;
  const bool valid = r < N_kv;
  float x[kQCh];
  load_group(V + (static_cast<size_t>(bh) * N_kv + r) * DQ + kQCh * q, valid, x);
  const size_t npad = static_cast<size_t>(nblk) * kBN;
  store_codes(V8 + (static_cast<size_t>(bh) * npad + r) * DQ + kQCh * q, x, e4m3_multiplier(m), valid);
}

// ----------------------------------------------------------------- forward

struct Params {
  __nv_bfloat16* o;
  float* lse;
  const float* qinv;       // [B*H, q blocks]
  const float* kinv;       // [B*H, key blocks]
  const float* vamax;      // [B*H] largest |V|
  int BH, N_q, N_kv, causal;
  int n_qpairs, n_qblk, n_kv_tiles;
  float c0;                // scale * log2(e) (/ 128 with the Hadamard transform)
  float tau;
  DevCtl ctl;
};

__device__ __forceinline__ int tiles_for(const Params& p, int qbase) {
  if (qbase >= p.N_q) return 0;
  if (!p.causal) return p.n_kv_tiles;
  return min(p.n_kv_tiles, qbase / kBN + 1);
}

// x rounded to e4m3 as the P V product consumes it
__device__ __forceinline__ float e4m3_value(float x) {
  const uint32_t code = pack_e4m3x4(x, 0.f, 0.f, 0.f) & 0xffu;
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(code)));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xffffu)));
}

__global__ void __launch_bounds__(kThreads, 1)
fwd8_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
            const __grid_constant__ CUtensorMap tmV, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + kBarOff + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMiscOff + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  int pair, bh;
  if (p.causal) {
    pair = p.n_qpairs - 1 - static_cast<int>(blockIdx.x) / p.BH;
    bh = static_cast<int>(blockIdx.x) % p.BH;
  } else {
    pair = static_cast<int>(blockIdx.x) % p.n_qpairs;
    bh = static_cast<int>(blockIdx.x) / p.n_qpairs;
  }
  const int qbase0 = pair * 2 * kBM;
  const int n_t[2] = {tiles_for(p, qbase0), tiles_for(p, qbase0 + kBM)};
  const int n_max = max(n_t[0], n_t[1]);

  if (threadIdx.x == 0) {
    mbar_init(bar(kQFull + 0), 1);
    mbar_init(bar(kQFull + 1), 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(bar(kKVFull + s), 1);
      mbar_init(bar(kKVEmpty + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(kSFull + t), 1);
      mbar_init(bar(kPFull + t), 4);       // one arrive per softmax warp
      mbar_init(bar(kOFull + t), 1);
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  __syncwarp();   // warps whose lane 0 ran a role alone arrive whole
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmV);
      for (int t = 0; t < 2; ++t) {
        if (n_t[t] == 0) continue;
        mbar_arrive_expect_tx(bar(kQFull + t), kTileBytes);
        tma_load_3d(sb + kQOff + t * kTileBytes, &tmQ, bar(kQFull + t), 0, qbase0 + t * kBM, bh);
      }
      const uint64_t keep = l2_policy_evict_last();
      int slot = 0;
      uint32_t ph = 0;
      for (int j = 0; j < n_max; ++j) {
        for (int kind = 0; kind < 2; ++kind) {
          if (!mbar_wait(bar(kKVEmpty + slot), ph ^ 1, p.ctl, abort_flag)) goto producer_done;
          const uint32_t dst = sb + kKVOff + slot * kTileBytes;
          mbar_arrive_expect_tx(bar(kKVFull + slot), kTileBytes);
          tma_load_3d_hint(dst, kind == 0 ? &tmK : &tmV, bar(kKVFull + slot), 0, j * kBN, bh, keep);
          if (++slot == kSlots) { slot = 0; ph ^= 1; }
        }
      }
    producer_done:;
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_e4m3(kBM, kBN);           // S = Q K^T, both K-major
      constexpr uint32_t idesc_pv = idesc_e4m3(kBM, D, true);    // O += P V, V MN-major
      auto issue_S = [&](int t, int kslot, auto&& peek) {
        const uint32_t qa = sb + kQOff + t * kTileBytes;
        const uint32_t ka = sb + kKVOff + kslot * kTileBytes;
#pragma unroll
        for (int k = 0; k < D / 32; ++k) {
          mma_ss_f8(tmem + col_S(t), sdesc_sw128(qa + 32 * k, 0, 1024), sdesc_sw128(ka + 32 * k, 0, 1024), idesc,
                    k > 0 ? 1u : 0u);
          if (k == D / 32 - 2) peek();
        }
      };
      auto issue_PV = [&](int t, int vslot, bool acc) {
        const uint32_t va = sb + kKVOff + vslot * kTileBytes;
#pragma unroll
        for (int k = 0; k < kBN / 32; ++k)
          // 32 keys = 32 rows of 128 bytes per product; the tile is one
          // 128-byte panel wide, so both offsets are the 8-row stride
          mma_ts_f8(tmem + col_O(t), tmem + col_S(t) + 8 * k, sdesc_sw128(va + 4096 * k, 1024, 1024), idesc_pv,
                    (acc || k > 0) ? 1u : 0u);
      };
      // K_j and V_j are ring loads 2j and 2j+1; the softmax warps release them
      auto kv_bar = [](int i) { return kKVFull + i % kSlots; };
      auto kv_par = [](int i) { return static_cast<uint32_t>((i / kSlots) & 1); };
      bool ok = true;
      uint32_t pph[2] = {0, 0};
      for (int t = 0; t < 2 && ok; ++t)
        if (n_t[t] > 0) ok = mbar_wait(bar(kQFull + t), 0, p.ctl, abort_flag);
      if (ok) ok = mbar_wait(bar(kv_bar(0)), kv_par(0), p.ctl, abort_flag);
      if (ok) {
        tc_fence_after();
        for (int t = 0; t < 2; ++t)
          if (n_t[t] > 0) { issue_S(t, 0, [] {}); tc_commit(bar(kSFull + t)); }
      }
      bool kv_ready = false, p_ready[2] = {false, false};
      for (int j = 0; j < n_max && ok; ++j) {
        const int iv = 2 * j + 1, ik = 2 * j + 2;
        if (!kv_ready) {
          ok = mbar_wait(bar(kv_bar(iv)), kv_par(iv), p.ctl, abort_flag);
          if (ok && j + 1 < n_max) ok = mbar_wait(bar(kv_bar(ik)), kv_par(ik), p.ctl, abort_flag);
          if (!ok) break;
        }
        kv_ready = false;
        for (int t = 0; t < 2 && ok; ++t) {
          if (j >= n_t[t]) continue;
          if (!p_ready[t]) ok = mbar_wait(bar(kPFull + t), pph[t], p.ctl, abort_flag);
          pph[t] ^= 1;
          p_ready[t] = false;
          if (!ok) break;
          tc_fence_after();
          issue_PV(t, iv % kSlots, j > 0);
          if (j + 1 < n_t[t]) {
            if (t == 0) {
              issue_S(0, ik % kSlots, [&] {
                if (j < n_t[1]) p_ready[1] = mbar_test_wait(bar(kPFull + 1), pph[1]);
              });
            } else {
              issue_S(1, ik % kSlots, [&] {
                const int iv2 = iv + 2, ik2 = ik + 2;
                const bool a = mbar_test_wait(bar(kv_bar(iv2)), kv_par(iv2));
                const bool b = ik2 >= 2 * n_max || mbar_test_wait(bar(kv_bar(ik2)), kv_par(ik2));
                const bool c = j + 1 >= n_t[0] || mbar_test_wait(bar(kPFull + 0), pph[0]);
                kv_ready = a && b;
                p_ready[0] = c && j + 1 < n_t[0];
              });
            }
            tc_commit(bar(kSFull + t));
          } else {
            tc_commit(bar(kOFull + t));
          }
        }
      }
    }
  } else {
    // -------------------------------------------------------------- softmax
    const int t = (warp - 2) >> 2;
    const int rank = warp & 3;
    const int r_in_tile = rank * 32 + lane;
    const int row = qbase0 + t * kBM + r_in_tile;
    const int nt = n_t[t];
    const uint32_t lane_addr = static_cast<uint32_t>(rank * 32) << 16;
    const uint32_t tS = tmem + lane_addr + col_S(t);
    const uint32_t tO = tmem + lane_addr + col_O(t);
    const bool releaser = t == (n_t[1] > 0 ? 1 : 0);
    const int qblk = (qbase0 + t * kBM) / kBM;
    const float cq = nt > 0 ? p.c0 / p.qinv[static_cast<size_t>(bh) * p.n_qblk + qblk] : 0.f;
    const float* kinv = p.kinv + static_cast<size_t>(bh) * p.n_kv_tiles;
    float kinv_next = nt > 0 ? kinv[0] : 1.f;
    float m_ref = -INFINITY;
    float l = 0.f;
    float lr = 0.f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      const float c = cq / kinv_next;          // this key tile's logit scale
      if (j + 1 < nt) kinv_next = kinv[j + 1];
      ok = __all_sync(0xffffffffu, mbar_wait(bar(kSFull + t), j & 1, p.ctl, abort_flag));
      if (!ok) break;
      if (releaser && r_in_tile == 0) {
        mbar_arrive(bar(kKVEmpty + (2 * j) % kSlots));
        if (j > 0) mbar_arrive(bar(kKVEmpty + (2 * j - 1) % kSlots));
      }
      tc_fence_after();
      uint32_t s[128];
      tmem_ld_x128(tS, s);
      if (j == nt - 1) {
        int lim = p.N_kv - 1 - j * kBN;
        if (p.causal) lim = min(lim, row - j * kBN);
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (i > lim) s[i] = __float_as_uint(-INFINITY);
      }
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int i = 0; i < 128; i += 8) {
        mx[0] = max3(mx[0], __uint_as_float(s[i + 0]), __uint_as_float(s[i + 1]));
        mx[1] = max3(mx[1], __uint_as_float(s[i + 2]), __uint_as_float(s[i + 3]));
        mx[2] = max3(mx[2], __uint_as_float(s[i + 4]), __uint_as_float(s[i + 5]));
        mx[3] = max3(mx[3], __uint_as_float(s[i + 6]), __uint_as_float(s[i + 7]));
      }
      const float mxs = fmaxf(max3(mx[0], mx[1], mx[2]), mx[3]);
      const float m_blk = c * mxs;
      const float m_new = fmaxf(m_ref, m_blk);
      bool resc = false;
      float alpha = 1.f;
      if (j == 0) {
        m_ref = m_new;
      } else if (m_new - m_ref > p.tau) {
        resc = true;
        alpha = ex2_hw(m_ref - m_new);
        l *= alpha;
        lr *= alpha;
        m_ref = m_new;
      }
      if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t o[32];
          tmem_ld_x32(tO + 32 * ch, o);
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 r = mul2(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])),
                                  make_float2(alpha, alpha));
            o[i] = __float_as_uint(r.x);
            o[i + 1] = __float_as_uint(r.y);
          }
          tmem_st_x32(tO + 32 * ch, o);
        }
      }
      const float2 c2 = make_float2(c, c);
      const float2 neg2 = make_float2(-m_ref, -m_ref);
      float2 sum[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float2 x0 = fma2(make_float2(__uint_as_float(s[4 * i]), __uint_as_float(s[4 * i + 1])), c2, neg2);
        const float2 x1 = fma2(make_float2(__uint_as_float(s[4 * i + 2]), __uint_as_float(s[4 * i + 3])), c2, neg2);
        const float e0 = ex2_hw(x0.x), e1 = ex2_hw(x0.y), e2 = ex2_hw(x1.x), e3 = ex2_hw(x1.y);
        sum[i & 1] = add2(sum[i & 1], make_float2(e0 + e2, e1 + e3));
        pk[i] = pack_e4m3x4(e0, e1, e2, e3);
      }
      tmem_st_x32(tS, pk);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kPFull + t));
      l += (sum[0].x + sum[0].y) + (sum[1].x + sum[1].y);
      {
        const float pm = ex2_hw(fmaf(mxs, c, -m_ref));   // the block's largest P
        lr += e4m3_value(pm) - pm;                      // as rounded for P V
      }
    }
    // ------------------------------------------------------------- epilogue
    bool ready = ok && nt > 0;
    if (ready) ready = mbar_wait(bar(kOFull + t), 0, p.ctl, abort_flag);
    if (__all_sync(0xffffffffu, ready)) {
      tc_fence_after();
      const float vinv = e4m3_multiplier(p.vamax[bh]);
      const float inv_l = 1.f / ((l + lr) * vinv);
      __nv_bfloat16* orow = p.o + (static_cast<size_t>(bh) * p.N_q + row) * D;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t o[32];
        tmem_ld_x32(tO + 32 * ch, o);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
        if (row < p.N_q) {
          uint4* dst = reinterpret_cast<uint4*>(orow + 32 * ch);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
      if (row < p.N_q)
        p.lse[static_cast<size_t>(bh) * p.N_q + row] = (m_ref + log2f(l)) * 0.69314718055994531f;
    }
  }

  __syncwarp();   // warps whose lane 0 ran a role alone arrive whole
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace fwd8
}  // namespace fa
