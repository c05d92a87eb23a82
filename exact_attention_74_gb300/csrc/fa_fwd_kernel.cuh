// fa_fwd_kernel.cuh -- forward exact attention for sm_103a.
//
// One CTA computes two 128-row query tiles of one (batch, head) against the
// whole key sequence (or, causal, the keys up to its last query row):
//
//   warp 0       TMA producer: Q tiles once, then K_j, V_j into a ring of
//                shared-memory slots (mbarrier full/empty pairs).
//   warp 1       MMA issuer (one thread): S_t = Q_t K_j^T into tensor memory,
//                O_t += P_t V_j with P_t read from tensor memory, in the order
//                S0 S1 | PV0 S0' PV1 S1' | ... so that the tensor core works
//                on one tile while the softmax of the other runs.  The
//                tensor core's queue is only a couple of products deep and
//                every barrier operation of this thread is a shared-memory
//                round trip against the operand reads, so between two groups
//                it does one commit and the waits only, and tests the next
//                group's barriers while it is still queueing the current one.
//   warps 2-9    softmax of tile 0 (warps 2-5) and tile 1 (6-9); one thread
//                owns one query row (one tensor-memory lane).  They also hand
//                the K/V slots back to the producer: S_t,j complete implies
//                every earlier product is complete.
//
// The per-row recurrence is the online softmax of "FlashAttention: GPUメモリ
// 階層を活用したアテンション最適化の分析" §6.2 in base 2 (t = scale*log2e*s),
// with the conditional rescaling of "論文解説: FlashAttention-4 — Algorithm and
// Kernel Pipelining Co-Design for Asymmetric Hardware Scaling"
// (条件付きオンラインsoftmaxリスケーリング): the row keeps a reference maximum
// m_ref and P = 2^(t - m_ref); O and l are rescaled by 2^(m_ref - m_new) only
// when the row maximum rises more than tau above m_ref.  Normalisation is
// deferred to the epilogue (§8.1 of the first page), which also writes
// LSE = ln2 * (m_ref + log2 l), with l the sum of the fp32 probabilities.
// O is divided by l plus the bf16 rounding residual of each block's largest
// P (as the P V product consumes it): with tau > 0 that largest P (up to
// 2^tau) is not a power of two, and in near-one-hot rows its rounding would
// otherwise show in O undamped; the residuals of the other, smaller
// probabilities average out like any bf16 rounding of P.  A query tile whose
// rows see at most one key tile (the first tile of a causal grid, or
// N_kv <= 128) has few keys per row, where rounding a couple of comparable
// probabilities to bf16 (2^-8 relative each) moves O by up to 2^-8 |v|: that
// tile's single step writes P in two bf16 parts instead, hi = bf16(P) over S
// columns [0, 64) and lo = bf16(P - hi) over the dead columns [64, 128), and
// P V is two products, so that P is carried to ~2^-16 (this path is kept out
// of the main loop).  Some of the exponentials take the FMA-pipe cubic
// emulation (ソフトウェア指数関数エミュレーション) instead of MUFU.
//
// Causal masking skips every key tile that lies wholly above the diagonal;
// only the last key tile of each query tile needs an element mask (it holds
// both the diagonal and the N_kv tail).  Rows past N_q and keys past N_kv are
// zero-filled by TMA and never stored / masked out.
#pragma once

#include <cuda_bf16.h>

#include <type_traits>

#include "exp2.cuh"
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace fwd {

constexpr int kBM = 128;          // query rows per tile
constexpr int kBN = 128;          // keys per tile
constexpr int kThreads = 320;     // 10 warps
constexpr int kPanelBytes = 128 * 128;   // 128 rows x 128 B (64 bf16) swizzle panel

template <int D>
struct Cfg {
  static constexpr int kPanels = D / 64;
  static constexpr int kTileBytes = kBM * D * 2;
  static constexpr int kSlots = (D == 128) ? 4 : 8;
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = 2 * kTileBytes;
  static constexpr int kBarOff = kKVOff + kSlots * kTileBytes;
  // barrier indices
  static constexpr int kQFull = 0;                 // 2
  static constexpr int kKVFull = 2;                // kSlots
  static constexpr int kKVEmpty = 2 + kSlots;      // kSlots
  static constexpr int kSFull = 2 + 2 * kSlots;    // 2
  static constexpr int kPFull = 4 + 2 * kSlots;    // 2
  static constexpr int kOFull = 6 + 2 * kSlots;    // 2
  static constexpr int kNumBars = 8 + 2 * kSlots;
  static constexpr int kMiscOff = kBarOff + 8 * kNumBars;   // tmem base, abort flag
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;   // + base alignment slack
  // tensor-memory columns
  __device__ static constexpr uint32_t col_S(int t) { return 128u * t; }
  __device__ static constexpr uint32_t col_O(int t) { return 256u + static_cast<uint32_t>(D) * t; }
  static constexpr uint32_t kTmemCols = 512;
};

struct Params {
  __nv_bfloat16* o;
  float* lse;
  int BH, N_q, N_kv, causal;
  int n_qpairs;       // ceil(N_q / 256)
  int n_kv_tiles;     // ceil(N_kv / 128)
  float c;            // scale * log2(e)
  float tau;          // log2 units
  DevCtl ctl;
};

__device__ __forceinline__ int tiles_for(const Params& p, int qbase) {
  if (qbase >= p.N_q) return 0;
  if (!p.causal) return p.n_kv_tiles;
  return min(p.n_kv_tiles, qbase / kBN + 1);
}

template <int EMU>
__device__ __forceinline__ float ex2_mix(float x, int col) {
  if ((col & 31) < EMU) return ex2_poly3(x);
  return ex2_hw(x);
}

// SPLIT: the grid may hold query tiles whose rows see one key tile (causal,
// or N_kv <= 128), which take the two-part P path; grids without such tiles
// run an instance that carries none of its code.
template <int D, int EMU, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
           const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO, const Params p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + C::kBarOff + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work tile: a pair of query tiles of one (batch, head).  Causal grids run
  // the heaviest pairs (the last query rows) first.
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
    mbar_init(bar(C::kQFull + 0), 1);
    mbar_init(bar(C::kQFull + 1), 1);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(bar(C::kKVFull + s), 1);
      mbar_init(bar(C::kKVEmpty + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(C::kSFull + t), 1);
      mbar_init(bar(C::kPFull + t), 4);     // one arrive per softmax warp
      mbar_init(bar(C::kOFull + t), 1);
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
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
        const uint32_t dst = sb + C::kQOff + t * C::kTileBytes;
        mbar_arrive_expect_tx(bar(C::kQFull + t), C::kTileBytes);
        for (int pn = 0; pn < C::kPanels; ++pn)
          tma_load_3d(dst + pn * kPanelBytes, &tmQ, bar(C::kQFull + t), pn * 64, qbase0 + t * kBM, bh);
      }
      const uint64_t keep = l2_policy_evict_last();
      int slot = 0;
      uint32_t ph = 0;
      for (int j = 0; j < n_max; ++j) {
        for (int kind = 0; kind < 2; ++kind) {
          if (!mbar_wait(bar(C::kKVEmpty + slot), ph ^ 1, p.ctl, abort_flag)) goto producer_done;
          const uint32_t dst = sb + C::kKVOff + slot * C::kTileBytes;
          mbar_arrive_expect_tx(bar(C::kKVFull + slot), C::kTileBytes);
          for (int pn = 0; pn < C::kPanels; ++pn)
            tma_load_3d_hint(dst + pn * kPanelBytes, kind == 0 ? &tmK : &tmV, bar(C::kKVFull + slot),
                             pn * 64, j * kBN, bh, keep);
          if (++slot == C::kSlots) { slot = 0; ph ^= 1; }
        }
      }
    producer_done:;
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16(kBM, kBN, false, false);
      constexpr uint32_t idO = idesc_bf16(kBM, D, false, true);
      // S_t = Q_t K^T; after the sixth of its eight products (while the
      // issue stalls on the tensor core's queue) run `peek`, which tests the
      // barriers the next group waits on.
      auto issue_S = [&](int t, int kslot, auto&& peek) {
        const uint32_t qa = sb + C::kQOff + t * C::kTileBytes;
        const uint32_t ka = sb + C::kKVOff + kslot * C::kTileBytes;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * kPanelBytes + (k & 3) * 32;
          mma_ss(tmem + C::col_S(t), sdesc_sw128(qa + off, 0, 1024), sdesc_sw128(ka + off, 0, 1024),
                 idS, k > 0 ? 1u : 0u);
          if (k == D / 16 - 3) peek();
        }
      };
      auto issue_PV = [&](int t, int vslot, bool acc) {
        const uint32_t va = sb + C::kKVOff + vslot * C::kTileBytes;
#pragma unroll
        for (int k = 0; k < kBN / 16; ++k) {
          mma_ts(tmem + C::col_O(t), tmem + C::col_S(t) + 8 * k,
                 sdesc_sw128(va + k * 2048, kPanelBytes, 1024), idO, (acc || k > 0) ? 1u : 0u);
        }
      };
      // O_t += P_lo V for a tile whose P was written in two bf16 parts (its
      // only key step): the low part lies over S columns [64, 128).
      auto issue_PV_lo = [&](int t, int vslot) {
        const uint32_t va = sb + C::kKVOff + vslot * C::kTileBytes;
#pragma unroll
        for (int k = 0; k < kBN / 16; ++k)
          mma_ts(tmem + C::col_O(t), tmem + C::col_S(t) + 64 + 8 * k,
                 sdesc_sw128(va + k * 2048, kPanelBytes, 1024), idO, 1u);
      };
      // K_j and V_j are ring loads 2j and 2j+1, in the producer's order.
      // Their slots are released by the softmax warps (see there), so the
      // only shared-memory operations this thread does between two groups of
      // products are one commit and the waits.  Each of those takes a
      // round trip through shared memory, which the tensor core keeps busy;
      // the `peek` tests overlap them with the issue of the previous group.
      auto kv_bar = [](int i) { return C::kKVFull + i % C::kSlots; };
      auto kv_par = [](int i) { return static_cast<uint32_t>((i / C::kSlots) & 1); };
      bool ok = true;
      for (int t = 0; t < 2 && ok; ++t)
        if (n_t[t] > 0) ok = mbar_wait(bar(C::kQFull + t), 0, p.ctl, abort_flag);
      if (ok) ok = mbar_wait(bar(kv_bar(0)), kv_par(0), p.ctl, abort_flag);
      if (ok) {
        tc_fence_after();
        for (int t = 0; t < 2; ++t)
          if (n_t[t] > 0) { issue_S(t, 0, [] {}); tc_commit(bar(C::kSFull + t)); }
      }
      uint32_t pph[2] = {0, 0};
      bool kv_ready = false, p_ready[2] = {false, false};
      // One key step of both tiles.  `first` (a compile-time tag) marks the
      // first step, the only one where a tile may take its P in two parts:
      // the per-step loop itself carries no test for it.
      auto step = [&](const int j, auto first) {
        const int iv = 2 * j + 1, ik = 2 * j + 2;       // V_j, K_{j+1}
        const bool has_next = j + 1 < n_max;
        if (!kv_ready) {
          ok = mbar_wait(bar(kv_bar(iv)), kv_par(iv), p.ctl, abort_flag);
          if (ok && has_next) ok = mbar_wait(bar(kv_bar(ik)), kv_par(ik), p.ctl, abort_flag);
          if (!ok) return;
        }
        kv_ready = false;
        for (int t = 0; t < 2 && ok; ++t) {
          if (j >= n_t[t]) continue;
          if (!p_ready[t]) ok = mbar_wait(bar(C::kPFull + t), pph[t], p.ctl, abort_flag);
          pph[t] ^= 1;
          p_ready[t] = false;
          if (!ok) break;
          tc_fence_after();
          issue_PV(t, iv % C::kSlots, j > 0);
          if constexpr (decltype(first)::value)
            if (SPLIT && n_t[t] == 1) issue_PV_lo(t, iv % C::kSlots);
          if (j + 1 < n_t[t]) {
            if (t == 0) {
              issue_S(0, ik % C::kSlots, [&] {
                if (j < n_t[1]) p_ready[1] = mbar_test_wait(bar(C::kPFull + 1), pph[1]);
              });
            } else {
              issue_S(1, ik % C::kSlots, [&] {
                const int iv2 = iv + 2, ik2 = ik + 2;   // V_{j+1}, K_{j+2}
                const bool a = mbar_test_wait(bar(kv_bar(iv2)), kv_par(iv2));
                const bool b = ik2 >= 2 * n_max || mbar_test_wait(bar(kv_bar(ik2)), kv_par(ik2));
                const bool c = j + 1 >= n_t[0] || mbar_test_wait(bar(C::kPFull + 0), pph[0]);
                kv_ready = a && b;
                p_ready[0] = c && j + 1 < n_t[0];
              });
            }
            tc_commit(bar(C::kSFull + t));
          } else {
            tc_commit(bar(C::kOFull + t));
          }
        }
      };
      if (n_max > 0 && ok) step(0, std::true_type{});
      for (int j = 1; j < n_max && ok; ++j) step(j, std::false_type{});
    }
  } else {
    // -------------------------------------------------------------- softmax
    const int t = (warp - 2) >> 2;          // query tile of this warpgroup
    const int rank = warp & 3;              // tensor-memory lane quarter
    const int r_in_tile = rank * 32 + lane;
    const int row = qbase0 + t * kBM + r_in_tile;
    const int nt = n_t[t];
    const uint32_t lane_addr = static_cast<uint32_t>(rank * 32) << 16;
    const uint32_t tS = tmem + lane_addr + C::col_S(t);
    const uint32_t tO = tmem + lane_addr + C::col_O(t);
    const bool releaser = t == (n_t[1] > 0 ? 1 : 0);
    const float c = p.c;
    float m_ref = -INFINITY;
    float l = 0.f;      // sum of the fp32 probabilities: gives the LSE
    float lr = 0.f;     // rounding residuals of the blocks' largest P (see the header)
    bool ok = true;
    if (SPLIT && nt == 1) {
      // ---- the tile's only key step, P in two bf16 parts (see the header)
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kSFull + t), 0, p.ctl, abort_flag));
      if (ok) {
        if (releaser && r_in_tile == 0) mbar_arrive(bar(C::kKVEmpty + 0));
        tc_fence_after();
        uint32_t s[128];
        tmem_ld_x128(tS, s);
        int lim = p.N_kv - 1;
        if (p.causal) lim = min(lim, row);
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (i > lim) s[i] = __float_as_uint(-INFINITY);
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int i = 0; i < 128; i += 8) {
          mx[0] = max3(mx[0], __uint_as_float(s[i + 0]), __uint_as_float(s[i + 1]));
          mx[1] = max3(mx[1], __uint_as_float(s[i + 2]), __uint_as_float(s[i + 3]));
          mx[2] = max3(mx[2], __uint_as_float(s[i + 4]), __uint_as_float(s[i + 5]));
          mx[3] = max3(mx[3], __uint_as_float(s[i + 6]), __uint_as_float(s[i + 7]));
        }
        m_ref = c * fmaxf(max3(mx[0], mx[1], mx[2]), mx[3]);
        const float2 c2 = make_float2(c, c);
        const float2 neg2 = make_float2(-m_ref, -m_ref);
        float2 sum[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int q = 16 * h + i;
            const float2 x = fma2(make_float2(__uint_as_float(s[2 * q]), __uint_as_float(s[2 * q + 1])), c2, neg2);
            const float e0 = ex2_mix<EMU>(x.x, 2 * q);
            const float e1 = ex2_mix<EMU>(x.y, 2 * q + 1);
            sum[i & 1] = add2(sum[i & 1], make_float2(e0, e1));
            hi[i] = pack_bf16x2(e0, e1);
            lo[i] = pack_bf16x2(e0 - __uint_as_float(hi[i] << 16), e1 - __uint_as_float(hi[i] & 0xffff0000u));
          }
          tmem_st_x16(tS + 16 * h, hi);
          tmem_st_x16(tS + 64 + 16 * h, lo);
        }
        l = (sum[0].x + sum[0].y) + (sum[1].x + sum[1].y);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::kPFull + t));
      }
    }
    for (int j = 0; j < nt && !(SPLIT && nt == 1); ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kSFull + t), j & 1, p.ctl, abort_flag));
      if (!ok) break;
      // S_t,j complete means every product queued before it is complete too:
      // the tile that runs to the last key tile (tile 1 unless it is empty)
      // hands K_j and V_{j-1} back to the producer.
      if (releaser && r_in_tile == 0) {
        mbar_arrive(bar(C::kKVEmpty + (2 * j) % C::kSlots));
        if (j > 0) mbar_arrive(bar(C::kKVEmpty + (2 * j - 1) % C::kSlots));
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
      const float mxs = fmaxf(max3(mx[0], mx[1], mx[2]), mx[3]);   // raw scores
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
      float pmax = 0.f;   // largest P as computed (emulated exponentials differ slightly)
      uint32_t pk[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        const float2 x = fma2(make_float2(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])), c2, neg2);
        const float e0 = ex2_mix<EMU>(x.x, 2 * i);
        const float e1 = ex2_mix<EMU>(x.y, 2 * i + 1);
        sum[i & 1] = add2(sum[i & 1], make_float2(e0, e1));
        if constexpr (EMU > 0) pmax = max3(pmax, e0, e1);
        const uint32_t w = pack_bf16x2(e0, e1);
        pk[i] = w;
      }
      l += (sum[0].x + sum[0].y) + (sum[1].x + sum[1].y);
      {
        // the block's largest P: with every exponential on the ex2 unit,
        // recomputed exactly as its element was (same fused multiply-add)
        const float pm = EMU > 0 ? pmax : ex2_hw(fmaf(mxs, c, -m_ref));
        const float pmr = __uint_as_float(pack_bf16x2(pm, pm) << 16);   // as rounded for P V
        lr += pmr - pm;
      }
      tmem_st_x64(tS, pk);   // waits for its own stores
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::kPFull + t));
    }
    // ------------------------------------------------------------- epilogue
    bool ready = ok && nt > 0;
    if (ready) ready = mbar_wait(bar(C::kOFull + t), 0, p.ctl, abort_flag);
    if (__all_sync(0xffffffffu, ready)) {
      tc_fence_after();
      const float inv_l = 1.f / (l + lr);
      // O (bf16) of this warp's 32 rows into the tile's Q buffer, dead since
      // the tile's last S, in the 128-byte-swizzled layout of a TMA box
      // (64 columns x 32 rows per panel); lane 0 stores the boxes (rows
      // past N_q are clipped by the tensor map).  The buffer and row in the
      // tile come from a fresh read of the thread index: values that live
      // through the key loop only for this would take registers there.
      const uint32_t tid = tid_x_fresh();
      const uint32_t r_tile = tid & 127;                   // row in the query tile
      const uint32_t buf = C::kQOff + ((tid - 64) >> 7) * C::kTileBytes;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t o[32];
        tmem_ld_x32(tO + 32 * ch, o);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
        // columns 32 ch .. 32 ch + 31: panel ch / 2, 16-byte chunks 4 (ch & 1) .. + 3
        uint8_t* rowp = smem + buf + (ch >> 1) * kPanelBytes + r_tile * 128;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          *reinterpret_cast<uint4*>(rowp + (((4 * (ch & 1) + i) ^ (r_tile & 7)) * 16)) =
              make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        for (int pn = 0; pn < C::kPanels; ++pn)
          tma_store_3d(&tmO, sb + buf + pn * kPanelBytes + (r_tile & ~31u) * 128, 64 * pn, row - lane, bh);
        bulk_commit_group();
      }
      if (row < p.N_q)
        p.lse[static_cast<size_t>(bh) * p.N_q + row] = (m_ref + log2f(l)) * 0.69314718055994531f;
    }
  }

  if (warp >= 2 && lane == 0) bulk_wait_group_read<0>();   // O's boxes have been read
  __syncwarp();   // warps whose lane 0 ran a role alone arrive whole
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, int EMU, bool SPLIT>
cudaError_t launch(const FwdLaunch& a) {
  using C = Cfg<D>;
  Params p;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.BH = a.BH;
  p.N_q = a.N_q;
  p.N_kv = a.N_kv;
  p.causal = a.causal;
  p.n_qpairs = (a.N_q + 2 * kBM - 1) / (2 * kBM);
  p.n_kv_tiles = (a.N_kv + kBN - 1) / kBN;
  p.c = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  p.tau = a.tau;
  p.ctl = a.ctl;
  auto kern = fwd_kernel<D, EMU, SPLIT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(p.n_qpairs) * p.BH;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  kern<<<static_cast<unsigned>(grid), kThreads, C::kSmemBytes, a.stream>>>(a.tmQ, a.tmK, a.tmV, a.tmO, p);
  return cudaGetLastError();
}

template <int D, bool SPLIT>
cudaError_t launch_emu(const FwdLaunch& a) {
  switch (a.emu_per_32) {
    case 0: return launch<D, 0, SPLIT>(a);
    case 8: return launch<D, 8, SPLIT>(a);
    case 16: return launch<D, 16, SPLIT>(a);
    default: return cudaErrorInvalidValue;
  }
}

template <int D>
cudaError_t launch_any(const FwdLaunch& a) {
  // a query tile sees a single key tile only with a causal mask (the first
  // one) or when all keys fit in one tile
  const bool split = a.causal || a.N_kv <= kBN;
  return split ? launch_emu<D, true>(a) : launch_emu<D, false>(a);
}

}  // namespace fwd
}  // namespace fa
