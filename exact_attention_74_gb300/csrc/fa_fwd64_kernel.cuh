// fa_fwd64_kernel.cuh -- the forward at head dimension 64, with S, P and O in
// separate tensor-memory columns and one product-issuing thread per query
// tile.
//
// The arithmetic is the forward kernel's (fa_fwd_kernel.cuh: the online
// softmax of "FlashAttention: GPUメモリ階層を活用したアテンション最適化の分析"
// §6.2 in base 2 with the conditional rescaling of "論文解説:
// FlashAttention-4 — Algorithm and Kernel Pipelining Co-Design for
// Asymmetric Hardware Scaling", 条件付きオンラインsoftmaxリスケーリング, the
// same O normalisation and LSE, the same two-part P for tiles with one key
// tile); what differs is the schedule.  At d = 64 a key step's products are
// small next to its softmax, and writing P over S made every tile's next S
// wait for its P V: the step was softmax, notification, P V and S, and S's
// latency in turn.  Here each query tile t has
//   S_t at columns [256 t, 256 t + 128), P_t (bf16 pairs) at [256 t + 128,
//   256 t + 192), O_t at [256 t + 192, 256 t + 256)    (512 columns in all)
// and its own issuing thread (warp 1 for tile 0, warp 10 for tile 1), which
// issues S_t,j+1 as soon as the softmax has read S_t,j into registers and
// P_t,j V_j when P_t,j is written.  The softmax warps so find the next S
// ready when they finish a step, and the tensor core runs P V and the next S
// while they work.
//
//   warp 0       TMA producer: Q tiles once, K_j, V_j through a ring of
//                shared-memory slots
//   warps 1, 10  issuing thread of tile 0, tile 1
//   warps 2-9    softmax of tile 0 (2-5) and tile 1 (6-9), one query row per
//                thread; a tile's warps hand K_j back once S_t,j is complete
//                and V_j once P_t,j V_j is, so a slot is refilled after both
//                tiles (or the one tile that still reads it) are done with it.
#pragma once

#include "fa_fwd_kernel.cuh"

namespace fa {
namespace fwd64 {

using fwd::kBM;
using fwd::kBN;
using fwd::Params;
constexpr int D = 64;
constexpr int kThreads = 352;            // 11 warps
constexpr int kTileBytes = kBM * D * 2;  // 16 KB: one Q tile, or K_j, or V_j
constexpr int kSlots = 8;
constexpr int kQOff = 0;
constexpr int kKVOff = 2 * kTileBytes;
constexpr int kBarOff = kKVOff + kSlots * kTileBytes;
// barrier indices
constexpr int kQFull = 0;                 // 2
constexpr int kKVFull = 2;                // kSlots
constexpr int kKVEmpty = 2 + kSlots;      // kSlots; two arrivals per use
constexpr int kSFull = 2 + 2 * kSlots;    // 2: S_t,j complete (issuer's commit)
constexpr int kSFree = 4 + 2 * kSlots;    // 2: S_t,j read by the softmax (one arrival per warp)
constexpr int kPFull = 6 + 2 * kSlots;    // 2: P_t,j written (one arrival per warp)
constexpr int kPFree = 8 + 2 * kSlots;    // 2: P_t,j V_j complete (issuer's commit)
constexpr int kNumBars = 10 + 2 * kSlots;
constexpr int kMiscOff = kBarOff + 8 * kNumBars;
constexpr int kSmemBytes = kMiscOff + 16 + 1024;   // + base alignment slack
constexpr uint32_t kTmemCols = 512;
__device__ constexpr uint32_t col_S(int t) { return 256u * t; }
__device__ constexpr uint32_t col_P(int t) { return 256u * t + 128u; }
__device__ constexpr uint32_t col_O(int t) { return 256u * t + 192u; }

template <int EMU, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
fwd64_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
             const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO, const Params p) {
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
  const int n_t[2] = {fwd::tiles_for(p, qbase0), fwd::tiles_for(p, qbase0 + kBM)};
  const int n_max = max(n_t[0], n_t[1]);
  auto kv_slot = [](int i) { return i % kSlots; };
  auto kv_par = [](int i) { return static_cast<uint32_t>((i / kSlots) & 1); };

  if (threadIdx.x == 0) {
    mbar_init(bar(kQFull + 0), 1);
    mbar_init(bar(kQFull + 1), 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(bar(kKVFull + s), 1);
      mbar_init(bar(kKVEmpty + s), 2);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(kSFull + t), 1);
      mbar_init(bar(kSFree + t), 4);
      mbar_init(bar(kPFull + t), 4);
      mbar_init(bar(kPFree + t), 1);
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
      for (int i = 0; i < 2 * n_max; ++i) {          // K_j = load 2j, V_j = load 2j + 1
        const int s = kv_slot(i);
        if (!mbar_wait(bar(kKVEmpty + s), kv_par(i) ^ 1, p.ctl, abort_flag)) break;
        mbar_arrive_expect_tx(bar(kKVFull + s), kTileBytes);
        tma_load_3d_hint(sb + kKVOff + s * kTileBytes, (i & 1) ? &tmV : &tmK, bar(kKVFull + s), 0,
                         (i >> 1) * kBN, bh, keep);
      }
    }
  } else if ((warp == 1 || warp == 10) && lane == 0) {
    // ------------------------------------------- issuing thread of tile t
    const int t = warp == 1 ? 0 : 1;
    const int nt = n_t[t];
    constexpr uint32_t idS = idesc_bf16(kBM, kBN, false, false);
    constexpr uint32_t idO = idesc_bf16(kBM, D, false, true);
    const uint32_t qa = sb + kQOff + t * kTileBytes;
    auto issue_S = [&](int j) {          // S_t,j = Q_t K_j^T
      const uint32_t ka = sb + kKVOff + kv_slot(2 * j) * kTileBytes;
#pragma unroll
      for (int k = 0; k < D / 16; ++k)
        mma_ss(tmem + col_S(t), sdesc_sw128(qa + 32 * k, 0, 1024), sdesc_sw128(ka + 32 * k, 0, 1024), idS,
               k > 0 ? 1u : 0u);
    };
    auto issue_PV = [&](int j, uint32_t a_col, bool acc) {   // O_t += P V_j (P from tensor memory)
      const uint32_t va = sb + kKVOff + kv_slot(2 * j + 1) * kTileBytes;
#pragma unroll
      for (int k = 0; k < kBN / 16; ++k)
        mma_ts(tmem + col_O(t), tmem + a_col + 8 * k, sdesc_sw128(va + k * 2048, fwd::kPanelBytes, 1024), idO,
               (acc || k > 0) ? 1u : 0u);
    };
    bool ok = nt > 0;
    if (ok) ok = mbar_wait(bar(kQFull + t), 0, p.ctl, abort_flag);
    if (ok) ok = mbar_wait(bar(kKVFull + kv_slot(0)), kv_par(0), p.ctl, abort_flag);
    if (ok) {
      tc_fence_after();
      issue_S(0);
      tc_commit(bar(kSFull + t));
    }
    for (int j = 0; j < nt && ok; ++j) {
      if (j + 1 < nt) {        // the next S once the softmax has read this one
        ok = mbar_wait(bar(kSFree + t), j & 1, p.ctl, abort_flag);
        if (ok) ok = mbar_wait(bar(kKVFull + kv_slot(2 * j + 2)), kv_par(2 * j + 2), p.ctl, abort_flag);
        if (!ok) break;
        tc_fence_after();
        issue_S(j + 1);
        tc_commit(bar(kSFull + t));
      }
      ok = mbar_wait(bar(kPFull + t), j & 1, p.ctl, abort_flag);
      if (ok) ok = mbar_wait(bar(kKVFull + kv_slot(2 * j + 1)), kv_par(2 * j + 1), p.ctl, abort_flag);
      if (!ok) break;
      tc_fence_after();
      issue_PV(j, col_P(t), j > 0);
      // a tile with one key step takes P in two parts: the low part lies
      // over the (dead) S columns
      if (SPLIT && nt == 1) issue_PV(j, col_S(t), true);
      tc_commit(bar(kPFree + t));
    }
  } else if (warp >= 2 && warp <= 9) {
    // -------------------------------------------------------------- softmax
    const int t = (warp - 2) >> 2;          // query tile of this warpgroup
    const int rank = warp & 3;              // tensor-memory lane quarter
    const int r_in_tile = rank * 32 + lane;
    const int row = qbase0 + t * kBM + r_in_tile;
    const int nt = n_t[t];
    const int other = n_t[t ^ 1];
    const uint32_t lane_addr = static_cast<uint32_t>(rank * 32) << 16;
    const uint32_t tS = tmem + lane_addr + col_S(t);
    const uint32_t tP = tmem + lane_addr + col_P(t);
    const uint32_t tO = tmem + lane_addr + col_O(t);
    // One thread per tile hands a K/V slot back: once, or twice when the
    // other tile does not read that key tile at all.
    const bool hander = warp == (t == 0 ? 2 : 6) && lane == 0;
    auto hand_back = [&](int i) {
      if (!hander) return;
      mbar_arrive(bar(kKVEmpty + kv_slot(i)));
      if ((i >> 1) >= other) mbar_arrive(bar(kKVEmpty + kv_slot(i)));
    };
    const float c = p.c;
    float m_ref = -INFINITY;
    float l = 0.f;      // sum of the fp32 probabilities: gives the LSE
    float lr = 0.f;     // rounding residuals of the blocks' largest P
    bool ok = true;
    if (SPLIT && nt == 1) {
      // ---- the tile's only key step: P in two bf16 parts, hi over P's
      // columns and lo = bf16(P - hi) over the (dead) S columns [0, 64)
      ok = __all_sync(0xffffffffu, mbar_wait(bar(kSFull + t), 0, p.ctl, abort_flag));
      if (ok) {
        hand_back(0);                         // K_0
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
            const float e0 = fwd::ex2_mix<EMU>(x.x, 2 * q);
            const float e1 = fwd::ex2_mix<EMU>(x.y, 2 * q + 1);
            sum[i & 1] = add2(sum[i & 1], make_float2(e0, e1));
            hi[i] = pack_bf16x2(e0, e1);
            lo[i] = pack_bf16x2(e0 - __uint_as_float(hi[i] << 16), e1 - __uint_as_float(hi[i] & 0xffff0000u));
          }
          tmem_st_x16(tP + 16 * h, hi);
          tmem_st_x16(tS + 16 * h, lo);
        }
        l = (sum[0].x + sum[0].y) + (sum[1].x + sum[1].y);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kPFull + t));
      }
    }
    for (int j = 0; j < nt && !(SPLIT && nt == 1); ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar(kSFull + t), j & 1, p.ctl, abort_flag));
      if (!ok) break;
      hand_back(2 * j);                       // K_j: this tile's S_t,j is complete
      tc_fence_after();
      uint32_t s[128];
      tmem_ld_x128(tS, s);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kSFree + t));   // the next S may be written now
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
      // P_t,j-1 V_{j-1} must be complete before O is rescaled and before
      // P_t,j is written over P_t,j-1
      bool pv_done = j == 0;
      if (__any_sync(0xffffffffu, resc)) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(kPFree + t), (j - 1) & 1, p.ctl, abort_flag));
        if (!ok) break;
        pv_done = true;
        hand_back(2 * j - 1);                 // V_{j-1}
        tc_fence_after();
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
        const float e0 = fwd::ex2_mix<EMU>(x.x, 2 * i);
        const float e1 = fwd::ex2_mix<EMU>(x.y, 2 * i + 1);
        sum[i & 1] = add2(sum[i & 1], make_float2(e0, e1));
        if constexpr (EMU > 0) pmax = max3(pmax, e0, e1);
        pk[i] = pack_bf16x2(e0, e1);
      }
      l += (sum[0].x + sum[0].y) + (sum[1].x + sum[1].y);
      {
        // the block's largest P: with every exponential on the ex2 unit,
        // recomputed exactly as its element was (same fused multiply-add)
        const float pm = EMU > 0 ? pmax : ex2_hw(fmaf(mxs, c, -m_ref));
        const float pmr = __uint_as_float(pack_bf16x2(pm, pm) << 16);   // as rounded for P V
        lr += pmr - pm;
      }
      if (!pv_done) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(kPFree + t), (j - 1) & 1, p.ctl, abort_flag));
        if (!ok) break;
        hand_back(2 * j - 1);               // V_{j-1}
        tc_fence_after();
      }
      tmem_st_x64(tP, pk);   // waits for its own stores
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kPFull + t));
    }
    // ------------------------------------------------------------- epilogue
    bool ready = ok && nt > 0;
    if (ready) ready = mbar_wait(bar(kPFree + t), (nt - 1) & 1, p.ctl, abort_flag);
    if (__all_sync(0xffffffffu, ready)) {
      hand_back(2 * nt - 1);                  // V of the last step
      tc_fence_after();
      const float inv_l = 1.f / (l + lr);
      // O (bf16) of this warp's 32 rows into the tile's Q buffer, dead since
      // the tile's last S, as a 128-byte-swizzled TMA box (64 columns x 32
      // rows); lane 0 stores it (rows past N_q are clipped by the tensor map)
      uint8_t* rowp = smem + kQOff + t * kTileBytes + r_in_tile * 128;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t o[32];
        tmem_ld_x32(tO + 32 * ch, o);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          *reinterpret_cast<uint4*>(rowp + (((4 * ch + i) ^ (r_in_tile & 7)) * 16)) =
              make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_3d(&tmO, sb + kQOff + t * kTileBytes + rank * 32 * 128, 0, qbase0 + t * kBM + rank * 32, bh);
        bulk_commit_group();
      }
      if (row < p.N_q)
        p.lse[static_cast<size_t>(bh) * p.N_q + row] = (m_ref + log2f(l)) * 0.69314718055994531f;
    }
  }

  if (warp >= 2 && warp <= 9 && lane == 0) bulk_wait_group_read<0>();   // O's box has been read
  __syncwarp();   // warps whose lane 0 ran a role alone arrive whole
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int EMU, bool SPLIT>
cudaError_t launch(const FwdLaunch& a) {
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
  auto kern = fwd64_kernel<EMU, SPLIT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(p.n_qpairs) * p.BH;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  kern<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, a.stream>>>(a.tmQ, a.tmK, a.tmV, a.tmO, p);
  return cudaGetLastError();
}

template <bool SPLIT>
cudaError_t launch_emu(const FwdLaunch& a) {
  switch (a.emu_per_32) {
    case 0: return launch<0, SPLIT>(a);
    case 8: return launch<8, SPLIT>(a);
    case 16: return launch<16, SPLIT>(a);
    default: return cudaErrorInvalidValue;
  }
}

inline cudaError_t launch_any(const FwdLaunch& a) {
  const bool split = a.causal || a.N_kv <= kBN;
  return split ? launch_emu<true>(a) : launch_emu<false>(a);
}

}  // namespace fwd64
}  // namespace fa
