// fa_bwd64_kernel.cuh -- the backward main pass at head dimension 64 (the
// unordered dQ reduction), with every product's operands and results in
// their own tensor-memory columns.
//
// The arithmetic is the backward kernel's (fa_bwd_kernel.cuh): for one
// 128-key tile j and each query tile i it recomputes S^T and P^T from the
// saved LSE, dP^T = V dO^T, dS = P o (dP - D), and accumulates dV += P^T dO,
// dK += dS^T Q and the partial dQ_i = dS K, added into the fp32 accumulator
// with TMA reduce-adds.  What differs is the schedule.  The kernel at d = 128
// has no spare tensor memory: P and dS^T land over S, the partial dQ over dP,
// and so the next tile's S waits for dK and its dP for the drain of dQ.  At
// d = 64 there is room for
//   S^T [0, 128), P^T [128, 192) (bf16 pairs), dP^T [192, 320),
//   dQ [320, 384), dV [384, 448), dK [448, 512)
// with dK taking dS^T from shared memory (the buffer dQ reads, as a K-major
// operand) rather than from tensor memory.  Two threads issue the products
// (on one, the waits for P, dS and the drained dQ would hold back products
// whose own inputs are ready):
//   warp 1   S_{i+1}  as soon as the compute warps have read S_i,
//            dV_i     once P_i is written (and dO_i has landed),
//            dK_i     once dS_i is in shared memory;
//   warp 18  dP_{i+1} as soon as the compute warps have read dP_i,
//            dQ_i     once dS_i is in shared memory and dQ_{i-1} has left
//                     dQ's columns,
// so the compute warps find the next S and dP complete when they reach them.
// Sixteen compute warps (2-17), four per tensor-memory lane quarter, each
// take 32 of a tile's 128 query columns of P and dS: at d = 64 a step's
// element work is as large as at d = 128 while its products are half, and
// 32 columns per thread keep the warps within the registers that 19 warps
// leave each (96); warps 2-9 also drain dQ and write dK and dV.  They
// drain dQ_{i-1} right after handing P_i over, through a dedicated box
// area (the drain does not wait for a dead Q/dO buffer); the compute warps
// rewrite dS and the producer refills a Q/dO stage only once both threads' products of
// that tile have completed (per-stage barriers, so no wait can be mistaken
// for the same stage's next phase).
// "FlashAttention: GPUメモリ階層を活用したアテンション最適化の分析" §7.2
// (recomputation), "論文解説: FlashAttention-4 — Algorithm and Kernel
// Pipelining Co-Design for Asymmetric Hardware Scaling", Backwardパスの最適化
// (intermediates in tensor memory).
#pragma once

#include "fa_bwd_kernel.cuh"

namespace fa {
namespace bwd64 {

constexpr int D = 64;
constexpr int kBM = 128;          // keys per CTA
constexpr int kBN = 128;          // queries per step
constexpr int kThreads = 608;     // warps 0-18
constexpr int kTile = 128 * D * 2;                      // 16 KB
constexpr int kPanel = 128 * 128;                       // 128 rows x 128 B
constexpr int kK = 0;
constexpr int kV = kTile;
constexpr int kStage0 = 2 * kTile;
constexpr int kStageBytes = 2 * kTile + 1024;           // Q, dO, lse2[128], delta[128]
constexpr int kDS = kStage0 + 2 * kStageBytes;          // dS^T, 2 panels of 128 keys x 64 queries
constexpr int kDrain = kDS + 2 * kPanel;                // partial dQ: 8 boxes of 32 x 32 fp32
constexpr int kBar = kDrain + 8 * 4096;
enum : int {
  bKV = 0, bQ = 1, bDO = 3,                             // two of bQ and bDO (per stage)
  bS = 5, bSFree, bP, bPFree, bDP, bDPFree, bDS, bDQFree, bAcc,
  bDQ = 14, bKD = 16,                                   // per stage: dQ_i (warp 18), dK_i (warp 1) complete
  kNumBars = 18
};
constexpr int kMisc = kBar + 8 * kNumBars;
constexpr int kSmem = kMisc + 16;
static_assert(kSmem <= 232448, "shared memory");
static_assert(kStageBytes % 1024 == 0 && kDS % 1024 == 0 && kDrain % 1024 == 0, "alignment");
constexpr uint32_t kColS = 0, kColP = 128, kColDP = 192, kColDQ = 320, kColDV = 384, kColDK = 448;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kWarps = 16;   // compute warps: one arrival each
constexpr uint32_t kDrainWarps = 8;   // of them, those that drain dQ and write dK, dV

__global__ void __launch_bounds__(kThreads, 1)
main64_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
              const __grid_constant__ CUtensorMap tmDQ, const bwd::Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  if (sb & 1023u) {   // operand atoms need 1024-byte alignment
    if (threadIdx.x == 0) atomicOr(p.ctl.status, kStatusLaunchConfig);
    return;
  }
  auto bar = [&](int i) -> uint32_t { return sb + kBar + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMisc + 4);
  int* logical_slot = reinterpret_cast<int*>(smem + kMisc + 8);
  auto wait = [&](int b, int parity) -> bool {
    return mbar_wait(bar(b), static_cast<uint32_t>(parity) & 1u, p.ctl, abort_flag);
  };
  auto stage = [&](int s) -> uint32_t { return sb + kStage0 + s * kStageBytes; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    const int b = static_cast<int>(atomicAdd(p.ticket, 1u));
    mbar_init(bar(bKV), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(bQ + s), 1);
      mbar_init(bar(bDO + s), 1);
    }
    mbar_init(bar(bS), 1);
    mbar_init(bar(bPFree), 1);
    mbar_init(bar(bDP), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(bDQ + s), 1);
      mbar_init(bar(bKD + s), 1);
    }
    mbar_init(bar(bAcc), 1);
    mbar_init(bar(bSFree), kWarps);
    mbar_init(bar(bP), kWarps);
    mbar_init(bar(bDPFree), kWarps);
    mbar_init(bar(bDS), kWarps);
    mbar_init(bar(bDQFree), kDrainWarps);
    *abort_flag = 0;
    mbar_init_fence();
    *logical_slot = b;
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  __syncwarp();   // warps whose lane 0 ran a role alone arrive whole
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int logical = *logical_slot;
  int j, bh;
  bwd::block_tile<false>(p, logical, j, bh);
  const int i0 = p.causal ? j : 0;                  // first query tile that sees these keys
  const int n_it = max(0, p.n_q_tiles - i0);

  if (n_it > 0 && warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmdO);
      mbar_arrive_expect_tx(bar(bKV), 2 * kTile);
      tma_load_3d(sb + kK, &tmK, bar(bKV), 0, j * kBM, bh);
      tma_load_3d(sb + kV, &tmV, bar(bKV), 0, j * kBM, bh);
      const uint64_t keep = l2_policy_evict_last();
      for (int t = 0; t < n_it; ++t) {
        const int s = t & 1;
        const int i = i0 + t;
        // tile t-2's dQ and dK (the last readers of its Q and dO) are complete
        if (t >= 2 && !(wait(bDQ + s, (t - 2) >> 1) && wait(bKD + s, (t - 2) >> 1))) break;
        const uint32_t st = stage(s);
        mbar_arrive_expect_tx(bar(bQ + s), kTile + 1024);
        tma_load_3d_hint(st, &tmQ, bar(bQ + s), 0, i * kBN, bh, keep);
        const size_t row = static_cast<size_t>(bh) * p.nq_pad + static_cast<size_t>(i) * kBN;
        bulk_load(st + 2 * kTile, p.lse2 + row, 512, bar(bQ + s));
        bulk_load(st + 2 * kTile + 512, p.delta + row, 512, bar(bQ + s));
        mbar_arrive_expect_tx(bar(bDO + s), kTile);
        tma_load_3d_hint(st + kTile, &tmdO, bar(bDO + s), 0, i * kBN, bh, keep);
        if (t == max(0, n_it - 4)) {
          // the CTA one wave later reads a K/V tile nobody has touched yet
          const int nb = logical + p.n_sms;
          if (nb < static_cast<int>(gridDim.x)) {
            int nj, nbh;
            bwd::block_tile<false>(p, nb, nj, nbh);
            tma_prefetch_l2_3d(&tmK, 0, nj * kBM, nbh);
            tma_prefetch_l2_3d(&tmV, 0, nj * kBM, nbh);
          }
        }
      }
    }
  } else if (n_it > 0 && (warp == 1 || warp == 18)) {
    // ------------------------------------------------------- MMA issuers
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16(kBM, kBN, false, false);   // S^T, dP^T
      constexpr uint32_t idKV = idesc_bf16(kBM, D, false, true);     // dV (A tmem), dK (A smem K-major)
      constexpr uint32_t idQ = idesc_bf16(kBN, D, true, true);       // dQ (A = dS^T, MN-major)
      const uint32_t sK = sb + kK, sV = sb + kV, sDS = sb + kDS;
      bool ok = wait(bKV, 0);
      if (warp == 1) {
        // S^T = K Q^T, dV += P^T dO, dK += dS^T Q
        auto issue_S = [&](int s) {
          const uint32_t sQ = stage(s);
#pragma unroll
          for (int k = 0; k < D / 16; ++k)
            mma_ss(tmem + kColS, sdesc_sw128(sK + 32 * k, 0, 1024), sdesc_sw128(sQ + 32 * k, 0, 1024), idS, k > 0);
        };
        if (ok) ok = wait(bQ + 0, 0);
        if (ok) {
          tc_fence_after();
          issue_S(0);
          tc_commit(bar(bS));
        }
        for (int it = 0; it < n_it && ok; ++it) {
          const int s = it & 1, s1 = s ^ 1;
          const uint32_t sQ = stage(s), sdO = stage(s) + kTile;
          if (it + 1 < n_it) {          // the next S once S_i has been read
            ok = wait(bSFree, it) && wait(bQ + s1, (it + 1) >> 1);
            if (!ok) break;
            tc_fence_after();
            issue_S(s1);
            tc_commit(bar(bS));
          }
          ok = wait(bP, it) && wait(bDO + s, it >> 1);   // P_i in tensor memory, dO_i landed
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < kBN / 16; ++k)   // dV += P^T dO
            mma_ts(tmem + kColDV, tmem + kColP + 8 * k, sdesc_sw128(sdO + k * 2048, kPanel, 1024), idKV,
                   (it > 0 || k > 0) ? 1u : 0u);
          tc_commit(bar(bPFree));       // P's columns may take P_{i+1}
          ok = wait(bDS, it);           // dS_i in shared memory
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < kBN / 16; ++k) {  // dK += dS^T Q  (unscaled; dS^T K-major from shared memory)
            const uint32_t off = (k >> 2) * kPanel + (k & 3) * 32;
            mma_ss(tmem + kColDK, sdesc_sw128(sDS + off, 0, 1024), sdesc_sw128(sQ + k * 2048, kPanel, 1024), idKV,
                   (it > 0 || k > 0) ? 1u : 0u);
          }
          tc_commit(bar(bKD + s));      // dS_i and this stage's Q and dO no longer read here
        }
        if (ok) tc_commit(bar(bAcc));
      } else {
        // dP^T = V dO^T, dQ_i = dS K
        auto issue_dP = [&](int s) {
          const uint32_t sdO = stage(s) + kTile;
#pragma unroll
          for (int k = 0; k < D / 16; ++k)
            mma_ss(tmem + kColDP, sdesc_sw128(sV + 32 * k, 0, 1024), sdesc_sw128(sdO + 32 * k, 0, 1024), idS, k > 0);
        };
        if (ok) ok = wait(bDO + 0, 0);
        if (ok) {
          tc_fence_after();
          issue_dP(0);
          tc_commit(bar(bDP));
        }
        for (int it = 0; it < n_it && ok; ++it) {
          const int s = it & 1, s1 = s ^ 1;
          if (it + 1 < n_it) {          // the next dP once dP_i has been read
            ok = wait(bDPFree, it) && wait(bDO + s1, (it + 1) >> 1);
            if (!ok) break;
            tc_fence_after();
            issue_dP(s1);
            tc_commit(bar(bDP));
          }
          ok = wait(bDS, it);           // dS_i in shared memory
          if (ok && it >= 1) ok = wait(bDQFree, it - 1);   // dQ_{i-1} has left its columns
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < kBM / 16; ++k)   // dQ_i = dS K  (unscaled partial)
            mma_ss(tmem + kColDQ, sdesc_sw128(sDS + k * 2048, kPanel, 1024),
                   sdesc_sw128(sK + k * 2048, kPanel, 1024), idQ, k > 0);
          tc_commit(bar(bDQ + s));      // dQ_i ready; dS_i and this stage's dO no longer read here
        }
      }
    }
  } else if (warp >= 2 && warp <= 17) {
    // ------------------------------------------------ P and dS, dQ drainage
    const int quad = warp & 3;               // tensor-memory lane quarter
    const int part = (warp - 2) >> 2;        // query columns [32 part, 32 part + 32)
    const bool drainer = part < 2;           // warps 2-9 also drain dQ and write dK, dV
    const int half = part & 1;               // their half of dQ's (and dK's, dV's) columns
    const int r = quad * 32 + lane;          // key row within the tile (and dQ query row)
    const int kg = j * kBM + r;              // global key index
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    const bool key_ok = kg < p.N_kv;
    const float2 c2 = make_float2(p.c, p.c);
    auto signal = [&](int b) {              // one arrival per warp, after every lane's part
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(b));
    };
    // the partial dQ of tile ii: this warp's 32 rows x 32 columns through its
    // box in TMA's 128-byte swizzle, added into the accumulator by lane 0
    auto drain = [&](int ii, bool good) {
      uint32_t v[32];
      tmem_ld_x32(tmem + lane_addr + kColDQ + 32 * half, v);
      tc_fence_before();
      signal(bDQFree);
      if (!good) return;
      const uint32_t box = sb + kDrain + (half * 4 + quad) * 4096;
      if (lane == 0) bulk_wait_group_read<0>();   // its previous contents have been read
      __syncwarp();
      uint8_t* rowp = smem + (box - sb) + lane * 128;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        *reinterpret_cast<uint4*>(rowp + ((u ^ (lane & 7)) * 16)) =
            make_uint4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_reduce_add_3d(&tmDQ, box, 32 * half, (i0 + ii) * kBN + 32 * quad, bh);
        bulk_commit_group();
      }
    };
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int s = it & 1;
      const int i = i0 + it;
      ok = __all_sync(0xffffffffu, wait(bS, it) && wait(bQ + s, it >> 1));
      if (!ok) break;
      tc_fence_after();
      const float* lse_s = reinterpret_cast<const float*>(smem + kStage0 + s * kStageBytes + 2 * kTile);
      const float* dlt_s = reinterpret_cast<const float*>(smem + kStage0 + s * kStageBytes + 2 * kTile + 512);
      // queries q with q_g < k_g are masked (causal); only the diagonal tile
      // has any, and only the last key tile has keys past N_kv
      const int lim = (p.causal && i == j) ? r : 0;
      const bool masked = __any_sync(0xffffffffu, lim > 0 || !key_ok);
      // ---- P = 2^(S c - LSE log2 e)
      float pf[1][32];
      uint32_t pk[1][16];
      {
        uint32_t sv[32];
        tmem_ld_x32(tmem + lane_addr + kColS + 32 * part, sv);
        tc_fence_before();
        signal(bSFree);                     // the next S may be written now
#pragma unroll
        for (int cc = 0; cc < 1; ++cc) {
          const int ch = part;                 // 32-query chunk
#pragma unroll
          for (int u = 0; u < 32; u += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(lse_s + 32 * ch + u);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int q = u + 2 * h;
              const float2 nl = h ? make_float2(-l4.z, -l4.w) : make_float2(-l4.x, -l4.y);
              const float2 x = fma2(make_float2(__uint_as_float(sv[32 * cc + q]), __uint_as_float(sv[32 * cc + q + 1])),
                                    c2, nl);
              pf[cc][q] = ex2_hw(x.x);
              pf[cc][q + 1] = ex2_hw(x.y);
            }
          }
          if (masked) {
#pragma unroll
            for (int q = 0; q < 32; ++q)
              if (!key_ok || 32 * ch + q < lim) pf[cc][q] = 0.f;
          }
#pragma unroll
          for (int q = 0; q < 32; q += 2) pk[cc][q >> 1] = pack_bf16x2(pf[cc][q], pf[cc][q + 1]);
        }
      }
      if (it > 0) {                         // dV_{i-1} has read P_{i-1}
        ok = __all_sync(0xffffffffu, wait(bPFree, it - 1));
        if (!ok) break;
        tc_fence_after();
      }
      tmem_st_x16(tmem + lane_addr + kColP + 16 * part, pk[0]);
      tc_fence_before();
      signal(bP);                           // dV may use P_i now
      if (it > 0) {                         // dQ_{i-1} (dK_{i-1} too: dS may be rewritten)
        const int sp = (it - 1) & 1;
        ok = __all_sync(0xffffffffu, wait(bDQ + sp, (it - 1) >> 1) && wait(bKD + sp, (it - 1) >> 1));
        if (!ok) break;
        tc_fence_after();
        if (drainer) drain(it - 1, true);
      }
      // ---- dS = P o (dP - D)
      ok = __all_sync(0xffffffffu, wait(bDP, it));
      if (!ok) break;
      tc_fence_after();
      uint32_t dpv[32];
      tmem_ld_x32(tmem + lane_addr + kColDP + 32 * part, dpv);
      tc_fence_before();
      signal(bDPFree);                      // the next dP may be written now
#pragma unroll
      for (int cc = 0; cc < 1; ++cc) {
        const int ch = part;
        uint32_t dk[16];
        const uint32_t* dp = dpv + 32 * cc;
#pragma unroll
        for (int u = 0; u < 32; u += 4) {
          const float4 d4 = *reinterpret_cast<const float4*>(dlt_s + 32 * ch + u);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int q = u + 2 * h;
            const float2 nd = h ? make_float2(-d4.z, -d4.w) : make_float2(-d4.x, -d4.y);
            const float2 t = add2(make_float2(__uint_as_float(dp[q]), __uint_as_float(dp[q + 1])), nd);
            const float2 ds = mul2(make_float2(pf[cc][q], pf[cc][q + 1]), t);
            dk[q >> 1] = pack_bf16x2(ds.x, ds.y);
          }
        }
        // dS^T row r, queries 32ch..32ch+31: panel ch/2, 16-byte chunks (ch&1)*4 + u
        uint8_t* rowp = smem + kDS + (ch >> 1) * kPanel + r * 128;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int chunk = ((ch & 1) * 4 + u) ^ (r & 7);
          *reinterpret_cast<uint4*>(rowp + chunk * 16) = make_uint4(dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
        }
      }
      fence_async_smem();
      signal(bDS);                          // dQ and dK may read dS now
    }
    if (ok && n_it > 0 && drainer) {        // the last tile's partial dQ
      ok = __all_sync(0xffffffffu, wait(bDQ + ((n_it - 1) & 1), (n_it - 1) >> 1));
      if (ok) {
        tc_fence_after();
        drain(n_it - 1, true);
      }
    }
    // ----------------------------------------------------- dK, dV epilogue
    bool ready = ok && drainer;
    if (n_it > 0 && ready) ready = wait(bAcc, 0);
    ready = __all_sync(0xffffffffu, ready);
    if (drainer && (n_it == 0 || ready)) {
      if (n_it > 0) tc_fence_after();
      constexpr int kCpr = D / 16;                // 16-byte chunks per row slice
      constexpr int kRowsPerStore = 32 / kCpr;
      uint8_t* slice = smem + kDS + (warp - 2) * (32 * D);   // 32 rows x D/2 bf16
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        const float f = which == 0 ? 1.f : p.scale;
        uint32_t v[D / 2];
        if (n_it > 0) {
          tmem_ld_x32(tmem + lane_addr + (which == 0 ? kColDV : kColDK) + half * (D / 2), v);
        } else {
#pragma unroll
          for (int u = 0; u < D / 2; ++u) v[u] = 0u;
        }
        __syncwarp();
#pragma unroll
        for (int c = 0; c < kCpr; ++c) {
          uint32_t w4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w4[e] = pack_bf16x2(__uint_as_float(v[8 * c + 2 * e]) * f, __uint_as_float(v[8 * c + 2 * e + 1]) * f);
          *reinterpret_cast<uint4*>(slice + lane * (D / 2 * 2) + ((c ^ (lane % kCpr)) * 16)) =
              make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
        __syncwarp();
        __nv_bfloat16* outp = (which == 0 ? p.dv : p.dk) + static_cast<size_t>(bh) * p.N_kv * D + half * (D / 2);
#pragma unroll
        for (int k = 0; k < kCpr; ++k) {
          const int rr = k * kRowsPerStore + lane / kCpr;
          const int cc = lane % kCpr;
          const int key = j * kBM + quad * 32 + rr;
          const uint4 w = *reinterpret_cast<const uint4*>(slice + rr * (D / 2 * 2) + ((cc ^ (rr % kCpr)) * 16));
          if (key < p.N_kv) *reinterpret_cast<uint4*>(outp + static_cast<size_t>(key) * D + cc * 8) = w;
        }
      }
    }
    if (lane == 0) bulk_wait_group0();       // this warp's reductions have landed
  }

  __syncwarp();   // warps whose lane 0 ran a role alone arrive whole
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace bwd64
}  // namespace fa
