// fa_bwd_pair_kernel.cuh -- the backward main kernel at head dimension 64 on
// pairs of CTAs that share their tensor-core products (cta_group::2):
// "論文解説: FlashAttention-4 — Algorithm and Kernel Pipelining Co-Design for
// Asymmetric Hardware Scaling", Backwardパスの最適化, item 2 (products with
// 256-row tiles across two CTAs, half as many dQ reductions).
//
// A cluster of two CTAs owns 256 consecutive keys of one (batch, head): CTA
// r (its rank in the cluster) holds K and V of keys [128 r, 128 r + 128) of
// the pair and their rows of every product in its tensor memory.  One thread
// of CTA 0 (the leader) issues every product for both; a pair product takes
// A rows from both CTAs and B columns split between them:
//   S^T  = K Q^T     M = 256 keys, N = 128 queries: CTA r loads query rows
//                    [64 r, 64 r + 64) of the tile (all 64 columns)
//   dP^T = V dO^T    the same with dO
//   dV  += P^T dO    A = P^T in tensor memory; N = 64: CTA r loads dO columns
//                    [32 r, 32 r + 32) of all 128 query rows
//   dK  += dS^T Q    A = dS^T in tensor memory; Q columns [32 r, 32 r + 32)
//   dQ   = dS K      once per two query tiles: the M = 256 rows are query
//                    tile 2m (in CTA 0) and 2m + 1 (in CTA 1), K = the pair's
//                    256 keys, N = 64.  CTA r holds, for its own query tile,
//                    dS^T of all 256 keys (its compute warps write the rows
//                    of their own keys in place; the other CTA's warps stage
//                    theirs and send them with bulk copies into this CTA's
//                    shared memory) and K columns [32 r, 32 r + 32) of all
//                    256 keys.
// Each query tile so receives one fp32 partial per 256 keys instead of one
// per 128.  The single-CTA kernel cannot be paired this way at d = 128:
// dQ must be a pair product too (a kernel may not mix single-CTA and pair
// tcgen05 instructions), and its 256-key dS^T and K operands do not fit
// beside the K, V and two Q/dO stages in 227 KB of shared memory.
//
// Roles per CTA (320 threads):
//   warp 0, lane 0   TMA loads of this CTA's operands into its own shared
//                    memory, counted on its own barriers
//   warp 1           the tensor-memory allocation (both CTAs together);
//                    lane 0 of the leader issues the products, lane 0 of
//                    CTA 1 forwards its landed loads (and the dS rows CTA 0
//                    copied into it) to the leader's barriers
//   warps 2-9        as in the single-CTA kernel: P into tensor memory, dS
//                    as dS^T into tensor memory and into shared memory (the
//                    dQ operand of the CTA whose query tile this is), the
//                    partial dQ of this CTA's query tile out of tensor memory
//                    and into the fp32 accumulator (TMA reduce-add), and the
//                    dK, dV epilogue of this CTA's keys.
// Signals into the leader: its own compute threads arrive one by one, each
// of CTA 1's compute warps once; the leader's commits arrive on the same
// barrier in both CTAs.
#pragma once

#include <cuda_bf16.h>

#include "fa_bwd_kernel.cuh"   // Params, prep and convert kernels
#include "ptx_pair.cuh"

namespace fa {
namespace bwd_pair {

constexpr int D = 64;
constexpr int kBM = 128;                  // keys per CTA (256 per pair)
constexpr int kBN = 128;                  // queries per step
constexpr int kThreads = 320;
constexpr int kHalf = 8192;               // 64 rows x 128 B, or 128 rows x 64 B
// shared memory (byte offsets; every operand 1024-byte aligned)
constexpr int kK = 0;                     // K of this CTA's keys, 128 x 64, 128-byte swizzle
constexpr int kV = 16384;
constexpr int kKc = 32768;                // K columns [32 r, 32 r + 32) of the pair's 256 keys, 64-byte swizzle
constexpr int kStage0 = 49152;
constexpr int kQh = 0, kQc = kHalf, kdOh = 2 * kHalf, kdOc = 3 * kHalf;   // within a stage
constexpr int kLse = 4 * kHalf, kDlt = 4 * kHalf + 512;
constexpr int kStageBytes = 4 * kHalf + 1024;
constexpr int kDSPanel = 256 * 128;       // dS^T, 256 keys x 64 queries
constexpr int kDS = kStage0 + 2 * kStageBytes;
constexpr int kDrain = kDS + 2 * kDSPanel;   // partial dQ: 8 boxes of 32 x 32 fp32
constexpr int kBar = kDrain + 8 * 4096;
enum : int {
  bKV = 0, bQ = 1, bDO = 3, bFree = 5,     // two of each of bQ, bDO, bFree (per stage)
  bDQFree = 7,                             // two: one per partial-dQ buffer
  bS = 9, bDP, bP, bDS0, bDS1, bDST, bDQ, bAcc, bDone, bDSIn, bDSFwd, kNumBars
};
constexpr int kMisc = kBar + 8 * kNumBars;
constexpr int kSmem = kMisc + 16;
static_assert(kSmem <= 232448, "shared memory");
static_assert(kStageBytes % 1024 == 0 && kDS % 1024 == 0 && kDrain % 1024 == 0, "alignment");
// tensor-memory columns: S^T (P^T over [0, 64), dS^T over [64, 128) as bf16
// pairs), dP^T, dV, dK, two partial-dQ buffers (pairs of query tiles
// alternate between them, so each is read out while the next is computed)
constexpr uint32_t kColS = 0, kColDS = 64, kColDP = 128, kColDV = 256, kColDK = 320, kColDQ = 384;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kLeadArrivals = 256 + 8;   // the leader's compute threads, CTA 1's compute warps
constexpr uint16_t kBoth = 3;                  // commit to both CTAs

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
pair_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
            const __grid_constant__ CUtensorMap tmKc, const __grid_constant__ CUtensorMap tmQh,
            const __grid_constant__ CUtensorMap tmQc, const __grid_constant__ CUtensorMap tmdOh,
            const __grid_constant__ CUtensorMap tmdOc, const __grid_constant__ CUtensorMap tmDQ,
            const bwd::Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  // the same offset in both CTAs, so both return here or neither does
  if (sb & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.ctl.status, kStatusLaunchConfig);
    return;
  }
  auto bar = [&](int i) -> uint32_t { return sb + kBar + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMisc + 4);
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const uint32_t peer_abort = map_shared(sb + kMisc + 4, rank ^ 1u);
  auto wait = [&](int b, int parity) -> bool {
    return pair_wait(bar(b), static_cast<uint32_t>(parity) & 1u, p.ctl, abort_flag, peer_abort);
  };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_pairs = (p.n_kv_tiles + 1) >> 1;
  const int cid = static_cast<int>(blockIdx.x >> 1);
  const int pr = cid % n_pairs;                    // pair of key tiles within the head
  const int bh = cid / n_pairs;
  const int jr = 2 * pr + static_cast<int>(rank);  // this CTA's 128-key tile
  const int i0 = p.causal ? 2 * pr : 0;            // first query tile that sees the pair's keys
  const int n_it = max(0, p.n_q_tiles - i0);

  if (threadIdx.x == 0) {
    const uint32_t fed = leader ? 2u : 1u;        // the leader also counts CTA 1's forwarded loads
    mbar_init(bar(bKV), fed);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(bQ + s), fed);
      mbar_init(bar(bDO + s), fed);
      mbar_init(bar(bFree + s), 1);
    }
    mbar_init(bar(bS), 1);
    mbar_init(bar(bDP), 1);
    mbar_init(bar(bDQ), 1);
    mbar_init(bar(bAcc), 1);
    mbar_init(bar(bDone), 1);
    mbar_init(bar(bDSIn), 1);
    mbar_init(bar(bDSFwd), 1);
    mbar_init(bar(bP), kLeadArrivals);
    mbar_init(bar(bDS0), kLeadArrivals);
    mbar_init(bar(bDS1), kLeadArrivals);
    mbar_init(bar(bDST), kLeadArrivals);
    mbar_init(bar(bDQFree), kLeadArrivals);
    mbar_init(bar(bDQFree + 1), kLeadArrivals);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  cluster_sync();               // both CTAs' barriers initialised, tensor memory allocated
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto stage = [&](int s) -> uint32_t { return sb + kStage0 + s * kStageBytes; };

  if (n_it > 0 && warp == 0) {
    // ---------------------------------------------------------------- loads
    if (lane == 0) {
      tma_prefetch_map(&tmQh);
      tma_prefetch_map(&tmQc);
      tma_prefetch_map(&tmdOh);
      tma_prefetch_map(&tmdOc);
      mbar_arrive_expect_tx(bar(bKV), 3 * 16384);
      tma_load_3d(sb + kK, &tmK, bar(bKV), 0, jr * kBM, bh);
      tma_load_3d(sb + kV, &tmV, bar(bKV), 0, jr * kBM, bh);
      tma_load_3d(sb + kKc, &tmKc, bar(bKV), 32 * static_cast<int>(rank), 2 * pr * kBM, bh);
      tma_load_3d(sb + kKc + kHalf, &tmKc, bar(bKV), 32 * static_cast<int>(rank), (2 * pr + 1) * kBM, bh);
      const uint64_t keep = l2_policy_evict_last();   // the head's other pairs read the same Q, dO
      const int qh = 64 * static_cast<int>(rank), qc = 32 * static_cast<int>(rank);
      for (int t = 0; t < n_it; ++t) {
        const int s = t & 1;
        const int i = i0 + t;
        if (t >= 2 && !wait(bFree + s, (t - 2) >> 1)) break;   // tile t-2's products are done
        const uint32_t st = stage(s);
        mbar_arrive_expect_tx(bar(bQ + s), 2 * kHalf + 1024);
        tma_load_3d_hint(st + kQh, &tmQh, bar(bQ + s), 0, i * kBN + qh, bh, keep);
        tma_load_3d_hint(st + kQc, &tmQc, bar(bQ + s), qc, i * kBN, bh, keep);
        const size_t row = static_cast<size_t>(bh) * p.nq_pad + static_cast<size_t>(i) * kBN;
        bulk_load(st + kLse, p.lse2 + row, 512, bar(bQ + s));
        bulk_load(st + kDlt, p.delta + row, 512, bar(bQ + s));
        mbar_arrive_expect_tx(bar(bDO + s), 2 * kHalf);
        tma_load_3d_hint(st + kdOh, &tmdOh, bar(bDO + s), 0, i * kBN + qh, bh, keep);
        tma_load_3d_hint(st + kdOc, &tmdOc, bar(bDO + s), qc, i * kBN, bh, keep);
      }
    }
  } else if (n_it > 0 && warp == 1 && lane == 0 && leader) {
    // ------------------------------------------------------- product issuer
    constexpr uint32_t idS = idesc_bf16(2 * kBM, kBN, false, false);   // S^T, dP^T
    constexpr uint32_t idKV = idesc_bf16(2 * kBM, D, false, true);     // dV, dK (B MN-major)
    constexpr uint32_t idQ = idesc_bf16(2 * kBN, D, true, true);       // dQ (A = dS^T, MN-major)
    const uint32_t sK = sb + kK, sV = sb + kV, sKc = sb + kKc, sDS = sb + kDS;
    auto issue_S = [&](int s) {
      const uint32_t b = stage(s) + kQh;
#pragma unroll
      for (int k = 0; k < D / 16; ++k)
        mma_ss_pair(tmem + kColS, sdesc_sw128(sK + 32 * k, 0, 1024), sdesc_sw128(b + 32 * k, 0, 1024), idS, k > 0);
    };
    auto issue_dP = [&](int s) {
      const uint32_t b = stage(s) + kdOh;
#pragma unroll
      for (int k = 0; k < D / 16; ++k)
        mma_ss_pair(tmem + kColDP, sdesc_sw128(sV + 32 * k, 0, 1024), sdesc_sw128(b + 32 * k, 0, 1024), idS, k > 0);
    };
    bool ok = wait(bKV, 0);
    if (ok) ok = wait(bQ + 0, 0);
    if (ok) {
      tc_fence_after();
      issue_S(0);
      tc_commit_pair(bar(bS), kBoth);
      ok = wait(bDO + 0, 0);
    }
    if (ok) {
      tc_fence_after();
      issue_dP(0);
      tc_commit_pair(bar(bDP), kBoth);
    }
    // dS of query tile i lives in the dQ operand of CTA (i - i0) & 1: the
    // owning CTA's warps write their rows in place, the other CTA's rows
    // arrive by bulk copy (counted on the owner's bDSIn; CTA 1 forwards its
    // count on bDSFwd).  The pair's dQ product waits for both tiles.
    for (int it = 0; it < n_it && ok; ++it) {
      const int s = it & 1;
      const uint32_t st = stage(s);
      const bool odd = it & 1;
      const bool next = it + 1 < n_it;
      const bool pair_end = odd || !next;
      const int m = it >> 1;
      if (!odd) mbar_arrive_expect_tx(bar(bDSIn), kBM * kBN * 2);   // CTA 1's dS rows of tile i
      ok = wait(bP, it);                            // P_i in both CTAs' tensor memory
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < kBN / 16; ++k)            // dV += P^T dO
        mma_ts_pair(tmem + kColDV, tmem + kColS + 8 * k, sdesc_sw64(st + kdOc + 1024 * k, 0, 512), idKV,
                    (it > 0 || k > 0) ? 1u : 0u);
      ok = wait(bDST, it);                          // dS^T_i in both CTAs' tensor memory
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < kBN / 16; ++k)            // dK += dS^T Q  (unscaled)
        mma_ts_pair(tmem + kColDK, tmem + kColDS + 8 * k, sdesc_sw64(st + kQc + 1024 * k, 0, 512), idKV,
                    (it > 0 || k > 0) ? 1u : 0u);
      tc_commit_pair(bar(bFree + s), kBoth);        // this stage's Q and dO are no longer read
      if (next) {                                   // S of the next tile (P_i was consumed by dV first)
        ok = wait(bQ + (s ^ 1), (it + 1) >> 1);
        if (!ok) break;
        tc_fence_after();
        issue_S(s ^ 1);
        tc_commit_pair(bar(bS), kBoth);
      }
      // Even tile: CTA 1 staged its rows in place and copied them into CTA 0;
      // they must have left before its warps overwrite them with the next
      // tile's rows, which they do only once the next dP is ready.
      if (!odd) ok = wait(bDS0, m) && wait(bDSIn, m);
      if (!ok) break;
      if (next) {
        ok = wait(bDO + (s ^ 1), (it + 1) >> 1);
        if (!ok) break;
        tc_fence_after();
        issue_dP(s ^ 1);
        tc_commit_pair(bar(bDP), kBoth);
      }
      if (pair_end) {
        if (odd) ok = wait(bDS1, m) && wait(bDSFwd, m);
        if (ok && m >= 2) ok = wait(bDQFree + (m & 1), (m - 2) >> 1);   // this buffer's previous dQ was read
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 2 * kBM / 16; ++k)      // dQ of both query tiles over the pair's 256 keys
          mma_ss_pair(tmem + kColDQ + 64 * (m & 1), sdesc_sw128(sDS + 2048 * k, kDSPanel, 1024),
                      sdesc_sw64(sKc + 1024 * k, 0, 512), idQ, k > 0);
        tc_commit_pair(bar(bDQ), kBoth);
      }
    }
    if (ok) tc_commit_pair(bar(bAcc), kBoth);
    // every product issued has completed before the tensor memory is released
    tc_commit_pair(bar(bDone), 1);
    wait(bDone, 0);
  } else if (n_it > 0 && warp == 1 && lane == 0) {
    // ---------------------------------------- CTA 1: forward landed loads
    // The leader's operand barriers count this CTA's loads once they have
    // landed here (in load order; a stage is reloaded only after the leader
    // has seen its previous contents and issued the products reading them).
    bool ok = wait(bKV, 0);
    if (ok) mbar_arrive_remote_relaxed(map_shared(bar(bKV), 0));
    // CTA 0's dS rows of an odd tile land here; their count is forwarded
    // after the next tile's loads, which the leader needs first.
    auto forward_ds = [&](int t) {
      mbar_arrive_expect_tx(bar(bDSIn), kBM * kBN * 2);
      ok = wait(bDSIn, t >> 1);
      if (ok) mbar_arrive_remote_relaxed(map_shared(bar(bDSFwd), 0));
    };
    for (int t = 0; t < n_it && ok; ++t) {
      const int s = t & 1;
      ok = wait(bQ + s, t >> 1);
      if (!ok) break;
      mbar_arrive_remote_relaxed(map_shared(bar(bQ + s), 0));
      ok = wait(bDO + s, t >> 1);
      if (!ok) break;
      mbar_arrive_remote_relaxed(map_shared(bar(bDO + s), 0));
      if (t >= 1 && ((t - 1) & 1)) forward_ds(t - 1);
    }
    if (ok && ((n_it - 1) & 1)) forward_ds(n_it - 1);
  } else if (warp >= 2) {
    // ------------------------------------------ P and dS rows, dQ drainage
    const int quad = warp & 3;               // tensor-memory lane quarter
    const int half = (warp - 2) >> 2;        // query columns [64 half, 64 half + 64)
    const int r = quad * 32 + lane;          // key row within this CTA's tile (and dQ query row)
    const int kg = jr * kBM + r;             // global key index
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    const bool key_ok = kg < p.N_kv;
    const float2 c2 = make_float2(p.c, p.c);
    const uint32_t pair_bar = 1 + quad;      // named barriers of the two warps of this lane quarter
    const uint32_t pair_bar2 = 5 + quad;
    // One arrival into the leader: each thread of the leader (its products
    // read only its own tensor and shared memory for these signals, so a
    // CTA-scope release is enough, or none for completed tensor-memory
    // reads), each warp of CTA 1 once, after every lane's tensor-memory
    // stores (tcgen05 fence) or shared-memory writes (async-proxy fence) and
    // the warp barrier.  CTA 1's arrival releases at cluster scope only
    // where its warps' own shared-memory writes are read next (a release at
    // that scope costs about half a microsecond per arrival).
    auto signal_leader = [&](int b, bool smem_writes) {
      if (leader) {
        if (b == bDQFree || b == bDQFree + 1) mbar_arrive_relaxed(bar(b));
        else mbar_arrive(bar(b));
      } else {
        __syncwarp();
        if (lane == 0) {
          if (smem_writes) mbar_arrive_remote(map_shared(bar(b), 0));
          else mbar_arrive_remote_relaxed(map_shared(bar(b), 0));
        }
      }
    };
    // The partial dQ of pair mm (its product has completed): this CTA's query
    // tile of the pair, out of tensor-memory buffer mm & 1 through this
    // warp's 32 x 32 box (rows 32 quad, columns 32 half, TMA's 128-byte
    // swizzle) and added into the accumulator by lane 0.
    auto drain = [&](int mm, bool good) {
      tc_fence_after();
      uint32_t v[32];
      tmem_ld_x32(tmem + lane_addr + kColDQ + 64 * (mm & 1) + 32 * half, v);
      tc_fence_before();
      signal_leader(bDQFree + (mm & 1), false);
      const int tile = i0 + 2 * mm + static_cast<int>(rank);
      if (!good || tile >= i0 + n_it) return;
      const uint32_t box = sb + kDrain + (half * 4 + quad) * 4096;
      if (lane == 0) bulk_wait_group_read<0>();      // its previous contents have been read
      __syncwarp();
      uint8_t* rowp = smem + (box - sb) + lane * 128;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        *reinterpret_cast<uint4*>(rowp + ((u ^ (lane & 7)) * 16)) =
            make_uint4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_reduce_add_3d(&tmDQ, box, 32 * half, tile * kBN + 32 * quad, bh);
        bulk_commit_group();
      }
    };
    // A failed (timed-out) wait does not end the loop: the warp keeps going
    // through every step's named-barrier hand-offs with its partner warp
    // (each of which may still be waiting on one) and only stops producing
    // results; once this CTA's abort flag is set every further wait returns
    // at once.
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int s = it & 1;
      const int i = i0 + it;
      if (ok) ok = wait(bS, it);
      if (ok) ok = wait(bQ + s, it >> 1);
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
      const float* lse_s = reinterpret_cast<const float*>(smem + kStage0 + s * kStageBytes + kLse);
      const float* dlt_s = reinterpret_cast<const float*>(smem + kStage0 + s * kStageBytes + kDlt);
      // queries q with q_g < k_g are masked (causal): all of them in the query
      // tile before this CTA's diagonal, the lower triangle on it; only the
      // last key tile has keys past N_kv
      const int lim = !p.causal ? 0 : (i < jr ? kBN : (i == jr ? r : 0));
      const bool masked = __any_sync(0xffffffffu, lim > 0 || !key_ok);
      // ---- P = 2^(S c - LSE log2 e), as soon as S is ready
      float pf[2][32];
      uint32_t pk_keep[2][16];
      {
        uint32_t sv[64];
        tmem_ld_x64(tmem + lane_addr + kColS + 64 * half, sv);
        // P of chunk ch lands on S columns the first warp of the pair has
        // read only after this signal; the second warp's dS^T later lands on
        // S columns [64, 96) that it reads here, and it signals in turn.
        named_bar_arrive(half == 0 ? pair_bar : pair_bar2, 64);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int ch = 2 * half + cc;
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
          for (int q = 0; q < 32; q += 2) pk_keep[cc][q >> 1] = pack_bf16x2(pf[cc][q], pf[cc][q + 1]);
        }
      }
      if (half == 0) {
        tmem_st_x16(tmem + lane_addr + kColS + 16 * 0, pk_keep[0]);
        tmem_st_x16(tmem + lane_addr + kColS + 16 * 1, pk_keep[1]);
      }
      if (half == 1) {
        named_bar_sync(pair_bar, 64);
        tmem_st_x16(tmem + lane_addr + kColS + 16 * 2, pk_keep[0]);
        tmem_st_x16(tmem + lane_addr + kColS + 16 * 3, pk_keep[1]);
      }
      tc_fence_before();
      signal_leader(bP, false);        // dV may use P now
      // ---- dS = P o (dP - D), once dP is ready
      if (ok) ok = wait(bDP, it);
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
      uint32_t dpv[64];
      tmem_ld_x64(tmem + lane_addr + kColDP + 64 * half, dpv);
      uint32_t dsk[2][16];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int ch = 2 * half + cc;
        uint32_t (&dk)[16] = dsk[cc];
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
      }
      // dS^T (bf16 pairs) into tensor memory over the dead S columns [64, 128)
      if (half == 0) named_bar_sync(pair_bar2, 64);
      tmem_st_x16(tmem + lane_addr + kColDS + 32 * half, dsk[0]);
      tmem_st_x16(tmem + lane_addr + kColDS + 32 * half + 16, dsk[1]);
      tc_fence_before();
      signal_leader(bDST, false);      // dK may read dS^T now
      // The same values as rows of dS^T (key 128 rank + r, this warp's 64
      // queries, 4 KB per warp) into the dQ operand of the CTA owning query
      // tile i (CTA it & 1).  The owner writes them in place; CTA 1 (even
      // tiles) stages them in place as well and CTA 0 (odd tiles) in this
      // warp's drain box, and one bulk copy per warp sends them over.  The
      // buffers still hold the previous pair's dS until that pair's dQ
      // product has completed.
      const bool odd = it & 1;
      if (!odd && it >= 2) {
        if (ok) ok = wait(bDQ, (it >> 1) - 1);
        ok = __all_sync(0xffffffffu, ok);
      }
      const bool local = static_cast<uint32_t>(odd) == rank;
      const uint32_t rows_off = kDS + half * kDSPanel + (128 * rank + 32 * quad) * 128;
      const uint32_t box_off = kDrain + (half * 4 + quad) * 4096;
      const bool boxed = !local && rank == 0;
      if (boxed) {
        if (lane == 0) bulk_wait_group_read<0>();   // the box's last partial dQ has been read
        __syncwarp();
      }
      {
        uint8_t* rowp = smem + (boxed ? box_off : rows_off) + lane * 128;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
#pragma unroll
          for (int u = 0; u < 4; ++u)
            *reinterpret_cast<uint4*>(rowp + (((cc * 4 + u) ^ (lane & 7)) * 16)) =
                make_uint4(dsk[cc][4 * u], dsk[cc][4 * u + 1], dsk[cc][4 * u + 2], dsk[cc][4 * u + 3]);
      }
      fence_async_smem();
      if (!local) {
        __syncwarp();
        if (lane == 0)
          bulk_copy_to_peer(map_shared(sb + rows_off, rank ^ 1u), sb + (boxed ? box_off : rows_off), 4096,
                            map_shared(bar(bDSIn), rank ^ 1u));
      }
      // this CTA's rows of dS_i are in place (or on their way, counted on bDSIn)
      signal_leader(odd ? bDS1 : bDS0, local);
      if (!odd && it >= 2) drain((it >> 1) - 1, ok);   // the previous pair's partial dQ
    }
    if (n_it > 0) {                                     // the last pair's
      const int m = (n_it - 1) >> 1;
      if (ok) ok = wait(bDQ, m);
      ok = __all_sync(0xffffffffu, ok);
      drain(m, ok);
    }
    // ----------------------------------------------------- dK, dV epilogue
    bool ready = ok;
    if (n_it > 0 && ready) ready = wait(bAcc, 0);
    ready = __all_sync(0xffffffffu, ready);
    if (n_it == 0 || ready) {
      if (n_it > 0) tc_fence_after();
      // Each warp owns 32 key rows x 32 columns of dV and of dK; its rows go
      // through its own slice of the (now unused) dS^T buffer so that the
      // global stores cover whole 128-byte lines.
      constexpr int kCpr = D / 16;
      constexpr int kRowsPerStore = 32 / kCpr;
      uint8_t* slice = smem + kDS + (warp - 2) * (32 * D);
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
          const int key = jr * kBM + quad * 32 + rr;
          const uint4 w = *reinterpret_cast<const uint4*>(slice + rr * (D / 2 * 2) + ((cc ^ (rr % kCpr)) * 16));
          if (key < p.N_kv) *reinterpret_cast<uint4*>(outp + static_cast<size_t>(key) * D + cc * 8) = w;
        }
      }
    }
    if (lane == 0) bulk_wait_group0();             // this warp's reductions have landed
  }

  // Neither CTA leaves (or releases the pair's tensor memory) while the
  // other may still write into its shared memory or read its operands.
  __syncwarp();
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

}  // namespace bwd_pair
}  // namespace fa
