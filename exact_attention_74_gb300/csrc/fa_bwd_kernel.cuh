// fa_bwd_kernel.cuh -- backward exact attention for sm_103a.
//
// The backward pass recomputes S and P from the saved LSE instead of storing
// them ("FlashAttention: GPUメモリ階層を活用したアテンション最適化の分析" §7.2)
// and keeps its intermediates in tensor memory ("論文解説: FlashAttention-4 —
// Algorithm and Kernel Pipelining Co-Design for Asymmetric Hardware Scaling",
// Backwardパスの最適化).  With D_i = sum_c dO_ic O_ic it forms
//   P = exp(scale q.k - LSE),  dP = dO V^T,  dS = P o (dP - D),
//   dV = P^T dO,  dK = scale dS^T Q,  dQ = scale dS K.
//
// Three kernels:
//   prep  -- per query row: D, LSE * log2(e) (both padded to a multiple of 128
//            rows per head: padding rows get D = 0, LSE = +inf so their P is 0),
//            the per-tile counters and the CTA ticket; in the unordered mode it
//            also clears the fp32 dQ accumulator (the fixed-order mode's first
//            partial of each query tile is stored, not added).
//   main  -- one CTA per (128-key tile, batch*head), K and V resident in shared
//            memory, looping over the query tiles that can see its keys
//            (causal: only tiles at or below the diagonal):
//              warp 0    TMA producer (Q, dO tiles, LSE and D rows, 2 stages);
//                        before refilling a stage it issues the TMA reduce-adds
//                        of the dQ partial the compute warps staged there
//              warp 1    MMA issuer, per query tile i, in this order:
//                          dV += P^T dO          once P_i is in tensor memory
//                          dQ_i = dS K           once dS_i is in shared memory
//                          dK += dS^T Q          once dS^T_i is in tensor memory
//                          S^T_{i+1} = K Q^T     (overwrites P_i after dV read it)
//                          dP^T_{i+1} = V dO^T   once dQ_i has left tensor memory
//                        so dV overlaps the dS work, and once dK is done
//                        tile i's Q and dO are dead and hold the drain of dQ_i
//                        (the next tile's Q must arrive before its S, so the
//                        S product stays after dK)
//              warps 2-9 two warps per tensor-memory lane quarter (one key
//                        row per thread), each warp of a pair on half of the
//                        128 query columns: P (as soon as S is ready) back
//                        into tensor memory, then dS (once dP is ready) into
//                        shared memory (128-byte swizzle); then the same warps
//                        drain their half of the partial dQ: tensor memory ->
//                        registers -> tile i's dead Q/dO buffers in the TMA
//                        layout, handed to the producer, which adds it into
//                        the fp32 accumulator with TMA reduce-adds
//            dK and dV stay in tensor memory for the whole loop and are
//            written once at the end.  CTAs number themselves with a ticket
//            when they start and take their (key tile, head) from it.
//   convert -- dQ = bf16(scale * accumulator).
// Tensor-memory columns: S^T [0,128), over which P^T [0,64) and dS^T
// [64,128) land as bf16 pairs (the A operands of dV and dK); dP^T and then
// the partial dQ [128,256); dV [256,256+D); dK [256+D,256+2D).
#pragma once

#include <cuda_bf16.h>

#include "fa_internal.h"
#include "ptx.cuh"
#include "exp2.cuh"

namespace fa {
namespace bwd {

constexpr int kBM = 128;          // keys per CTA
constexpr int kBN = 128;          // queries per step
constexpr int kThreads = 320;
constexpr int kPanel = 128 * 128; // 128 rows x 128 B swizzle panel

template <int D>
struct Cfg {
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kK = 0;
  static constexpr int kV = kTile;
  static constexpr int kStage0 = 2 * kTile;
  static constexpr int kStageBytes = 2 * kTile + 1024;    // Q, dO, lse2[128], delta[128]
  static constexpr int kDS = kStage0 + 2 * kStageBytes;   // dS^T tile, 2 panels of 128 keys x 64 queries
  static constexpr int kBar = kDS + 2 * kPanel;
  // barrier indices
  static constexpr int kKVFull = 0, kQFull = 1, kStaged = 3, kSFull = 5, kPFull = 6, kDQFull = 7,
                       kDQFree = 8, kAccFull = 9, kDPFull = 10, kDOFull = 11, kDSFull = 13, kDSTFull = 14,
                       kStagedQ = 15, kNumBars = 17;
  static constexpr int kMisc = kBar + 8 * kNumBars;
  static constexpr int kSmem = kMisc + 16;
  static constexpr uint32_t kColS = 0, kColDS = 64, kColDP = 128, kColDV = 256, kColDK = 256 + D;
  static constexpr uint32_t kTmemCols = 512;
  static __device__ constexpr int q_off(int s) { return kStage0 + s * kStageBytes; }
  static __device__ constexpr int do_off(int s) { return kStage0 + s * kStageBytes + kTile; }
  static __device__ constexpr int lse_off(int s) { return kStage0 + s * kStageBytes + 2 * kTile; }
  static __device__ constexpr int dlt_off(int s) { return kStage0 + s * kStageBytes + 2 * kTile + 512; }
};

struct Params {
  float* dq_acc;
  unsigned* ticket;      // CTAs number themselves in the order they start
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  const float* lse2;     // [BH, nq_pad]
  const float* delta;    // [BH, nq_pad]
  unsigned* counters;    // [BH, n_q_tiles]: dQ partials added so far (deterministic order)
  int BH, N_q, N_kv, nq_pad, causal, deterministic;
  int n_q_tiles, n_kv_tiles;
  int n_sms;             // CTAs resident at once (one per SM)
  float c;               // scale * log2(e)
  float scale;
  DevCtl ctl;
};

// Logical CTA index b -> (key tile j, batch*head).  Head-major: the CTAs
// resident at one time cover only a few heads, so their fp32 dQ
// accumulators (and Q, dO tiles) stay in L2; within a head, key tile 0 runs
// first (with a causal mask it sees the most query tiles).  In the
// fixed-order mode each query tile takes its partials in decreasing key-tile
// order, so key tiles run from the last one, and b is a ticket each CTA
// draws when it starts: every CTA a CTA waits for drew a smaller ticket, so
// it has already started (and waits for nobody after it), whatever order the
// hardware dispatches CTAs in and whatever else runs on the GPU.  Without a
// mask every query tile takes all key tiles' partials, so a head's CTAs
// running side by side would each wait on the one just ahead: a group of
// kDetGroup heads is interleaved key tile by key tile, so one wave holds a
// few consecutive key tiles of each head of the group and most of a CTA's
// predecessors finished a wave earlier.  (With a causal mask the later key
// tiles see fewer query tiles and finish early by themselves.)
constexpr int kDetGroup = 16;

template <bool DET>
__device__ __forceinline__ void block_tile(const Params& p, int b, int& j, int& bh) {
  if (!DET || p.causal) {
    const int jj = b % p.n_kv_tiles;
    j = DET ? p.n_kv_tiles - 1 - jj : jj;
    bh = b / p.n_kv_tiles;
    return;
  }
  const int per_group = kDetGroup * p.n_kv_tiles;
  const int g = b / per_group;
  const int rem = b - g * per_group;
  const int heads = min(kDetGroup, p.BH - g * kDetGroup);   // the last group may be smaller
  j = p.n_kv_tiles - 1 - rem / heads;
  bh = g * kDetGroup + rem % heads;
}

// ------------------------------------------------------------------- prep

template <int D>
__global__ void __launch_bounds__(256)
prep_kernel(const __nv_bfloat16* __restrict__ O, const __nv_bfloat16* __restrict__ dO,
            const float* __restrict__ lse, float* __restrict__ lse2, float* __restrict__ delta,
            float* __restrict__ dq_acc, unsigned* __restrict__ counters, unsigned* __restrict__ ticket,
            int clear_acc, int BH, int N_q, int nq_pad) {
  // A row of O (and of dO) is D bf16 = L 16-byte pieces, one per lane; a warp
  // takes 32 / L rows at a time and keeps kU such groups of loads in flight.
  constexpr int L = D / 8;
  constexpr int kRows = 32 / L;
  constexpr int kU = 4;
  const int lane = threadIdx.x & 31;
  const int sub = lane / L;               // row of the group
  const int li = lane % L;                // 16-byte piece of the row
  if (blockIdx.x == 0 && threadIdx.x == 0) *ticket = 0u;
  const long long rows = static_cast<long long>(BH) * nq_pad;
  const long long wpb = blockDim.x / 32;
  const long long step = static_cast<long long>(gridDim.x) * wpb * kRows * kU;
  for (long long r0 = (static_cast<long long>(blockIdx.x) * wpb + threadIdx.x / 32) * kRows * kU; r0 < rows;
       r0 += step) {
    uint4 a[kU], b[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const long long r = r0 + u * kRows + sub;
      const int bh = static_cast<int>(r / nq_pad);
      const int q = static_cast<int>(r % nq_pad);
      a[u] = b[u] = make_uint4(0u, 0u, 0u, 0u);
      if (r < rows && q < N_q) {
        const size_t off = (static_cast<size_t>(bh) * N_q + q) * D + li * 8;
        a[u] = *reinterpret_cast<const uint4*>(O + off);
        b[u] = *reinterpret_cast<const uint4*>(dO + off);
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const long long r = r0 + u * kRows + sub;
      const int bh = static_cast<int>(r / nq_pad);
      const int q = static_cast<int>(r % nq_pad);
      const uint32_t aw[4] = {a[u].x, a[u].y, a[u].z, a[u].w}, bw[4] = {b[u].x, b[u].y, b[u].z, b[u].w};
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc = fmaf(__uint_as_float(aw[e] << 16), __uint_as_float(bw[e] << 16), acc);
        acc = fmaf(__uint_as_float(aw[e] & 0xffff0000u), __uint_as_float(bw[e] & 0xffff0000u), acc);
      }
#pragma unroll
      for (int o = L / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (r >= rows) continue;
      if (li == 0) {
        if ((q & 127) == 0) counters[r >> 7] = 0u;   // one per 128-row query tile
        if (q < N_q) {
          delta[r] = acc;
          lse2[r] = lse[static_cast<size_t>(bh) * N_q + q] * 1.4426950408889634f;
        } else {
          delta[r] = 0.f;
          lse2[r] = INFINITY;
        }
      }
      if (clear_acc && q < N_q) {
        float4* row = reinterpret_cast<float4*>(dq_acc + (static_cast<size_t>(bh) * N_q + q) * D);
#pragma unroll
        for (int k = 0; k < D / 4 / L; ++k) row[li + k * L] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
}

// ---------------------------------------------------------------- convert

__global__ void __launch_bounds__(256)
convert_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dq, long long n8, float scale) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
    uint4 w;
    w.x = pack_bf16x2(a.x * scale, a.y * scale);
    w.y = pack_bf16x2(a.z * scale, a.w * scale);
    w.z = pack_bf16x2(b.x * scale, b.y * scale);
    w.w = pack_bf16x2(b.z * scale, b.w * scale);
    reinterpret_cast<uint4*>(dq)[i] = w;
  }
}

// ------------------------------------------------------------------- main

// DET: the fixed-order (bit-reproducible) dQ reduction, compiled as its own
// instance so that the unordered kernel carries none of its code.
template <int D, bool DET>
__global__ void __launch_bounds__(kThreads, 1)
main_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
            const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
            const __grid_constant__ CUtensorMap tmDQ, const Params p) {
  using C = Cfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  if (sb & 1023u) {   // operand atoms need 1024-byte alignment
    if (threadIdx.x == 0) atomicOr(p.ctl.status, kStatusLaunchConfig);
    return;
  }
  auto bar = [&](int i) -> uint32_t { return sb + C::kBar + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMisc + 4);
  int* logical_slot = reinterpret_cast<int*>(smem + C::kMisc + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    // the ticket (its latency overlaps the set-up below)
    const int b = static_cast<int>(atomicAdd(p.ticket, 1u));
    mbar_init(bar(C::kKVFull), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::kQFull + s), 1);      // Q tile + LSE and D rows
      mbar_init(bar(C::kDOFull + s), 1);     // dO tile
      mbar_init(bar(C::kStaged + s), 8);       // one arrive per compute warp once its dQ boxes are staged
      mbar_init(bar(C::kStagedQ + s), 8);      // ... once its boxes in the Q buffer are
    }
    mbar_init(bar(C::kSFull), 1);
    mbar_init(bar(C::kDPFull), 1);
    mbar_init(bar(C::kPFull), 256);
    mbar_init(bar(C::kDSFull), 256);
    mbar_init(bar(C::kDSTFull), 256);
    mbar_init(bar(C::kDQFull), 1);
    mbar_init(bar(C::kDQFree), 256);
    mbar_init(bar(C::kAccFull), 1);
    *abort_flag = 0;
    mbar_init_fence();
    *logical_slot = b;
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
  __syncwarp();   // warps whose lane 0 ran a role alone arrive whole
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int logical = *logical_slot;
  int j, bh;
  block_tile<DET>(p, logical, j, bh);
  const int i0 = p.causal ? j : 0;                  // first query tile that sees these keys
  const int n_it = max(0, p.n_q_tiles - i0);

  if (n_it > 0 && warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmdO);
      mbar_arrive_expect_tx(bar(C::kKVFull), 2 * C::kTile);
      for (int pn = 0; pn < D / 64; ++pn) {
        tma_load_3d(sb + C::kK + pn * kPanel, &tmK, bar(C::kKVFull), pn * 64, j * kBM, bh);
        tma_load_3d(sb + C::kV + pn * kPanel, &tmV, bar(C::kKVFull), pn * 64, j * kBM, bh);
      }
      const uint64_t keep = l2_policy_evict_last();
      constexpr int kBoxes = D / 64;            // 32-column boxes per compute warp
      // Fixed order: once a partial has landed, the next key tile may add
      // into that query tile.  The landing wait is taken after this step's
      // loads are issued, so it overlaps them instead of delaying them.
      // The count only has to order the next key tile's reduce-add after
      // this one at L2, where both the partials and the count are applied:
      // the bulk group has completed (L2 has acknowledged this partial)
      // before the relaxed add on the count is even issued, and the next key
      // tile issues its partial only after it has read the raised count.
      // This leans on that completion, not on a release in the PTX memory
      // model's sense: a GPU-scope release waits behind the loads just
      // issued and cost the fixed-order mode a tenth of its speed.
      unsigned* release_cnt = nullptr;
      auto release = [&] {
        if (release_cnt == nullptr) return;
        bulk_wait_group0();
        fence_proxy_async_global();
        red_relaxed_gpu_add(release_cnt, 1u);
        release_cnt = nullptr;
      };
      for (int t = 0; t < n_it + 2; ++t) {
        const int s = t & 1;
        if (t >= 2) {
          // Tile t-2 staged its partial dQ in stage s (its Q and dO were no
          // longer read): add it into the accumulator in two groups, the
          // boxes held in the Q buffer first (the compute warps stage those
          // first and signal them on their own: the next Q waits on them),
          // and refill each buffer as soon as its boxes have been read.
          if (!mbar_wait(bar(C::kStagedQ + s), ((t - 2) >> 1) & 1, p.ctl, abort_flag)) break;
          const int ip = i0 + t - 2;
          unsigned* cnt = p.counters + static_cast<size_t>(bh) * p.n_q_tiles + ip;
          bool first = false;     // fixed order: the first partial of a query tile is stored
          if constexpr (DET) {
            // key tiles above this one (up to the last that sees query tile ip) add first
            const int top = p.causal ? min(ip, p.n_kv_tiles - 1) : p.n_kv_tiles - 1;
            first = j == top;
            if (!wait_counter(cnt, static_cast<unsigned>(top - j), p.ctl, abort_flag)) break;
            fence_proxy_async_global();
          }
          // box (hf, c, rk): columns hf * D/2 + 32 c, rows 32 rk of the tile,
          // at q_off + c * kTile + (4 hf + rk) * 4 KB; group c
          for (int c = 0; c < 2; ++c) {
            if (c == 1 && !mbar_wait(bar(C::kStaged + s), ((t - 2) >> 1) & 1, p.ctl, abort_flag)) break;
            if (c < kBoxes)
              for (int hf = 0; hf < 2; ++hf)
                for (int rk = 0; rk < 4; ++rk) {
                  const uint32_t src = sb + C::q_off(s) + c * C::kTile + (hf * 4 + rk) * 4096;
                  const int x = hf * (D / 2) + 32 * c, y = ip * kBN + rk * 32;
                  if (first) tma_store_3d(&tmDQ, src, x, y, bh);
                  else tma_reduce_add_3d(&tmDQ, src, x, y, bh);
                }
            bulk_commit_group();
          }
          if (*abort_flag) break;
          if constexpr (DET) release_cnt = cnt;
        }
        if (t == max(0, n_it - 4)) {
          // The CTA that this SM (or another) runs one wave later reads a
          // K/V tile nobody has touched yet: start it towards L2 now.
          const int nb = logical + p.n_sms;
          if (nb < static_cast<int>(gridDim.x)) {
            int nj, nbh;
            block_tile<DET>(p, nb, nj, nbh);
            for (int pn = 0; pn < D / 64; ++pn) {
              tma_prefetch_l2_3d(&tmK, pn * 64, nj * kBM, nbh);
              tma_prefetch_l2_3d(&tmV, pn * 64, nj * kBM, nbh);
            }
          }
        }
        if (t >= n_it) {
          if constexpr (DET) release();
          continue;
        }
        const int i = i0 + t;
        if (t >= 2) bulk_wait_group_read<1>();    // Q-buffer boxes read
        const uint32_t fq = bar(C::kQFull + s);
        mbar_arrive_expect_tx(fq, C::kTile + 1024);
        for (int pn = 0; pn < D / 64; ++pn)
          tma_load_3d_hint(sb + C::q_off(s) + pn * kPanel, &tmQ, fq, pn * 64, i * kBN, bh, keep);
        const size_t row = static_cast<size_t>(bh) * p.nq_pad + static_cast<size_t>(i) * kBN;
        bulk_load(sb + C::lse_off(s), p.lse2 + row, 512, fq);
        bulk_load(sb + C::dlt_off(s), p.delta + row, 512, fq);
        if (t >= 2) bulk_wait_group_read<0>();    // dO-buffer boxes read
        const uint32_t fd = bar(C::kDOFull + s);
        mbar_arrive_expect_tx(fd, C::kTile);
        for (int pn = 0; pn < D / 64; ++pn)
          tma_load_3d_hint(sb + C::do_off(s) + pn * kPanel, &tmdO, fd, pn * 64, i * kBN, bh, keep);
        if constexpr (DET) release();
      }
      if constexpr (DET) release();
      bulk_wait_group0();                       // every reduction has landed
    }
  } else if (n_it > 0 && warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16(kBM, kBN, false, false);
      constexpr uint32_t idKV = idesc_bf16(kBM, D, false, true);
      constexpr uint32_t idQ = idesc_bf16(kBN, D, true, true);
      const uint32_t sK = sb + C::kK, sV = sb + C::kV, sDS = sb + C::kDS;
      auto issue_S = [&](int st) {       // S^T = K Q^T
        const uint32_t sQ = sb + C::q_off(st);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * kPanel + (k & 3) * 32;
          mma_ss(tmem + C::kColS, sdesc_sw128(sK + off, 0, 1024), sdesc_sw128(sQ + off, 0, 1024), idS, k > 0);
        }
      };
      auto issue_dP = [&](int st) {      // dP^T = V dO^T
        const uint32_t sdO = sb + C::do_off(st);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * kPanel + (k & 3) * 32;
          mma_ss(tmem + C::kColDP, sdesc_sw128(sV + off, 0, 1024), sdesc_sw128(sdO + off, 0, 1024), idS, k > 0);
        }
      };
      bool ok = mbar_wait(bar(C::kKVFull), 0, p.ctl, abort_flag);
      if (ok) ok = mbar_wait(bar(C::kQFull + 0), 0, p.ctl, abort_flag);
      if (ok) {
        tc_fence_after();
        issue_S(0);
        tc_commit(bar(C::kSFull));
        ok = mbar_wait(bar(C::kDOFull + 0), 0, p.ctl, abort_flag);
      }
      if (ok) {
        tc_fence_after();
        issue_dP(0);
        tc_commit(bar(C::kDPFull));
      }
      for (int it = 0; it < n_it && ok; ++it) {
        const int s = it & 1;
        const uint32_t sQ = sb + C::q_off(s), sdO = sb + C::do_off(s);
        const bool next = it + 1 < n_it;
        const int s1 = (it + 1) & 1;
        ok = mbar_wait(bar(C::kPFull), it & 1, p.ctl, abort_flag);   // P_i in tensor memory
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < kBN / 16; ++k) {   // dV += P^T dO
          mma_ts(tmem + C::kColDV, tmem + C::kColS + 8 * k, sdesc_sw128(sdO + k * 2048, kPanel, 1024), idKV,
                 (it > 0 || k > 0) ? 1u : 0u);
        }
        ok = mbar_wait(bar(C::kDSFull), it & 1, p.ctl, abort_flag);  // dS_i in shared memory
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < kBM / 16; ++k) {   // dQ_i = dS K  (unscaled partial)
          mma_ss(tmem + C::kColDP, sdesc_sw128(sDS + k * 2048, kPanel, 1024),
                 sdesc_sw128(sK + k * 2048, kPanel, 1024), idQ, k > 0);
        }
        ok = mbar_wait(bar(C::kDSTFull), it & 1, p.ctl, abort_flag); // dS^T_i in tensor memory
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < kBN / 16; ++k) {   // dK += dS^T Q  (unscaled; dS^T from tensor memory)
          mma_ts(tmem + C::kColDK, tmem + C::kColDS + 8 * k, sdesc_sw128(sQ + k * 2048, kPanel, 1024), idKV,
                 (it > 0 || k > 0) ? 1u : 0u);
        }
        // dQ_i is ready and this stage's Q and dO are no longer read: the
        // drain may stage dQ_i in them
        tc_commit(bar(C::kDQFull));
        if (next) {                             // S of the next tile (P_i was consumed by dV first)
          ok = mbar_wait(bar(C::kQFull + s1), ((it + 1) >> 1) & 1, p.ctl, abort_flag);
          if (!ok) break;
          tc_fence_after();
          issue_S(s1);
          tc_commit(bar(C::kSFull));
        }
        if (next) {                             // dP of the next tile once dQ_i is drained
          ok = mbar_wait(bar(C::kDOFull + s1), ((it + 1) >> 1) & 1, p.ctl, abort_flag);
          if (ok) ok = mbar_wait(bar(C::kDQFree), it & 1, p.ctl, abort_flag);
          if (!ok) break;
          tc_fence_after();
          issue_dP(s1);
          tc_commit(bar(C::kDPFull));
        }
      }
      if (ok) tc_commit(bar(C::kAccFull));
    }
  } else if (warp >= 2) {
    // ------------------------------------------ P and dS rows, dQ drainage
    const int rank = warp & 3;               // tensor-memory lane quarter
    const int half = (warp - 2) >> 2;        // query columns [64 half, 64 half + 64)
    const int r = rank * 32 + lane;          // key row (and dQ query row) within the tile
    const int kg = j * kBM + r;              // global key index
    const uint32_t lane_addr = static_cast<uint32_t>(rank * 32) << 16;
    const bool key_ok = kg < p.N_kv;
    const float2 c2 = make_float2(p.c, p.c);
    const uint32_t pair_bar = 1 + rank;      // named barriers of the two warps of this lane quarter:
    const uint32_t pair_bar2 = 5 + rank;     // first -> second warp (S read), second -> first
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int s = it & 1;
      const int i = i0 + it;
      bool w = mbar_wait(bar(C::kSFull), it & 1, p.ctl, abort_flag);
      if (w) w = mbar_wait(bar(C::kQFull + s), (it >> 1) & 1, p.ctl, abort_flag);
      ok = __all_sync(0xffffffffu, w);
      if (!ok) {
        named_bar_arrive(half == 0 ? pair_bar : pair_bar2, 64);   // the other warp may wait on it
        break;
      }
      tc_fence_after();
      const float* lse_s = reinterpret_cast<const float*>(smem + C::lse_off(s));
      const float* dlt_s = reinterpret_cast<const float*>(smem + C::dlt_off(s));
      // queries q with q_g < k_g are masked (causal); only the diagonal tile has
      // any, and only the last key tile has keys past N_kv
      const int lim = (p.causal && i == j) ? r : 0;
      const bool masked = __any_sync(0xffffffffu, lim > 0 || !key_ok);
      // ---- P = 2^(S c - LSE log2 e), as soon as S is ready
      float pf[2][32];
      uint32_t pk_keep[2][16];
      {
        // both 32-query chunks of this warp in one tensor-memory round trip
        uint32_t sv[64];
        tmem_ld_x64(tmem + lane_addr + C::kColS + 64 * half, sv);
        // P of chunk ch lands on the S columns of queries [16 ch, 16 ch + 16),
        // which the first warp of the pair has now read: the second warp
        // writes after this signal.
        // The second warp's dS^T later lands on the S columns [64, 96) that
        // the second warp reads: it signals once it has read them.
        named_bar_arrive(half == 0 ? pair_bar : pair_bar2, 64);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int ch = 2 * half + cc;        // 32-query chunk
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
        tmem_st_x16(tmem + lane_addr + C::kColS + 16 * 0, pk_keep[0]);
        tmem_st_x16(tmem + lane_addr + C::kColS + 16 * 1, pk_keep[1]);
      }
      if (half == 1) {
        named_bar_sync(pair_bar, 64);
        tmem_st_x16(tmem + lane_addr + C::kColS + 16 * 2, pk_keep[0]);
        tmem_st_x16(tmem + lane_addr + C::kColS + 16 * 3, pk_keep[1]);
      }
      tc_fence_before();
      mbar_arrive(bar(C::kPFull));            // dV may use P now
      // ---- dS = P o (dP - D), once dP is ready
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kDPFull), it & 1, p.ctl, abort_flag));
      if (!ok) break;
      tc_fence_after();
      uint32_t dpv[64];
      tmem_ld_x64(tmem + lane_addr + C::kColDP + 64 * half, dpv);   // both chunks at once
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
        // dS^T row r, queries 32ch..32ch+31: panel ch/2, 16-byte chunks (ch&1)*4 + u
        uint8_t* rowp = smem + C::kDS + (ch >> 1) * kPanel + r * 128;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int chunk = ((ch & 1) * 4 + u) ^ (r & 7);
          *reinterpret_cast<uint4*>(rowp + chunk * 16) =
              make_uint4(dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
        }
      }
      fence_async_smem();
      mbar_arrive(bar(C::kDSFull));           // dQ may read dS now
      // dS^T (bf16 pairs) also into tensor memory over the dead S columns
      // [64, 128), where dK reads it (queued after dQ, so this is off the
      // critical path): the first warp's half overwrites S columns the
      // second warp read, so it waits for that warp's signal.
      if (half == 0) named_bar_sync(pair_bar2, 64);
      tmem_st_x16(tmem + lane_addr + C::kColDS + 32 * half, dsk[0]);
      tmem_st_x16(tmem + lane_addr + C::kColDS + 32 * half + 16, dsk[1]);
      tc_fence_before();
      mbar_arrive(bar(C::kDSTFull));          // dK may read dS^T now
      // ---- drain this warp's half of the partial dQ (rows = queries of tile i)
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kDQFull), it & 1, p.ctl, abort_flag));
      if (!ok) break;
      tc_fence_after();
      constexpr int kBoxes = D / 64;          // 32-column boxes per warp
      uint32_t v[kBoxes][32];
      if constexpr (kBoxes == 2) {
        uint32_t vv[64];
        tmem_ld_x64(tmem + lane_addr + C::kColDP + half * (D / 2), vv);
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          v[0][u] = vv[u];
          v[1][u] = vv[32 + u];
        }
      } else {
        tmem_ld_x32(tmem + lane_addr + C::kColDP + half * (D / 2), v[0]);
      }
      tc_fence_before();
      mbar_arrive_relaxed(bar(C::kDQFree));   // the tensor-memory reads are complete
      // Stage each 32-row x 32-column fp32 box in tile i's dead Q/dO buffers,
      // laid out as TMA's 128-byte swizzle expects (row = lane, 16-byte chunk
      // j at j ^ (row & 7)); the producer adds the boxes into the accumulator.
      // Box c of this warp (columns half * D/2 + 32 c, rows 32 rank) goes to
      // q_off + c * kTile + (4 half + rank) * 4 KB: with d = 128 box 0 is in
      // the Q buffer and box 1 in the dO buffer, and the Q buffer's boxes are
      // signalled first, since the next Q tile waits for them to be read.
      const uint32_t stage = sb + C::q_off(s);
#pragma unroll
      for (int c = 0; c < kBoxes; ++c) {
        const uint32_t box = stage + c * C::kTile + (half * 4 + rank) * 4096;
        uint8_t* rowp = smem + (box - sb) + lane * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          *reinterpret_cast<uint4*>(rowp + ((u ^ (lane & 7)) * 16)) =
              make_uint4(v[c][4 * u], v[c][4 * u + 1], v[c][4 * u + 2], v[c][4 * u + 3]);
        if (c == 0) {
          fence_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(C::kStagedQ + s));
        }
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::kStaged + s));   // the producer reduces the rest
    }
    // ----------------------------------------------------- dK, dV epilogue
    bool ready = ok;
    if (n_it > 0 && ready) ready = mbar_wait(bar(C::kAccFull), 0, p.ctl, abort_flag);
    ready = __all_sync(0xffffffffu, ready);
    if (n_it == 0 || ready) {
      if (n_it > 0) tc_fence_after();
      // Each warp owns 32 key rows x D/2 columns of dV and of dK.  Its rows
      // go through its own slice of the (now unused) dS buffer, so that the
      // global stores cover whole 128-byte lines instead of one 16-byte
      // piece of 32 different rows.
      constexpr int kCpr = D / 16;                // 16-byte chunks per row slice
      constexpr int kRowsPerStore = 32 / kCpr;
      uint8_t* slice = smem + C::kDS + (warp - 2) * (32 * D);   // 32 rows x D/2 bf16
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        const float f = which == 0 ? 1.f : p.scale;
        uint32_t v[D / 2];
        if (n_it > 0) {
          const uint32_t col = (which == 0 ? C::kColDV : C::kColDK) + half * (D / 2);
          if constexpr (D == 128) tmem_ld_x64(tmem + lane_addr + col, v);
          else tmem_ld_x32(tmem + lane_addr + col, v);
        } else {
#pragma unroll
          for (int u = 0; u < D / 2; ++u) v[u] = 0u;
        }
        __syncwarp();                             // the previous output's reads are done
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
          const int rr = k * kRowsPerStore + lane / kCpr;    // row within the warp's 32
          const int cc = lane % kCpr;
          const int key = j * kBM + rank * 32 + rr;
          const uint4 w = *reinterpret_cast<const uint4*>(slice + rr * (D / 2 * 2) + ((cc ^ (rr % kCpr)) * 16));
          if (key < p.N_kv) *reinterpret_cast<uint4*>(outp + static_cast<size_t>(key) * D + cc * 8) = w;
        }
      }
    }
  }

  __syncwarp();   // warps whose lane 0 ran a role alone arrive whole
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D>
cudaError_t launch(const BwdLaunch& a) {
  using C = Cfg<D>;
  const int nq_pad = (a.N_q + kBN - 1) / kBN * kBN;
  // workspace: dq_acc [BH*N_q*D] (rounded to 256 B), then delta, lse2 [BH*nq_pad] each
  float* lse2 = a.delta + static_cast<size_t>(a.BH) * nq_pad;
  {
    const long long rows = static_cast<long long>(a.BH) * nq_pad;
    const long long blocks = (rows + 8 * 4 * (256 / D) - 1) / (8 * 4 * (256 / D));   // rows per block: 8 warps x 4 groups
    prep_kernel<D><<<static_cast<unsigned>(blocks < 65535 * 8 ? blocks : 65535 * 8), 256, 0, a.stream>>>(
        static_cast<const __nv_bfloat16*>(a.o), static_cast<const __nv_bfloat16*>(a.dO), a.lse, lse2, a.delta,
        a.dq_acc, a.counters, a.ticket, a.deterministic ? 0 : 1, a.BH, a.N_q, nq_pad);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  Params p;
  p.dq_acc = a.dq_acc;
  p.ticket = a.ticket;
  p.dk = static_cast<__nv_bfloat16*>(a.dk);
  p.dv = static_cast<__nv_bfloat16*>(a.dv);
  p.lse2 = lse2;
  p.delta = a.delta;
  p.counters = a.counters;
  p.deterministic = a.deterministic;
  p.BH = a.BH;
  p.N_q = a.N_q;
  p.N_kv = a.N_kv;
  p.nq_pad = nq_pad;
  p.causal = a.causal;
  p.n_q_tiles = nq_pad / kBN;
  p.n_kv_tiles = (a.N_kv + kBM - 1) / kBM;
  p.c = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  p.scale = a.scale;
  p.ctl = a.ctl;
  p.n_sms = a.n_sms;
  auto kern = a.deterministic ? main_kernel<D, true> : main_kernel<D, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(p.n_kv_tiles) * p.BH;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  kern<<<static_cast<unsigned>(grid), kThreads, C::kSmem, a.stream>>>(a.tmQ, a.tmK, a.tmV, a.tmdO, a.tmDQ, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long n8 = static_cast<long long>(a.BH) * a.N_q * D / 8;
  const long long blocks = (n8 + 255) / 256;
  convert_kernel<<<static_cast<unsigned>(blocks < 8192 ? blocks : 8192), 256, 0, a.stream>>>(
      a.dq_acc, static_cast<__nv_bfloat16*>(a.dq), n8, a.scale);
  return cudaGetLastError();
}

}  // namespace bwd
}  // namespace fa
