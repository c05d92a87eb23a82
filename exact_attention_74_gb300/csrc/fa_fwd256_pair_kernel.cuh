// fa_fwd256_pair_kernel.cuh -- forward exact attention for head dimension 256
// on pairs of CTAs that share their tensor-core products (cta_group::2).
//
// One query tile's O takes half of tensor memory at d = 256, so a CTA owns
// one 128-row query tile, and each 128-key step streams K and V (128 KB)
// into its shared memory.  Two CTAs of a cluster own query tiles 2 qp and
// 2 qp + 1 of one (batch, head) and share every product as one M = 256 pair
// product ("論文解説: FlashAttention-4 — Algorithm and Kernel Pipelining
// Co-Design for Asymmetric Hardware Scaling", 2-CTA MMA mode): CTA r loads
// only keys [64 r, 64 r + 64) of K_j (the N half of S = Q K_j^T it supplies)
// and channels [128 r, 128 r + 128) of V_j (the N half of P_j V_j), 64 KB
// per step, half of what one CTA alone streams.
//
//   tensor memory   (each CTA, its own 128 rows) S_j in one of two
//                   128-column buffers [0,128) / [128,256), P_j as bf16
//                   pairs over the first 64 columns of its buffer, O
//                   [256,512)
//   shared memory   Q (64 KB, resident) and a ring of five 32 KB slots, each
//                   one of this CTA's K or V halves, loaded K_0, then
//                   K_{j+1} ahead of V_j
//   warp 0          TMA producer (each CTA, its own halves)
//   warp 1          leader: the one issuing thread, in the order S_0, S_1,
//                   then per step O += P_j V_j (eight pair products, N = 256,
//                   P from each CTA's tensor memory) once both CTAs'
//                   softmax warps have written P_j, followed by S_{j+2}
//                   (sixteen pair products, N = 128) into the buffer P_j
//                   occupies; CTA 1: forwards each of its landed loads to
//                   the leader's barrier, which counts both CTAs
//   warps 2-5       softmax of this CTA's rows, one thread per row, the same
//                   online softmax with conditional rescaling as the
//                   single-CTA kernels (条件付きオンラインsoftmaxリスケーリング)
//
// One thread issues P V_j and then S_{j+2}, so the tensor core runs S_{j+2}
// after P V_j has read P_j without waiting for P V_j's completion: with S on
// a thread of its own, S_{j+2} had to wait for that completion, and the
// tensor core drained every step.  The leader's commits arrive on the same
// barrier in both CTAs, so each CTA waits only on its own barriers.  With a
// causal mask the pair runs the steps of its second tile; the first tile's
// last step is fully masked.
#pragma once

#include <cuda_bf16.h>

#include "exp2.cuh"
#include "fa_internal.h"
#include "ptx_pair.cuh"

namespace fa {
namespace fwd256p {

constexpr int D = 256;
constexpr int kBM = 128;                  // query rows per CTA (256 per pair)
constexpr int kBN = 128;                  // keys per step
constexpr int kThreads = 192;             // 6 warps
constexpr int kSlots = 5;                 // K/V ring
constexpr int kQPanel = 128 * 128;        // 128 rows x 128 B (64 bf16) swizzle panel
constexpr int kKPanel = 64 * 128;         // K half: 64 keys, 4 panels of 64 rows x 128 B
constexpr int kVPanel = 128 * 128;        // V half: 128 keys x 128 channels, 2 panels
constexpr int kQBytes = 4 * kQPanel;      // 64 KB
constexpr int kSlotBytes = 4 * kKPanel;   // 32 KB (= 2 * kVPanel)
constexpr int kQOff = 0;
constexpr int kKVOff = kQBytes;
constexpr int kBarOff = kKVOff + kSlots * kSlotBytes;
// barrier indices
constexpr int kQFull = 0;                 // Q in shared memory (leader: of both CTAs)
constexpr int kKVFull = 1;                // kSlots (leader: both CTAs' halves)
constexpr int kKVEmpty = 1 + kSlots;      // kSlots
constexpr int kSFull = 1 + 2 * kSlots;    // 2 (per S buffer)
constexpr int kPFull = 3 + 2 * kSlots;    // 2 (per S buffer; leader: both CTAs' P)
constexpr int kOFull = 5 + 2 * kSlots;
constexpr int kPVDone = 6 + 2 * kSlots;   // 2 (per S buffer): P V has read the buffer's P
constexpr int kDone = 8 + 2 * kSlots;     // leader: every product issued has completed
constexpr int kNumBars = 9 + 2 * kSlots;
constexpr int kMiscOff = kBarOff + 8 * kNumBars;   // tmem base, abort flag
constexpr int kSmemBytes = kMiscOff + 16;
// tensor-memory columns
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint16_t kBoth = 3;             // commit to both CTAs of the pair

struct Params {
  __nv_bfloat16* o;
  float* lse;
  int BH, N_q, N_kv, causal;
  int n_qtiles;   // ceil(N_q / 128)
  int n_pairs;    // ceil(n_qtiles / 2)
  int n_steps;    // ceil(N_kv / 128)
  float c;        // scale * log2(e)
  float tau;      // log2 units
  DevCtl ctl;
};

// K/V ring in load order: K_0, then K_{j+1} ahead of V_j, and V_{n-1} last.
__device__ __forceinline__ int k_load(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int v_load(int j, int n) { return j < n - 1 ? 2 * j + 2 : 2 * n - 1; }
__device__ __forceinline__ int ring_slot(int i) { return i % kSlots; }
__device__ __forceinline__ int ring_round(int i) { return i / kSlots; }

template <int EMU>
__device__ __forceinline__ float ex2_mix(float x, int col) {
  if ((col & 31) < EMU) return ex2_poly3(x);
  return ex2_hw(x);
}

template <int EMU>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
fwd256p_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  // the same offset in both CTAs, so both return here or neither does
  if (sb & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.ctl.status, kStatusLaunchConfig);
    return;
  }
  auto bar = [&](int i) -> uint32_t { return sb + kBarOff + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMiscOff + 4);
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const uint32_t peer_abort = map_shared(sb + kMiscOff + 4, rank ^ 1u);
  auto wait = [&](int b, int parity) -> bool {
    return pair_wait(bar(b), static_cast<uint32_t>(parity) & 1u, p.ctl, abort_flag, peer_abort);
  };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work: query tiles 2 qp + r of one (batch, head); causal grids run the
  // heaviest pairs (the last query rows) first.
  const int cid = static_cast<int>(blockIdx.x >> 1);
  int qp, bh;
  if (p.causal) {
    qp = p.n_pairs - 1 - cid / p.BH;
    bh = cid % p.BH;
  } else {
    qp = cid % p.n_pairs;
    bh = cid / p.n_pairs;
  }
  const int qbase = (2 * qp + static_cast<int>(rank)) * kBM;
  // key steps the pair sees (causal: keys up to the second tile's last row)
  const int n = p.causal ? min(p.n_steps, 2 * qp + 2) : p.n_steps;

  if (threadIdx.x == 0) {
    const uint32_t fed = leader ? 2u : 1u;   // the leader also counts CTA 1's forwarded loads
    mbar_init(bar(kQFull), fed);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(bar(kKVFull + s), fed);
      mbar_init(bar(kKVEmpty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(kSFull + b), 1);
      mbar_init(bar(kPFull + b), 8);        // one arrive per softmax warp of either CTA
      mbar_init(bar(kPVDone + b), 1);
    }
    mbar_init(bar(kOFull), 1);
    mbar_init(bar(kDone), 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
  __syncwarp();
  tc_fence_before();
  cluster_sync();                           // both CTAs' barriers initialised, tensor memory allocated
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmV);
      mbar_arrive_expect_tx(bar(kQFull), kQBytes);
      for (int pn = 0; pn < 4; ++pn)
        tma_load_3d(sb + kQOff + pn * kQPanel, &tmQ, bar(kQFull), pn * 64, qbase, bh);
      const uint64_t keep = l2_policy_evict_last();
      const int r = static_cast<int>(rank);
      for (int i = 0; i < 2 * n; ++i) {
        const int s = ring_slot(i);
        if (!wait(kKVEmpty + s, ring_round(i) + 1)) break;
        bool is_k;
        int step;
        if (i == 0) {
          is_k = true;
          step = 0;
        } else {
          const int m = i - 1, blk = m >> 1;
          is_k = blk < n - 1 && (m & 1) == 0;
          step = is_k ? blk + 1 : blk;
        }
        const uint32_t dst = sb + kKVOff + s * kSlotBytes;
        mbar_arrive_expect_tx(bar(kKVFull + s), kSlotBytes);
        if (is_k) {   // this CTA's 64 keys of K_step, all 256 channels
          for (int pn = 0; pn < 4; ++pn)
            tma_load_3d_hint(dst + pn * kKPanel, &tmK, bar(kKVFull + s), pn * 64, step * kBN + 64 * r, bh, keep);
        } else {      // the 128 keys of V_step, this CTA's 128 channels
          for (int pn = 0; pn < 2; ++pn)
            tma_load_3d_hint(dst + pn * kVPanel, &tmV, bar(kKVFull + s), 128 * r + 64 * pn, step * kBN, bh,
                             keep);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // --------------------------------------------- MMA issuer, leader
      constexpr uint32_t idS = idesc_bf16(2 * kBM, kBN, false, false);
      constexpr uint32_t idO = idesc_bf16(2 * kBM, D, false, true);
      auto slot_addr = [&](int i) { return sb + kKVOff + ring_slot(i) * kSlotBytes; };
      auto kv_wait = [&](int i) { return wait(kKVFull + ring_slot(i), ring_round(i)); };
      // S_j = Q K_j^T into S buffer j & 1
      auto issue_S = [&](int j) -> bool {
        const int ik = k_load(j);
        if (!kv_wait(ik)) return false;
        tc_fence_after();
        const uint32_t ka = slot_addr(ik);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t qa = sb + kQOff + (k >> 2) * kQPanel + (k & 3) * 32;
          const uint32_t kb = ka + (k >> 2) * kKPanel + (k & 3) * 32;
          mma_ss_pair(tmem + kColS + 128 * (j & 1), sdesc_sw128(qa, 0, 1024), sdesc_sw128(kb, 0, 1024), idS,
                      k > 0 ? 1u : 0u);
        }
        tc_commit_pair(bar(kSFull + (j & 1)), kBoth);
        tc_commit_pair(bar(kKVEmpty + ring_slot(ik)), kBoth);   // K_j read in both CTAs
        return true;
      };
      bool ok = wait(kQFull, 0);
      if (ok) ok = issue_S(0);
      if (ok && n > 1) ok = issue_S(1);
      for (int j = 0; j < n && ok; ++j) {   // O += P_j V_j, P_j over S buffer j & 1
        if (!(ok = wait(kPFull + (j & 1), j >> 1))) break;
        const int iv = v_load(j, n);
        if (!(ok = kv_wait(iv))) break;
        tc_fence_after();
        const uint32_t va = slot_addr(iv);
#pragma unroll
        for (int k = 0; k < kBN / 16; ++k)
          mma_ts_pair(tmem + kColO, tmem + kColS + 128 * (j & 1) + 8 * k, sdesc_sw128(va + k * 2048, kVPanel, 1024),
                      idO, (j > 0 || k > 0) ? 1u : 0u);
        tc_commit_pair(bar(kKVEmpty + ring_slot(iv)), kBoth);   // V_j read in both CTAs
        tc_commit_pair(bar(kPVDone + (j & 1)), kBoth);           // (and P V_j complete)
        // S_{j+2} overwrites P_j: issued after P V_j by the same thread, the
        // tensor core runs it after P V_j has read its operand
        if (j + 2 < n) ok = issue_S(j + 2);
      }
      if (ok) tc_commit_pair(bar(kOFull), kBoth);
      // every product issued completes before the pair's tensor memory is
      // released
      tc_commit_pair(bar(kDone), 1);
      wait(kDone, 0);
    } else if (lane == 0) {
      // ------------------------------------ CTA 1: forward its landed loads
      // (in load order; a slot is reloaded only after the leader has seen its
      // previous contents and issued the products that read them)
      bool ok = wait(kQFull, 0);
      if (ok) mbar_arrive_remote_relaxed(map_shared(bar(kQFull), 0));
      for (int i = 0; i < 2 * n && ok; ++i) {
        ok = wait(kKVFull + ring_slot(i), ring_round(i));
        if (ok) mbar_arrive_remote_relaxed(map_shared(bar(kKVFull + ring_slot(i)), 0));
      }
    }
  } else {
    // ------------------------------------------------------- softmax (2-5)
    const int quad = warp & 3;              // tensor-memory lane quarter
    const int r_in_tile = quad * 32 + lane;
    const int row = qbase + r_in_tile;
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tO = tmem + lane_addr + kColO;
    const float c = p.c;
    bool ok = true;
    float m_ref = -INFINITY;
    float l = 0.f;      // sum of the fp32 probabilities: gives the LSE
    float lr = 0.f;     // rounding residuals of the blocks' largest P
    const int key_lim = p.causal ? min(p.N_kv - 1, row) : p.N_kv - 1;   // last key this row sees
    for (int j = 0; j < n && ok; ++j) {
      const int b = j & 1;
      ok = __all_sync(0xffffffffu, wait(kSFull + b, j >> 1));
      if (!ok) break;
      tc_fence_after();
      const uint32_t tS = tmem + lane_addr + kColS + 128 * b;
      uint32_t s[128];
      tmem_ld_x128(tS, s);
      const int lim = key_lim - j * kBN;
      if (__any_sync(0xffffffffu, lim < kBN - 1)) {
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
        // P_{j-1} V_{j-1} may still be accumulating into O: wait for it
        ok = __all_sync(0xffffffffu, wait(kPVDone + ((j - 1) & 1), (j - 1) >> 1));
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
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
        pk[i] = pack_bf16x2(e0, e1);
      }
      tmem_st_x64(tS, pk);   // waits for its own stores
      tc_fence_before();
      __syncwarp();
      // one arrival per warp of either CTA on the leader's barrier
      if (lane == 0) {
        if (leader) mbar_arrive(bar(kPFull + b));
        else mbar_arrive_remote_relaxed(map_shared(bar(kPFull + b), 0));
      }
      l += (sum[0].x + sum[0].y) + (sum[1].x + sum[1].y);
      {
        // the block's largest P: with every exponential on the ex2 unit,
        // recomputed exactly as its element was (same fused multiply-add)
        const float pm = EMU > 0 ? pmax : ex2_hw(fmaf(mxs, c, -m_ref));
        const float pmr = __uint_as_float(pack_bf16x2(pm, pm) << 16);   // as rounded for P V
        lr += pmr - pm;
      }
    }
    // ------------------------------------------------------------- epilogue
    bool ready = ok && n > 0;
    if (ready) ready = wait(kOFull, 0);
    if (__all_sync(0xffffffffu, ready)) {
      tc_fence_after();
      const float inv_l = 1.f / (l + lr);
      __nv_bfloat16* orow = p.o + (static_cast<size_t>(bh) * p.N_q + row) * D;
#pragma unroll 1
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


  // Neither CTA leaves (or releases the pair's tensor memory) while the
  // other may still read its operands or arrive on its barriers.
  __syncwarp();
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

template <int EMU>
cudaError_t launch(const FwdLaunch& a) {
  Params p;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.BH = a.BH;
  p.N_q = a.N_q;
  p.N_kv = a.N_kv;
  p.causal = a.causal;
  p.n_qtiles = (a.N_q + kBM - 1) / kBM;
  p.n_pairs = (p.n_qtiles + 1) / 2;
  p.n_steps = (a.N_kv + kBN - 1) / kBN;
  p.c = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  p.tau = a.tau;
  p.ctl = a.ctl;
  auto kern = fwd256p_kernel<EMU>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  // two CTAs (one cluster) per pair of query tiles of every (batch, head)
  const long long grid = 2LL * p.n_pairs * p.BH;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  kern<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, a.stream>>>(a.tmQ, a.tmK, a.tmV, p);
  return cudaGetLastError();
}

inline cudaError_t launch_any(const FwdLaunch& a) {
  switch (a.emu_per_32) {
    case 0: return launch<0>(a);
    case 8: return launch<8>(a);
    case 16: return launch<16>(a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fwd256p
}  // namespace fa
