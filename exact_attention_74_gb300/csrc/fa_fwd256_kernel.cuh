// fa_fwd256_kernel.cuh -- forward exact attention for head dimension 256.
//
// At d = 256 one query tile's O already takes half of tensor memory (256
// fp32 columns), so the two-tile ping-pong of the d <= 128 kernel does not
// fit.  Instead one CTA owns one 128-row query tile and overlaps the work of
// consecutive key steps of that tile (128 keys per step):
//
//   tensor memory   S_j in one of two 128-column buffers [0,128) / [128,256),
//                   P_j as bf16 pairs over the first 64 columns of its
//                   buffer, O [256,512)
//   shared memory   Q (64 KB, resident) and a ring of five 32 KB slots, each
//                   holding half a key step: K_j's features 0-127 or
//                   128-255, V_j's keys 0-63 or 64-127
//   warp 0          TMA producer: Q once, then the half tiles: K_0, and
//                   from then on K_{j+1} ahead of V_j
//   warp 1          issues S_{j+1} = Q K_{j+1}^T (both operands in shared
//                   memory, N = 128) as soon as each half of K_{j+1} is in
//                   and P V_{j-1} has read its buffer, so the tensor core
//                   computes the next scores while the softmax of the
//                   current ones runs
//   warp 6          issues O += P_j V_j once P_j is written, half by half
//   warps 2-5       softmax, one thread per query row (one tensor-memory lane)
//
// Steps of 128 keys keep every product at the tensor core's full rate
// (products 64 columns wide run at two thirds of it), and half-tile slots
// let the next step's K stream in while the current step's products still
// read the other half: with whole 64 KB tiles in two slots, K_{j+1} could
// only load after S_j had finished.  The ring holds five halves, so the load
// order decides what waits: with K_{j+1} queued behind V_j its first half
// reused the slot of V_{j-1}'s second half and started only when P V_{j-1}
// had finished, exactly when S_{j+1} needed it; queued ahead of V_j it
// reuses a slot that P V_{j-2} released a step earlier, and the load
// latency hides behind the softmax.  With one thread issuing both streams,
// the next S waited behind that thread's wait for P and its P V products;
// on threads of their own, each goes out as soon as its inputs are ready.
//
// The per-row recurrence is the same online softmax in base 2 with the
// conditional rescaling of "論文解説: FlashAttention-4 — Algorithm and Kernel
// Pipelining Co-Design for Asymmetric Hardware Scaling" (条件付きオンライン
// softmaxリスケーリング) as the d <= 128 kernel, including the deferred
// normalisation by l plus each block's max-element rounding residual.  The
// rare O rescale must not race with the previous step's P V (queued after
// S_j), so it first waits for that product's completion barrier.
#pragma once

#include <cuda_bf16.h>

#include "exp2.cuh"
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace fwd256 {

constexpr int D = 256;
constexpr int kBM = 128;                  // query rows per CTA
constexpr int kBN = 128;                  // keys per step
constexpr int kThreads = 224;             // 7 warps
constexpr int kSlots = 5;                 // K/V ring of half tiles
constexpr int kQPanel = 128 * 128;        // 128 rows x 128 B (64 bf16) swizzle panel
constexpr int kKPanel = 128 * 128;        // K half tile: 2 panels of 128 rows x 128 B
constexpr int kVPanel = 64 * 128;         // V half tile: 4 panels of 64 rows x 128 B
constexpr int kQBytes = 4 * kQPanel;      // 64 KB
constexpr int kSlotBytes = 2 * kKPanel;   // 32 KB
constexpr int kQOff = 0;
constexpr int kKVOff = kQBytes;
constexpr int kBarOff = kKVOff + kSlots * kSlotBytes;
// barrier indices
constexpr int kQFull = 0;                 // Q tile in shared memory
constexpr int kKVFull = 1;                // kSlots
constexpr int kKVEmpty = 1 + kSlots;      // kSlots
constexpr int kSFull = 1 + 2 * kSlots;    // 2 (per S buffer)
constexpr int kPFull = 3 + 2 * kSlots;    // 2 (per S buffer)
constexpr int kOFull = 5 + 2 * kSlots;
constexpr int kPVDone = 6 + 2 * kSlots;   // 2 (per S buffer): P V has read the buffer's P
constexpr int kNumBars = 8 + 2 * kSlots;
constexpr int kMiscOff = kBarOff + 8 * kNumBars;   // tmem base, abort flag
constexpr int kSmemBytes = kMiscOff + 16 + 1024;   // + base alignment slack
// tensor-memory columns
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 256;
constexpr uint32_t kTmemCols = 512;

struct Params {
  __nv_bfloat16* o;
  float* lse;
  int BH, N_q, N_kv, causal;
  int n_qtiles;   // ceil(N_q / 128)
  int n_steps;    // ceil(N_kv / 128)
  float c;        // scale * log2(e)
  float tau;      // log2 units
  DevCtl ctl;
};

// K/V ring of half tiles, in load order: K_0's features 0-127 and 128-255,
// then per step j < n - 1 the two halves of K_{j+1} followed by V_j's keys
// 0-63 and 64-127, and last V_{n-1}'s halves.  K_j's half h is load
// 4j - 2 + h (h for j = 0); V_j's is 4j + 4 + h (4j + 2 + h for the last step).
__device__ __forceinline__ int k_load(int j, int h) { return j == 0 ? h : 4 * j - 2 + h; }
__device__ __forceinline__ int v_load(int j, int h, int n) { return (j < n - 1 ? 4 * j + 4 : 4 * j + 2) + h; }
__device__ __forceinline__ int ring_slot(int i) { return i % kSlots; }
__device__ __forceinline__ uint32_t ring_phase(int i) { return static_cast<uint32_t>((i / kSlots) & 1); }

template <int EMU>
__device__ __forceinline__ float ex2_mix(float x, int col) {
  if ((col & 31) < EMU) return ex2_poly3(x);
  return ex2_hw(x);
}

template <int EMU>
__global__ void __launch_bounds__(kThreads, 1)
fwd256_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
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

  // Work tile: one query tile of one (batch, head); causal grids run the
  // heaviest tiles (the last query rows) first.
  int qt, bh;
  if (p.causal) {
    qt = p.n_qtiles - 1 - static_cast<int>(blockIdx.x) / p.BH;
    bh = static_cast<int>(blockIdx.x) % p.BH;
  } else {
    qt = static_cast<int>(blockIdx.x) % p.n_qtiles;
    bh = static_cast<int>(blockIdx.x) / p.n_qtiles;
  }
  const int qbase = qt * kBM;
  // key steps this tile sees (causal: keys up to its last row, qbase + 127)
  const int n = p.causal ? min(p.n_steps, (qbase + kBM) / kBN) : p.n_steps;

  if (threadIdx.x == 0) {
    mbar_init(bar(kQFull), 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(bar(kKVFull + s), 1);
      mbar_init(bar(kKVEmpty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(kSFull + b), 1);
      mbar_init(bar(kPFull + b), 4);        // one arrive per softmax warp
    }
    mbar_init(bar(kOFull), 1);
    mbar_init(bar(kPVDone + 0), 1);
    mbar_init(bar(kPVDone + 1), 1);
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
      mbar_arrive_expect_tx(bar(kQFull), kQBytes);
      for (int pn = 0; pn < 4; ++pn)
        tma_load_3d(sb + kQOff + pn * kQPanel, &tmQ, bar(kQFull), pn * 64, qbase, bh);
      const uint64_t keep = l2_policy_evict_last();
      for (int i = 0; i < 4 * n; ++i) {
        const int s = ring_slot(i);
        if (!mbar_wait(bar(kKVEmpty + s), ring_phase(i) ^ 1, p.ctl, abort_flag)) break;
        const uint32_t dst = sb + kKVOff + s * kSlotBytes;
        int part, step;   // part: K features 0-127, 128-255; V keys 0-63, 64-127
        if (i < 2) {
          part = i;
          step = 0;
        } else {
          const int m = i - 2, blk = m >> 2, r = m & 3;
          if (blk < n - 1) {
            part = r;
            step = r < 2 ? blk + 1 : blk;
          } else {
            part = 2 + r;
            step = blk;
          }
        }
        const int key0 = step * kBN;
        mbar_arrive_expect_tx(bar(kKVFull + s), kSlotBytes);
        if (part < 2) {
          for (int pn = 0; pn < 2; ++pn)
            tma_load_3d_hint(dst + pn * kKPanel, &tmK, bar(kKVFull + s), (2 * part + pn) * 64, key0, bh, keep);
        } else {
          for (int pn = 0; pn < 4; ++pn)
            tma_load_3d_hint(dst + pn * kVPanel, &tmV, bar(kKVFull + s), pn * 64, key0 + 64 * (part - 2), bh,
                             keep);
        }
      }
    }
  } else if (warp == 1 || warp == 6) {
    // ---------------------------------------------- MMA issuers (S; P V)
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16(kBM, kBN, false, false);
      constexpr uint32_t idO = idesc_bf16(kBM, D, false, true);
      auto slot_addr = [&](int i) { return sb + kKVOff + ring_slot(i) * kSlotBytes; };
      auto kv_wait = [&](int i) { return mbar_wait(bar(kKVFull + ring_slot(i)), ring_phase(i), p.ctl, abort_flag); };
      bool ok = true;
      if (warp == 1) {
        ok = mbar_wait(bar(kQFull), 0, p.ctl, abort_flag);
        for (int j = 0; j < n && ok; ++j) {   // S_j = Q K_j^T into S buffer j & 1
          // the buffer held P_{j-2}: P V_{j-2} must have read it
          if (j >= 2 && !(ok = mbar_wait(bar(kPVDone + (j & 1)), ((j - 2) >> 1) & 1, p.ctl, abort_flag))) break;
          for (int h = 0; h < 2; ++h) {       // feature halves of K_j, one ring slot each
            const int ik = k_load(j, h);
            if (!(ok = kv_wait(ik))) break;
            tc_fence_after();
            const uint32_t ka = slot_addr(ik);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint32_t qa = sb + kQOff + (2 * h + (k >> 2)) * kQPanel + (k & 3) * 32;
              const uint32_t kb = ka + (k >> 2) * kKPanel + (k & 3) * 32;
              mma_ss(tmem + kColS + 128 * (j & 1), sdesc_sw128(qa, 0, 1024), sdesc_sw128(kb, 0, 1024), idS,
                     (h > 0 || k > 0) ? 1u : 0u);
            }
            if (h == 1) tc_commit(bar(kSFull + (j & 1)));
            tc_commit(bar(kKVEmpty + ring_slot(ik)));   // this half of K_j read
          }
        }
      } else {
        for (int j = 0; j < n && ok; ++j) {   // O += P_j V_j, P_j over S buffer j & 1
          if (!(ok = mbar_wait(bar(kPFull + (j & 1)), (j >> 1) & 1, p.ctl, abort_flag))) break;
          for (int h = 0; h < 2; ++h) {       // key halves of V_j, one ring slot each
            const int iv = v_load(j, h, n);
            if (!(ok = kv_wait(iv))) break;
            tc_fence_after();
            const uint32_t va = slot_addr(iv);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_ts(tmem + kColO, tmem + kColS + 128 * (j & 1) + 32 * h + 8 * k,
                     sdesc_sw128(va + k * 2048, kVPanel, 1024), idO, (j > 0 || h > 0 || k > 0) ? 1u : 0u);
            tc_commit(bar(kKVEmpty + ring_slot(iv)));   // this half of V_j read
          }
          if (ok) tc_commit(bar(kPVDone + (j & 1)));   // P V_j complete
        }
        if (ok) tc_commit(bar(kOFull));
      }
    }
  } else {
    // ------------------------------------------------------- softmax (2-5)
    const int rank = warp & 3;              // tensor-memory lane quarter
    const int r_in_tile = rank * 32 + lane;
    const int row = qbase + r_in_tile;
    const uint32_t lane_addr = static_cast<uint32_t>(rank * 32) << 16;
    const uint32_t tO = tmem + lane_addr + kColO;
    const float c = p.c;
    bool ok = true;
    float m_ref = -INFINITY;
    float l = 0.f;      // sum of the fp32 probabilities: gives the LSE
    float lr = 0.f;     // rounding residuals of the blocks' largest P
    const int key_lim = p.causal ? min(p.N_kv - 1, row) : p.N_kv - 1;   // last key this row sees
    for (int j = 0; j < n && ok; ++j) {
      const int b = j & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(kSFull + b), (j >> 1) & 1, p.ctl, abort_flag));
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
        ok = __all_sync(0xffffffffu, mbar_wait(bar(kPVDone + ((j - 1) & 1)), ((j - 1) >> 1) & 1, p.ctl, abort_flag));
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
      if (lane == 0) mbar_arrive(bar(kPFull + b));
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
    if (ready) ready = mbar_wait(bar(kOFull), 0, p.ctl, abort_flag);
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

  __syncwarp();   // warps whose lane 0 ran a role alone arrive whole
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
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
  p.n_steps = (a.N_kv + kBN - 1) / kBN;
  p.c = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  p.tau = a.tau;
  p.ctl = a.ctl;
  auto kern = fwd256_kernel<EMU>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(p.n_qtiles) * p.BH;
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

}  // namespace fwd256
}  // namespace fa
