// fa_fwd8_256_kernel.cuh -- the 8-bit forward at head dimension 256.
//
// "FlashAttention-3: Fast and Accurate Attention with Asynchrony and
// Low-precision" 技術 3 on e4m3 codes (quantised by the kernels of
// fa_fwd8_kernel.cuh), at the head dimension its 8-bit measurements centre
// on.  At d = 256 one query tile's O takes half of tensor memory, so, as in
// the bf16 d = 256 kernel, one CTA owns one 128-row query tile and overlaps
// consecutive key steps of it; a step is one 128-key quantisation block:
//
//   tensor memory   S_j in one of two 128-column buffers [0,128) / [128,256)
//                   (P_j, four e4m3 per column, over its first 32 columns),
//                   O [256,512)
//   warp 0          TMA producer: the Q codes once (32 KB), then K_j, V_j
//                   (32 KB each: two 128-byte panels) into a five-slot ring,
//                   K_0 first and then K_{j+1} ahead of V_j
//   warps 1, 6      issuing threads of the even and the odd key steps: each
//                   issues O += P_j V_j (four kind::f8f6f4 products of
//                   N = 256, V as the MN-major operand) once P_j is written,
//                   followed by S_{j+2} = Q K_{j+2}^T (eight products of
//                   K = 32, both operands in shared memory) into the buffer
//                   P_j occupies
//   warps 2-5       softmax, one thread per query row: S_j scaled by
//                   c = scale log2(e) / (inv_q inv_k_j), the online softmax
//                   with conditional rescaling, P rounded to e4m3
//
// The tensor core runs one thread's products in order, so S_{j+2} follows
// P V_j without waiting for its completion; the two threads keep each
// other's waits off the tensor core's queue.  P V_j goes into the queue after
// P V_{j-1} (an issue barrier between the threads, not a completion wait):
// P V_0 initialises O, and a fixed order keeps the sums reproducible.  The
// rare O rescale must not race with the previous step's P V, so it first
// waits for that product's completion barrier.  O is divided by
// (l + residuals) inv_v at the end, as in the d = 128 kernel.
#pragma once

#include "fa_fwd8_kernel.cuh"

namespace fa {
namespace fwd8_256 {

constexpr int D = 256;
constexpr int kBM = 128;                  // query rows per CTA
constexpr int kBN = 128;                  // keys per step: one quantisation block
constexpr int kThreads = 224;             // 7 warps
constexpr int kSlots = 5;                 // K/V ring
constexpr int kPanel = 128 * 128;         // 128 rows x 128 B swizzle panel
constexpr int kTileBytes = 2 * kPanel;    // 128 rows x 256 B
constexpr int kQOff = 0;
constexpr int kKVOff = kTileBytes;
constexpr int kBarOff = kKVOff + kSlots * kTileBytes;
// barrier indices
constexpr int kQFull = 0;
constexpr int kKVFull = 1;                // kSlots
constexpr int kKVEmpty = 1 + kSlots;      // kSlots
constexpr int kSFull = 1 + 2 * kSlots;    // 2 (per S buffer)
constexpr int kPFull = 3 + 2 * kSlots;    // 2 (per S buffer)
constexpr int kOFull = 5 + 2 * kSlots;
constexpr int kPVDone = 6 + 2 * kSlots;   // 2 (per S buffer): P V has read the buffer's P
constexpr int kPVIssued = 8 + 2 * kSlots; // P V_j issued (orders P V_{j+1} after it)
constexpr int kNumBars = 9 + 2 * kSlots;
constexpr int kMiscOff = kBarOff + 8 * kNumBars;   // tmem base, abort flag
constexpr int kSmemBytes = kMiscOff + 16 + 1024;   // + base alignment slack
// tensor-memory columns
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 256;
constexpr uint32_t kTmemCols = 512;

struct Params {
  __nv_bfloat16* o;
  float* lse;
  const float* qinv;       // [B*H, query blocks]
  const float* kinv;       // [B*H, key blocks]
  const float* vamax;      // [B*H] largest |V|
  int BH, N_q, N_kv, causal;
  int n_qtiles;            // ceil(N_q / 128)
  int n_steps;             // ceil(N_kv / 128)
  float c0;                // scale * log2(e) (/ 256 with the Hadamard transform)
  float tau;
  DevCtl ctl;
};

// K/V ring in load order: K_0, then K_{j+1} ahead of V_j, and V_{n-1} last.
__device__ __forceinline__ int k_load(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int v_load(int j, int n) { return j < n - 1 ? 2 * j + 2 : 2 * n - 1; }
__device__ __forceinline__ int ring_slot(int i) { return i % kSlots; }
__device__ __forceinline__ uint32_t ring_phase(int i) { return static_cast<uint32_t>((i / kSlots) & 1); }

__global__ void __launch_bounds__(kThreads, 1)
fwd8_256_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
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
  // key steps this tile sees (causal: keys up to its last row)
  const int n = p.causal ? min(p.n_steps, qt + 1) : p.n_steps;

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
    mbar_init(bar(kPVIssued), 1);
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
      mbar_arrive_expect_tx(bar(kQFull), kTileBytes);
      for (int pn = 0; pn < 2; ++pn)
        tma_load_3d(sb + kQOff + pn * kPanel, &tmQ, bar(kQFull), pn * 128, qbase, bh);
      const uint64_t keep = l2_policy_evict_last();
      for (int i = 0; i < 2 * n; ++i) {
        const int s = ring_slot(i);
        if (!mbar_wait(bar(kKVEmpty + s), ring_phase(i) ^ 1, p.ctl, abort_flag)) break;
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
        const uint32_t dst = sb + kKVOff + s * kTileBytes;
        mbar_arrive_expect_tx(bar(kKVFull + s), kTileBytes);
        for (int pn = 0; pn < 2; ++pn)       // channels 128 pn .. 128 pn + 127 of 128 keys
          tma_load_3d_hint(dst + pn * kPanel, is_k ? &tmK : &tmV, bar(kKVFull + s), pn * 128, step * kBN, bh, keep);
      }
    }
  } else if (warp == 1 || warp == 6) {
    // ------------------------------- MMA issuers: steps j of parity par
    if (lane == 0) {
      const int par = warp == 1 ? 0 : 1;
      constexpr uint32_t idS = idesc_e4m3(kBM, kBN);            // S = Q K^T, both K-major
      constexpr uint32_t idO = idesc_e4m3(kBM, D, true);        // O += P V, V MN-major
      auto slot_addr = [&](int i) { return sb + kKVOff + ring_slot(i) * kTileBytes; };
      auto kv_wait = [&](int i) { return mbar_wait(bar(kKVFull + ring_slot(i)), ring_phase(i), p.ctl, abort_flag); };
      auto issue_S = [&](int j) -> bool {   // S_j = Q K_j^T into S buffer j & 1
        const int ik = k_load(j);
        if (!kv_wait(ik)) return false;
        tc_fence_after();
        const uint32_t qa = sb + kQOff;
        const uint32_t ka = slot_addr(ik);
#pragma unroll
        for (int k = 0; k < D / 32; ++k) {
          const uint32_t off = (k >> 2) * kPanel + (k & 3) * 32;
          mma_ss_f8(tmem + kColS + 128 * (j & 1), sdesc_sw128(qa + off, 0, 1024), sdesc_sw128(ka + off, 0, 1024),
                    idS, k > 0 ? 1u : 0u);
        }
        tc_commit(bar(kSFull + (j & 1)));
        tc_commit(bar(kKVEmpty + ring_slot(ik)));        // K_j read
        return true;
      };
      bool ok = mbar_wait(bar(kQFull), 0, p.ctl, abort_flag);
      if (ok && par < n) ok = issue_S(par);
      for (int j = par; j < n && ok; j += 2) {   // O += P_j V_j, P_j over S buffer j & 1
        if (!(ok = mbar_wait(bar(kPFull + (j & 1)), (j >> 1) & 1, p.ctl, abort_flag))) break;
        const int iv = v_load(j, n);
        if (!(ok = kv_wait(iv))) break;
        // the other thread's P V_{j-1} goes into the tensor core's queue first
        if (j >= 1 && !(ok = mbar_wait(bar(kPVIssued), (j - 1) & 1, p.ctl, abort_flag))) break;
        tc_fence_after();
        const uint32_t va = slot_addr(iv);
#pragma unroll
        for (int k = 0; k < kBN / 32; ++k)
          mma_ts_f8(tmem + kColO, tmem + kColS + 128 * (j & 1) + 8 * k, sdesc_sw128(va + 4096 * k, kPanel, 1024),
                    idO, (j > 0 || k > 0) ? 1u : 0u);
        tc_fence_before();
        mbar_arrive(bar(kPVIssued));
        tc_commit(bar(kKVEmpty + ring_slot(iv)));    // V_j read
        tc_commit(bar(kPVDone + (j & 1)));           // (and every earlier P V complete)
        if (j == n - 1) tc_commit(bar(kOFull));
        // S_{j+2} overwrites P_j: issued after P V_j by the same thread, the
        // tensor core runs it after P V_j has read its operand
        if (j + 2 < n) ok = issue_S(j + 2);
      }
    }
  } else {
    // ------------------------------------------------------- softmax (2-5)
    const int rank = warp & 3;              // tensor-memory lane quarter
    const int r_in_tile = rank * 32 + lane;
    const int row = qbase + r_in_tile;
    const uint32_t lane_addr = static_cast<uint32_t>(rank * 32) << 16;
    const uint32_t tO = tmem + lane_addr + kColO;
    const float cq = n > 0 ? p.c0 / p.qinv[static_cast<size_t>(bh) * p.n_qtiles + qt] : 0.f;
    const float* kinv = p.kinv + static_cast<size_t>(bh) * p.n_steps;
    float kinv_next = n > 0 ? kinv[0] : 1.f;
    float m_ref = -INFINITY;
    float l = 0.f;
    float lr = 0.f;
    bool ok = true;
    const int key_lim = p.causal ? min(p.N_kv - 1, row) : p.N_kv - 1;   // last key this row sees
    for (int j = 0; j < n && ok; ++j) {
      const int b = j & 1;
      const float c = cq / kinv_next;          // this key block's logit scale
      if (j + 1 < n) kinv_next = kinv[j + 1];
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
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float2 x0 = fma2(make_float2(__uint_as_float(s[4 * i]), __uint_as_float(s[4 * i + 1])), c2, neg2);
        const float2 x1 = fma2(make_float2(__uint_as_float(s[4 * i + 2]), __uint_as_float(s[4 * i + 3])), c2, neg2);
        const float e0 = ex2_hw(x0.x), e1 = ex2_hw(x0.y), e2 = ex2_hw(x1.x), e3 = ex2_hw(x1.y);
        sum[i & 1] = add2(sum[i & 1], make_float2(e0 + e2, e1 + e3));
        pk[i] = pack_e4m3x4(e0, e1, e2, e3);
      }
      tmem_st_x32(tS, pk);   // waits for its own stores
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kPFull + b));
      l += (sum[0].x + sum[0].y) + (sum[1].x + sum[1].y);
      {
        const float pm = ex2_hw(fmaf(mxs, c, -m_ref));   // the block's largest P
        lr += fwd8::e4m3_value(pm) - pm;                // as rounded for P V
      }
    }
    // ------------------------------------------------------------- epilogue
    bool ready = ok && n > 0;
    if (ready) ready = mbar_wait(bar(kOFull), 0, p.ctl, abort_flag);
    if (__all_sync(0xffffffffu, ready)) {
      tc_fence_after();
      const float vinv = fwd8::e4m3_multiplier(p.vamax[bh]);
      const float inv_l = 1.f / ((l + lr) * vinv);
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

}  // namespace fwd8_256
}  // namespace fa
