// fa_testing.cu -- test-only entry points of include/fa_testing.h: the
// exponential paths, one tensor-core tile product, and the watchdog.
#include <cuda_bf16.h>

#include "exp2.cuh"
#include "fa.h"
#include "fa_internal.h"
#include "fa_testing.h"
#include "ptx.cuh"
#include "ptx_pair.cuh"

namespace fa {
namespace testing {

__global__ void exp2_kernel(const float* x, float* y, long long n, int mode) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    y[i] = mode == 1 ? ex2_poly3(x[i]) : ex2_hw(x[i]);
}

// One 128 x 128 x K product with the operand paths of the attention kernels.
// Shared memory: A panels, B panels, two barriers, the tensor-memory base.
constexpr int kTileThreads = 128;

__global__ void __launch_bounds__(kTileThreads, 1)
mma_tile_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __nv_bfloat16* A, float* Cout, int K, int mode, DevCtl ctl) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const int tile_bytes = 128 * K * 2;
  const uint32_t sA = sb, sB = sb + tile_bytes;
  const uint32_t bar_full = sb + 2 * tile_bytes, bar_done = bar_full + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 2 * tile_bytes + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 2 * tile_bytes + 20);
  const bool b_mn = mode & 1, a_tmem = mode & 2, a_mn = mode & 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(bar_full, 1);
    mbar_init(bar_done, 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), 256);
  __syncwarp();   // warps whose lane 0 ran a role alone arrive whole
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(bar_full, (a_tmem ? 0 : tile_bytes) + tile_bytes);
    if (a_mn) {
      // A is [K, 128]: two 64-column panels of K rows each
      for (int pn = 0; pn < 2; ++pn) tma_load_3d(sA + pn * K * 128, &tmA, bar_full, pn * 64, 0, 0);
    } else {
      for (int pn = 0; pn < K / 64 && !a_tmem; ++pn)
        tma_load_3d(sA + pn * 16384, &tmA, bar_full, pn * 64, 0, 0);
    }
    if (!b_mn) {
      for (int pn = 0; pn < K / 64; ++pn) tma_load_3d(sB + pn * 16384, &tmB, bar_full, pn * 64, 0, 0);
    } else {
      // B is [K, 128]: two 64-column panels of K rows each
      for (int pn = 0; pn < 2; ++pn) tma_load_3d(sB + pn * K * 128, &tmB, bar_full, pn * 64, 0, 0);
    }
  }
  if (a_tmem) {
    // Thread r writes row r of A into tensor-memory lane r, columns 128.. as
    // packed bf16 pairs (low half = even k).
    const uint32_t* arow = reinterpret_cast<const uint32_t*>(A + static_cast<size_t>(threadIdx.x) * K);
    const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
    for (int ch = 0; ch < K / 32; ++ch) {
      uint32_t r[16];
      for (int i = 0; i < 16; ++i) r[i] = arow[ch * 16 + i];
      tmem_st_x16(tmem + lane_addr + 128 + 16 * ch, r);
    }
    tc_fence_before();
  }
  __syncwarp();
  __syncthreads();
  if (threadIdx.x == 0) {
    tc_fence_after();
    if (mbar_wait(bar_full, 0, ctl, abort_flag)) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(128, 128, a_mn, b_mn);
      for (int k = 0; k < K / 16; ++k) {
        const uint64_t bd = b_mn ? sdesc_sw128(sB + k * 2048, K * 128, 1024)
                                 : sdesc_sw128(sB + (k >> 2) * 16384 + (k & 3) * 32, 0, 1024);
        if (a_tmem)
          mma_ts(tmem, tmem + 128 + 8 * k, bd, idesc, k > 0);
        else if (a_mn)
          mma_ss(tmem, sdesc_sw128(sA + k * 2048, K * 128, 1024), bd, idesc, k > 0);
        else
          mma_ss(tmem, sdesc_sw128(sA + (k >> 2) * 16384 + (k & 3) * 32, 0, 1024), bd, idesc, k > 0);
      }
      tc_commit(bar_done);
    }
  }
  __syncwarp();
  if (__all_sync(0xffffffffu, mbar_wait(bar_done, 0, ctl, abort_flag))) {
    tc_fence_after();
    const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
    float* crow = Cout + static_cast<size_t>(threadIdx.x) * 128;
    for (int ch = 0; ch < 4; ++ch) {
      uint32_t r[32];
      tmem_ld_x32(tmem + lane_addr + 32 * ch, r);
      for (int i = 0; i < 32; ++i) crow[32 * ch + i] = __uint_as_float(r[i]);
    }
  }
  (void)lane;
  __syncwarp();   // warps whose lane 0 ran a role alone arrive whole
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// One 256 x 128 x K product of a CTA pair (cta_group::2).  Shared memory of
// each CTA: its A rows (K/64 panels of 128 rows), its half of B (K-major:
// K/64 panels of 64 rows; N-major: one 64-column panel of K rows), two
// barriers, the tensor-memory base and the abort flag.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kTileThreads, 1)
mma_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __nv_bfloat16* A, float* Cout, int K, int mode, DevCtl ctl) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  if (sb & 1023u) {   // the same offset in both CTAs, so both return here or neither does
    if (threadIdx.x == 0) atomicOr(ctl.status, kStatusLaunchConfig);
    return;
  }
  const int a_bytes = 128 * K * 2, b_bytes = 64 * K * 2;
  const uint32_t sA = sb, sB = sb + a_bytes;
  const uint32_t bar_full = sb + a_bytes + b_bytes, bar_done = bar_full + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + a_bytes + b_bytes + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + a_bytes + b_bytes + 20);
  const bool b_mn = mode & 1, a_tmem = mode & 2;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const uint32_t peer_abort = map_shared(smem_u32(const_cast<int*>(abort_flag)), rank ^ 1u);
  const int warp = threadIdx.x >> 5;
  auto wait = [&](uint32_t b, uint32_t parity) { return pair_wait(b, parity, ctl, abort_flag, peer_abort); };

  if (threadIdx.x == 0) {
    mbar_init(bar_full, leader ? 2 : 1);   // the leader also counts CTA 1's forwarded arrival
    mbar_init(bar_done, 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 0) tmem_alloc_pair(smem_u32(tmem_slot), 256);
  __syncwarp();
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int r = static_cast<int>(rank);

  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(bar_full, (a_tmem ? 0 : a_bytes) + b_bytes);
    for (int pn = 0; pn < K / 64 && !a_tmem; ++pn)
      tma_load_3d(sA + pn * 16384, &tmA, bar_full, pn * 64, 128 * r, 0);
    if (!b_mn) {
      for (int pn = 0; pn < K / 64; ++pn) tma_load_3d(sB + pn * 8192, &tmB, bar_full, pn * 64, 64 * r, 0);
    } else {
      tma_load_3d(sB, &tmB, bar_full, 64 * r, 0, 0);   // columns 64 r .. 64 r + 63 of [K, 128], K rows
    }
  }
  if (a_tmem) {
    // thread t writes row 128 r + t of A into tensor-memory lane t, columns
    // 128.. as packed bf16 pairs (low half = even k)
    const uint32_t* arow = reinterpret_cast<const uint32_t*>(A + static_cast<size_t>(128 * r + threadIdx.x) * K);
    const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
    for (int ch = 0; ch < K / 32; ++ch) {
      uint32_t v[16];
      for (int i = 0; i < 16; ++i) v[i] = arow[ch * 16 + i];
      tmem_st_x16(tmem + lane_addr + 128 + 16 * ch, v);
    }
    tc_fence_before();
  }
  __syncwarp();
  __syncthreads();
  if (threadIdx.x == 0 && !leader) {
    // this CTA's operands are in place: count them on the leader's barrier
    if (wait(bar_full, 0)) mbar_arrive_remote_relaxed(map_shared(bar_full, 0));
  }
  if (threadIdx.x == 0 && leader) {
    if (wait(bar_full, 0)) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(256, 128, false, b_mn);
      for (int k = 0; k < K / 16; ++k) {
        const uint64_t bd = b_mn ? sdesc_sw128(sB + k * 2048, K * 128, 1024)
                                 : sdesc_sw128(sB + (k >> 2) * 8192 + (k & 3) * 32, 0, 1024);
        if (a_tmem)
          mma_ts_pair(tmem, tmem + 128 + 8 * k, bd, idesc, k > 0);
        else
          mma_ss_pair(tmem, sdesc_sw128(sA + (k >> 2) * 16384 + (k & 3) * 32, 0, 1024), bd, idesc, k > 0);
      }
      tc_commit_pair(bar_done, 3);   // both CTAs
    }
  }
  __syncwarp();
  if (__all_sync(0xffffffffu, wait(bar_done, 0))) {
    tc_fence_after();
    const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
    float* crow = Cout + static_cast<size_t>(128 * r + threadIdx.x) * 128;
    for (int ch = 0; ch < 4; ++ch) {
      uint32_t v[32];
      tmem_ld_x32(tmem + lane_addr + 32 * ch, v);
      for (int i = 0; i < 32; ++i) crow[32 * ch + i] = __uint_as_float(v[i]);
    }
  }
  __syncwarp();
  tc_fence_before();
  cluster_sync();   // neither CTA leaves while the other may still use its memory
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 256);
  }
}

__global__ void wait_timeout_kernel(DevCtl ctl) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    mbar_init_fence();
  }
  __syncwarp();
  __syncthreads();
  // Nothing ever arrives on `bar`: the bounded wait runs out and flags it.
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, ctl, &abort_flag);
}


// One 128 x 128 x 128 e4m3 tile product: rows converted on the device (thread
// r converts row r of A and of B), A in shared memory (mode 0) or tensor
// memory (mode 1), B in shared memory, both K-major with the 128-byte swizzle
// (one 128-byte row = 128 elements).  Writes C = A8 B8^T and A's codes.
__global__ void __launch_bounds__(128, 1)
mma_fp8_kernel(const float* A, const float* B, float* Cout, uint8_t* a_codes, int mode, DevCtl ctl) {
  __shared__ __align__(1024) uint8_t sA[128 * 128];
  __shared__ __align__(1024) uint8_t sB[128 * 128];
  __shared__ __align__(8) uint64_t bar_done;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  const int r = threadIdx.x, warp = r >> 5;
  const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
  if (r == 0) {
    mbar_init(smem_u32(&bar_done), 1);
    abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 0) tmem_alloc(smem_u32(&tmem_slot), 256);
  __syncwarp();   // warps whose lane 0 ran a role alone arrive whole
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  uint32_t wa[32], wb[32];
  for (int i = 0; i < 32; ++i) {
    const float* a = A + r * 128 + 4 * i;
    const float* b = B + r * 128 + 4 * i;
    wa[i] = pack_e4m3x4(a[0], a[1], a[2], a[3]);
    wb[i] = pack_e4m3x4(b[0], b[1], b[2], b[3]);
    reinterpret_cast<uint32_t*>(a_codes + r * 128)[i] = wa[i];
  }
  for (int ch = 0; ch < 8; ++ch) {          // 16-byte chunk ch of row r at ch ^ (r & 7)
    const int pc = (ch ^ (r & 7)) * 16 + r * 128;
    *reinterpret_cast<uint4*>(sA + pc) = make_uint4(wa[4 * ch], wa[4 * ch + 1], wa[4 * ch + 2], wa[4 * ch + 3]);
    *reinterpret_cast<uint4*>(sB + pc) = make_uint4(wb[4 * ch], wb[4 * ch + 1], wb[4 * ch + 2], wb[4 * ch + 3]);
  }
  if (mode == 1) tmem_st_x32(tmem + lane_addr + 128, wa);
  fence_async_smem();
  __syncwarp();   // warps whose lane 0 ran a role alone arrive whole
  tc_fence_before();
  __syncthreads();
  if (r == 0) {
    tc_fence_after();
    constexpr uint32_t idesc = idesc_e4m3(128, 128);
    for (int k = 0; k < 4; ++k) {            // 32 elements (32 bytes) per product
      const uint64_t bd = sdesc_sw128(smem_u32(sB) + 32 * k, 0, 1024);
      if (mode == 1)
        mma_ts_f8(tmem, tmem + 128 + 8 * k, bd, idesc, k > 0);
      else
        mma_ss_f8(tmem, sdesc_sw128(smem_u32(sA) + 32 * k, 0, 1024), bd, idesc, k > 0);
    }
    tc_commit(smem_u32(&bar_done));
  }
  __syncwarp();
  volatile int* ab = &abort_flag;
  if (__all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_done), 0, ctl, ab))) {
    tc_fence_after();
    for (int ch = 0; ch < 4; ++ch) {
      uint32_t v[32];
      tmem_ld_x32(tmem + lane_addr + 32 * ch, v);
      for (int i = 0; i < 32; ++i) Cout[r * 128 + 32 * ch + i] = __uint_as_float(v[i]);
    }
  }
  __syncwarp();   // warps whose lane 0 ran a role alone arrive whole
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

}  // namespace testing
}  // namespace fa

using namespace fa;


extern "C" {

int fa_test_exp2(const float* x, float* y, long long n, int mode, fa_stream_t stream) {
  if (n < 0 || (n > 0 && (!x || !y)) || (mode != 0 && mode != 1)) return FA_ERR_INVALID;
  if (n == 0) return FA_OK;
  DevCtl ctl;
  const int st = device_ctl(&ctl);
  if (st != FA_OK) return st;
  const long long blocks = (n + 255) / 256;
  testing::exp2_kernel<<<static_cast<unsigned>(blocks < 4096 ? blocks : 4096), 256, 0,
                         static_cast<cudaStream_t>(stream)>>>(x, y, n, mode);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_test_mma_tile(const void* A, const void* B, float* C, int K, int mode, fa_stream_t stream) {
  if (!A || !B || !C || (K != 64 && K != 128) || mode < 0 || mode > 5) return FA_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(C)) % 16)
    return FA_ERR_ALIGN;
  DevCtl ctl;
  int st = device_ctl(&ctl);
  if (st != FA_OK) return st;
  CUtensorMap tmA, tmB;
  if (mode & 4)
    st = make_map_bf16(&tmA, A, 128, K, 1, K);   // [K, 128]: panels of 64 columns, K rows
  else
    st = make_map_bf16(&tmA, A, K, 128, 1);
  if (st != FA_OK) return st;
  if (mode & 1)
    st = make_map_bf16(&tmB, B, 128, K, 1, K);   // [K, 128]: panels of 64 columns, K rows
  else
    st = make_map_bf16(&tmB, B, K, 128, 1);
  if (st != FA_OK) return st;
  const int smem = 2 * 128 * K * 2 + 64 + 1024;
  auto kern = testing::mma_tile_kernel;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  kern<<<1, testing::kTileThreads, smem, static_cast<cudaStream_t>(stream)>>>(
      tmA, tmB, static_cast<const __nv_bfloat16*>(A), C, K, mode, ctl);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_test_mma_pair(const void* A, const void* B, float* C, int K, int mode, fa_stream_t stream) {
  if (!A || !B || !C || (K != 64 && K != 128) || mode < 0 || mode > 3) return FA_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(C)) % 16)
    return FA_ERR_ALIGN;
  DevCtl ctl;
  int st = device_ctl(&ctl);
  if (st != FA_OK) return st;
  CUtensorMap tmA, tmB;
  if ((st = make_map_bf16(&tmA, A, K, 256, 1)) != FA_OK) return st;          // [256, K]: 128-row boxes
  if (mode & 1)
    st = make_map_bf16(&tmB, B, 128, K, 1, K);   // [K, 128]: 64-column boxes of K rows
  else
    st = make_map_bf16(&tmB, B, K, 128, 1, 64);  // [128, K]: 64-row boxes
  if (st != FA_OK) return st;
  const int smem = 128 * K * 2 + 64 * K * 2 + 64;
  auto kern = testing::mma_pair_kernel;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  kern<<<2, testing::kTileThreads, smem, static_cast<cudaStream_t>(stream)>>>(
      tmA, tmB, static_cast<const __nv_bfloat16*>(A), C, K, mode, ctl);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_test_mma_fp8(const float* A, const float* B, float* C, unsigned char* A_codes, int mode,
                    fa_stream_t stream) {
  if (!A || !B || !C || !A_codes) return FA_ERR_INVALID;
  if (mode != 0 && mode != 1) return FA_ERR_INVALID;
  DevCtl ctl;
  const int st = device_ctl(&ctl);
  if (st != FA_OK) return st;
  testing::mma_fp8_kernel<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(A, B, C, A_codes, mode, ctl);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_test_wait_timeout(unsigned long long timeout_ns, fa_stream_t stream) {
  if (timeout_ns < 1000ull || timeout_ns > 10000000000ull) return FA_ERR_INVALID;
  DevCtl ctl;
  const int st = device_ctl(&ctl);
  if (st != FA_OK) return st;
  ctl.timeout_ns = timeout_ns;
  testing::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(ctl);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // extern "C"
