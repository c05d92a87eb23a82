/*
 * fa_testing.h -- test-only entry points of the GB300 attention library.
 *
 * These expose, one at a time, the device building blocks the attention
 * kernels are made of, so that tests can check each against the CPU:
 *   - the two ways the kernels take 2^x (hardware ex2 and the FMA-pipe cubic
 *     emulation of "論文解説: FlashAttention-4 — Algorithm and Kernel
 *     Pipelining Co-Design for Asymmetric Hardware Scaling",
 *     ソフトウェア指数関数エミュレーション);
 *   - one TMA-loaded, tcgen05 tensor-core tile product with the operand
 *     layouts the attention kernels use;
 *   - the bounded-wait watchdog.
 * All pointers are caller-owned DEVICE pointers; calls are asynchronous on
 * `stream`; the return value is an fa_status (see fa.h).
 */
#ifndef FA_GB300_TESTING_H
#define FA_GB300_TESTING_H

#include "fa.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * fa_test_exp2 -- y[i] = 2^x[i] for i < n (fp32 in, fp32 out).
 *   mode 0: the hardware ex2 unit (approximate, flush-to-zero).
 *   mode 1: the cubic emulation: n = floor(x), f = x - n,
 *           p(f) = 1 + 0.6951 f + 0.2276 f^2 + 0.0771 f^3, exponent n added
 *           to p's exponent field by an integer operation; inputs below -126
 *           are clamped to -126 (so the result never drops below 2^-126).
 *   n >= 0 (0 launches nothing); x, y 4-byte aligned.
 */
int fa_test_exp2(const float* x, float* y, long long n, int mode, fa_stream_t stream);

/*
 * fa_test_mma_tile -- C = A * B^T for one tile on the tensor cores.
 *   A bf16 [128, K] row-major (K contiguous), K in {64, 128}.
 *   mode bit 0 clear: B bf16 [128, K] row-major (the S = Q K^T form: both
 *                     operands K-major);
 *   mode bit 0 set:   B bf16 [K, 128] row-major, i.e. C = A * B with the
 *                     B operand N-major (the O += P V form);
 *   mode bit 1 set:   A is first copied into tensor memory and the product
 *                     reads it from there (the P operand's path);
 *   mode bit 2 set:   A is given as [K, 128] row-major, i.e. C = A^T * ...
 *                     with the A operand M-major (the dQ = dS K form);
 *                     not combined with bit 1.
 *   Valid modes: 0, 1, 2, 3, 4, 5.
 *   C fp32 [128, 128] row-major (output).
 */
int fa_test_mma_tile(const void* A, const void* B, float* C, int K, int mode,
                     fa_stream_t stream);

/*
 * fa_test_mma_pair -- C = A * B^T (or A * B) for one 256 x 128 x K product
 * shared by the two CTAs of a cluster (tcgen05 cta_group::2, the 2-CTA MMA
 * mode of "論文解説: FlashAttention-4 — Algorithm and Kernel Pipelining
 * Co-Design for Asymmetric Hardware Scaling", Backwardパスの最適化): CTA r
 * holds rows [128 r, 128 r + 128) of A and of C and the r-th half of B's N
 * columns; CTA 0 issues the product.
 *   A bf16 [256, K] row-major (K contiguous), K in {64, 128}.
 *   mode bit 0 clear: B bf16 [128, K] row-major (both operands K-major);
 *   mode bit 0 set:   B bf16 [K, 128] row-major, i.e. C = A * B with B N-major;
 *   mode bit 1 set:   each CTA first copies its rows of A into tensor memory
 *                     and the product reads them from there.
 *   Valid modes: 0, 1, 2, 3.
 *   C fp32 [256, 128] row-major (output).
 * Device pointers, 16-byte aligned; returns FA_ERR_INVALID / FA_ERR_ALIGN
 * before any launch for bad arguments.
 */
int fa_test_mma_pair(const void* A, const void* B, float* C, int K, int mode, fa_stream_t stream);

/*
 * fa_test_mma_fp8 -- C = A8 * B8^T for one 128 x 128 x 128 tile with e4m3
 * operands (the products of the 8-bit forward path, fa_fwd_fp8).
 *   A, B fp32 [128, 128] row-major; each row is rounded to e4m3 on the
 *   device (nearest even, saturating to +-448) exactly as the 8-bit forward
 *   rounds its operands, and the codes of A are written to A_codes (u8
 *   [128, 128], the OCP e4m3 encoding).
 *   mode 0: A from shared memory; mode 1: A from tensor memory (the P
 *   operand's path).  C fp32 [128, 128] row-major (output).
 */
int fa_test_mma_fp8(const float* A, const float* B, float* C, unsigned char* A_codes, int mode,
                    fa_stream_t stream);

/*
 * fa_test_wait_timeout -- launch one CTA that waits on a barrier nothing
 * will ever arrive on, with a limit of timeout_ns; the wait runs out and the
 * kernel sets the device status to FA_ERR_TIMEOUT and returns.  Used to
 * check the watchdog path without faulting or hanging the GPU.
 */
int fa_test_wait_timeout(unsigned long long timeout_ns, fa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_TESTING_H */
