/*
 * fa.h -- exact scaled-dot-product attention on one NVIDIA GB300 (sm_103a).
 *
 * The operation (forward):
 *     S   = scale * Q K^T                     (N_q x N_kv per batch and head)
 *     P   = softmax(S) row by row, restricted to the allowed keys
 *     O   = P V
 *     LSE = log(sum over allowed keys of exp(S))      (natural log)
 * as defined in "FlashAttention: GPUメモリ階層を活用したアテンション最適化の分析"
 * §2.1 (standard attention) and §6.1 (safe softmax), computed tile by tile
 * with the online softmax of §6.2 so that S and P never reach HBM.  The
 * causal mask is the lower-triangular mask of §11.3, top-left aligned: query
 * i may attend key j iff j <= i (for N_q != N_kv as well).
 *
 * The backward pass returns dQ, dK, dV for a given dO, recomputing P from
 * the saved LSE (§7.2 of the same page); it is the exact gradient of
 * <dO, O>.  Its workspace holds D = rowsum(dO * O) and an fp32 dQ
 * accumulator.
 *
 * Layout: every tensor is contiguous row-major [B, H, N, d] with d innermost
 * (the (batch, heads, seq, head_dim) order of §11.1); LSE and D are [B, H, N_q].
 * Element types: Q, K, V, O, dO, dQ, dK, dV bf16; LSE fp32.
 *
 * Ownership: all pointers are DEVICE pointers owned by the caller.  The
 * library never frees or keeps them; calls are asynchronous on `stream`
 * (0 = the legacy default stream) and write only the named outputs (and, for
 * fa_bwd, the caller's workspace).
 *
 * Errors: every entry point returns an fa_status.  Argument checks happen on
 * the host before anything is launched; a rejected call launches nothing and
 * leaves all buffers untouched.  Besides sizes and alignment they include the
 * memory behind every tensor and workspace pointer: it must be device memory
 * the current device can address (cudaMalloc, a memory pool, managed memory);
 * host memory, pinned or not, is refused with FA_ERR_INVALID.  A launch failure returns FA_ERR_CUDA.  Every
 * wait inside the kernels is bounded in time; a wait that runs out sets a
 * device status word that fa_get_last_device_status() reports as
 * FA_ERR_TIMEOUT (the outputs of that call are then undefined).  Nothing
 * aborts, exits or throws across this interface.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID = 1,      /* null or non-device pointer, size < 1, causal not 0/1, bad scale */
  FA_ERR_UNSUPPORTED = 2,  /* head dimension d not supported by the call; no sm_103 device */
  FA_ERR_ALIGN = 3,        /* a pointer not 16-byte aligned (TMA requirement) */
  FA_ERR_WORKSPACE = 4,    /* fa_bwd workspace null or smaller than required */
  FA_ERR_CUDA = 5,         /* a CUDA runtime/driver call or a launch failed */
  FA_ERR_TIMEOUT = 6       /* a bounded in-kernel wait ran out (device status) */
} fa_status;

/* Opaque CUDA stream (cudaStream_t); 0 selects the legacy default stream. */
typedef void* fa_stream_t;

/*
 * fa_fwd -- forward attention.
 *   Q   bf16 [B, H, N_q,  d]      K, V bf16 [B, H, N_kv, d]
 *   O   bf16 [B, H, N_q,  d]      (output; fully overwritten, never read)
 *   LSE fp32 [B, H, N_q]          (output; natural-log logsumexp of scale*QK^T)
 *   B, H, N_q, N_kv >= 1; d in {64, 128, 256}; causal in {0, 1};
 *   scale finite and > 0 (typically 1/sqrt(d)).
 * Returns FA_OK once the kernel is enqueued on `stream`.  (d = 256, one of
 * the head dimensions of the sweep in "FlashAttention-3: Fast and Accurate
 * Attention with Asynchrony and Low-precision" 実験設定, has a forward
 * kernel of its own; the backward covers d in {64, 128}.)
 */
int fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
           int B, int H, int N_q, int N_kv, int d, int causal, float scale,
           fa_stream_t stream);

/*
 * fa_fwd_ex -- fa_fwd with the two exact-attention tuning knobs exposed.
 *   tau      conditional-rescaling threshold in log2 units ("論文解説:
 *            FlashAttention-4 ...", 条件付きオンラインsoftmaxリスケーリング):
 *            O and l are rescaled only when a row maximum rises by more than
 *            tau; 0 rescales on every rise.  Must be in [0, 16].  fa_fwd uses 8.
 *   emu_per_32  how many of every 32 exponentials take the FMA-pipe cubic
 *            2^x emulation (same page, ソフトウェア指数関数エミュレーション)
 *            instead of the hardware ex2 unit: one of 0, 8, 16, -1 (-1 = the
 *            library default, which fa_fwd uses).
 * The result is exact attention for every setting, up to rounding.
 */
int fa_fwd_ex(const void* Q, const void* K, const void* V, void* O, float* LSE,
              int B, int H, int N_q, int N_kv, int d, int causal, float scale,
              float tau, int emu_per_32, fa_stream_t stream);

/*
 * fa_fwd_fp8_workspace_bytes -- bytes of device workspace fa_fwd_fp8 needs,
 * in this order, each part rounded up to 256 bytes: e4m3 codes of Q, K and
 * V ([B, H, N rounded up to 128, d] bytes each; rows past N hold +0), fp32
 * multipliers of Q and of K ([B, H, N rounded up to 128 / 128]), the fp32
 * largest |V| of each 128-key block ([B, H, N_kv rounded up to 128 / 128])
 * and of each (batch, head) ([B, H]).  0 for invalid sizes or d not in
 * {128, 256}.
 */
size_t fa_fwd_fp8_workspace_bytes(int B, int H, int N_q, int N_kv, int d);

/*
 * fa_fwd_fp8 -- forward attention on 8-bit (e4m3) copies of Q, K and V, the
 * low-precision path of "FlashAttention-3: Fast and Accurate Attention with
 * Asynchrony and Low-precision" 技術 3 (block quantisation and incoherent
 * processing).
 *   Q, K, V, O, LSE, sizes, causal, scale: as fa_fwd; d is 128 or 256
 *   (else FA_ERR_UNSUPPORTED).
 *   signs    host pointer to d/32 32-bit words, or NULL.  Not NULL: before
 *            quantisation every row of Q and K has the channels whose bit is
 *            set (bit c % 32 of word c / 32) negated and is multiplied by the
 *            d x d Hadamard matrix (Sylvester order, entries +-1; the logit
 *            scale is divided by d to match)
 *            (the same random orthogonal matrix for Q and K, so Q K^T is
 *            unchanged); NULL: plain block quantisation.
 *   Quantisation: one multiplier 448 / amax per 128-row block of Q and of K
 *   (per batch and head), one per (batch, head) for V; codes are the
 *   products rounded to e4m3 (nearest even, saturating).  The products
 *   accumulate in fp32; P is rounded to e4m3 for P V.  O is bf16, LSE fp32.
 *   workspace: at least fa_fwd_fp8_workspace_bytes(...) bytes, 256-byte
 *   aligned, owned by the caller; rewritten by the call.
 * Returns FA_OK once the work is enqueued on `stream`.
 */
int fa_fwd_fp8(const void* Q, const void* K, const void* V, void* O, float* LSE,
               int B, int H, int N_q, int N_kv, int d, int causal, float scale,
               const unsigned int* signs, void* workspace, size_t workspace_bytes,
               fa_stream_t stream);

/*
 * fa_bwd_workspace_bytes -- bytes of device workspace fa_bwd / fa_bwd_ex need
 * for this problem: an fp32 dQ accumulator [B, H, N_q, d], then two fp32 row
 * vectors D = rowsum(dO * O) and LSE * log2(e), each [B, H, N_q rounded up
 * to a multiple of 128], then one 32-bit counter per 128-row query tile
 * [B, H, ceil(N_q / 128)], then one 32-bit ticket counter; every part is
 * rounded up to 256 bytes.  Returns 0 for invalid sizes and for d = 256 (no
 * backward).
 */
size_t fa_bwd_workspace_bytes(int B, int H, int N_q, int N_kv, int d);

/*
 * fa_bwd -- backward attention.
 *   Q, K, V, O, dO bf16 as in fa_fwd; LSE fp32 [B, H, N_q] from fa_fwd on the
 *   same inputs.  dQ bf16 [B, H, N_q, d], dK, dV bf16 [B, H, N_kv, d]
 *   (outputs; fully overwritten).  workspace: device memory of at least
 *   fa_bwd_workspace_bytes(...) bytes, 256-byte aligned, owned by the caller;
 *   its contents on entry are ignored (it is cleared inside the call).
 * Same size, causal and scale rules as fa_fwd; d in {64, 128} (256:
 * FA_ERR_UNSUPPORTED).
 */
int fa_bwd(const void* Q, const void* K, const void* V, const void* O,
           const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
           int B, int H, int N_q, int N_kv, int d, int causal, float scale,
           void* workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * fa_bwd_ex -- fa_bwd with a choice of reduction order for dQ.
 *   deterministic 0: as fa_bwd -- the partial dQ of every 128-key tile is
 *                    added into the fp32 accumulator in whatever order the
 *                    tiles finish (fastest; results may differ in the last
 *                    bits from run to run).
 *   deterministic 1: the partials of each 128-row query tile are added in a
 *                    fixed order (decreasing key tile), so repeated calls on
 *                    the same inputs give bit-identical dQ, dK and dV
 *                    ("論文解説: FlashAttention-4 ...", 実験結果: the
 *                    deterministic backward mode).  Key tiles then wait for
 *                    one another through the workspace counters; the work
 *                    items are numbered in the order their thread blocks
 *                    start, so a block only ever waits for blocks that are
 *                    already running, whatever else runs on the device.
 * Other arguments, the workspace and the errors are those of fa_bwd;
 * deterministic outside {0, 1} returns FA_ERR_INVALID.
 */
int fa_bwd_ex(const void* Q, const void* K, const void* V, const void* O,
              const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
              int B, int H, int N_q, int N_kv, int d, int causal, float scale,
              int deterministic, void* workspace, size_t workspace_bytes,
              fa_stream_t stream);

/*
 * fa_bwd_pair -- fa_bwd at head dimension 64 on pairs of thread blocks that
 * share their tensor-core products ("論文解説: FlashAttention-4 ...",
 * Backwardパスの最適化, item 2: 2-CTA MMA mode, 256-row tiles across two
 * CTAs).  Each pair of blocks (a cluster of two) owns 256 keys; every product
 * is one instruction for both blocks, and each 128-row query tile receives
 * one fp32 dQ partial per 256 keys instead of one per 128, so the dQ
 * reduce-adds into the workspace halve.  The result is the same gradient as
 * fa_bwd's up to the order of fp32 additions; the dQ reduction order is not
 * fixed (as fa_bwd, not fa_bwd_ex's fixed order).
 * Arguments, workspace (fa_bwd_workspace_bytes) and errors are those of
 * fa_bwd; d other than 64 returns FA_ERR_UNSUPPORTED.
 */
int fa_bwd_pair(const void* Q, const void* K, const void* V, const void* O,
                const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                int B, int H, int N_q, int N_kv, int d, int causal, float scale,
                void* workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * fa_bwd_noalloc -- fa_bwd for callers that cannot allocate device memory.
 *
 * (The pages describe no such call; it is an interface convenience.)  Some
 * callers have no way to obtain a workspace: code embedded in a host
 * framework that hands it only the input and output buffers, servers that
 * forbid allocation on the request path because cudaMalloc can fail under
 * memory pressure and cudaFree synchronises the whole device, or processes
 * whose device memory is reserved up front.  This entry point takes the same
 * arguments as fa_bwd without the workspace and uses scratch memory the
 * library reserves in device memory when it is loaded:
 * FA_BWD_NOALLOC_MAX_WORKSPACE bytes on every GPU that loads the library,
 * held until the process exits.  It allocates nothing.
 *
 *   - Problems whose fa_bwd_workspace_bytes(...) exceeds
 *     FA_BWD_NOALLOC_MAX_WORKSPACE return FA_ERR_WORKSPACE and launch nothing
 *     (at d = 128 that is about 32,000 query rows B*H*N_q; use fa_bwd with a
 *     workspace of your own beyond that).  Other argument errors are those
 *     of fa_bwd.
 *   - Every call looks up the scratch's device address on the current
 *     device (a CUDA runtime query, no allocation), so the address stays
 *     right if the device's context is reset.  The first call on a device may
 *     load the library's device code there; make that first call before any
 *     stream capture on that device.
 *   - Every call on a device shares the one scratch area.  Each call clears
 *     what it needs before using it, but calls that can overlap on the GPU
 *     (for example on two streams without ordering between them) race on it
 *     and give wrong results: order such calls, or use fa_bwd.
 */
#define FA_BWD_NOALLOC_MAX_WORKSPACE ((size_t)16 << 20)

int fa_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O,
                   const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                   int B, int H, int N_q, int N_kv, int d, int causal, float scale,
                   fa_stream_t stream);

/*
 * fa_get_last_device_status -- synchronise `stream`, then read and clear the
 * device status word of the current device.  Returns FA_OK, FA_ERR_TIMEOUT if
 * a bounded wait in any kernel of this library ran out since the last call,
 * FA_ERR_UNSUPPORTED if a kernel found its launch unusable on this device
 * (it then returned without computing), or FA_ERR_CUDA if the
 * synchronisation itself failed.
 */
int fa_get_last_device_status(fa_stream_t stream);

/*
 * fa_set_wait_timeout_ns -- time limit of every in-kernel wait, in
 * nanoseconds, for launches made after this call (process-wide; default
 * 1e9 = 1 s).  Values outside [1e3, 1e11] return FA_ERR_INVALID.
 */
int fa_set_wait_timeout_ns(unsigned long long ns);

/* fa_status_string -- a static, NUL-terminated description of a status code. */
const char* fa_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
