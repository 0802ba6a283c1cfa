/*
 * fp8fg.h -- C ABI of the GB300 (sm_103a) fine-grained FP8 quantization and
 * block-scaled FP8 GEMM library (libfp8fg.so).
 *
 * The method: online E4M3 quantization with one FP32 scale per group,
 * s = amax / 448 of the current group (no history), 1x128 tiles for
 * activations and gradients and 128x128 blocks for FP32 master weights; then
 * an FP8 GEMM that accumulates each 128-wide K chunk on the tensor cores,
 * multiplies the chunk's partial sums by the two group scales and promotes
 * them into FP32 accumulators, writing FP32 or BF16.
 *   - DeepSeek-V3 FP8 post (innerforce.co.kr), fine-grained quantization,
 *     Figure 7 (a): 1x128 tiles per token per 128 channels, 128x128 blocks
 *     per 128 input x 128 output channels, max-abs scaled to the FP8 maximum;
 *     the increased-precision accumulation paragraph (FP8 MMA on H800 keeps
 *     about 14 bits, so partial sums are promoted to FP32).
 *   - "DeepSeek FP8 Training" (arcalunar.github.io): the Fprop, Wgrad and
 *     Dgrad pipelines (operand roles, FP32 accumulation, BF16 / FP32 outputs).
 *   - "Unified E4M3 format in DeepSeek-V3" (codingmall.com): E4M3 for every
 *     tensor, online scales, promotion of partial results to FP32 registers
 *     at fixed intervals (Fine-Grained Quantization Strategy; Dynamic Scaling
 *     and Online Quantization; Enhanced Numerical Stability).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers (CUDA global memory), owned by
 *     the caller, who allocates every buffer.  Entry points allocate nothing
 *     and keep no per-call state.  Row-major layouts, last index contiguous.
 *   - All calls are asynchronous on `stream` (0 = the legacy default stream)
 *     and stream-ordered; none synchronises the host.  They are thread-safe.
 *   - Shapes are element counts (int64).  Returned: an fp8fg_status.  Argument
 *     errors are detected on the host before anything is launched, and then
 *     nothing is written.  A device that is not compute capability 10.3 gives
 *     FP8FG_ERR_UNSUPPORTED_DEVICE (there is no fallback path).
 *   - Every bounded wait inside a kernel that runs out of time records
 *     FP8FG_ERR_TIMEOUT in a library-owned device status word, which
 *     fp8fg_last_device_status() reads; such a kernel returns without hanging.
 *   - E4M3 is the OCP FP8 E4M3 format (bias 7, max 448, no infinities).
 *     Element codes are enc_RNE_satfinite(fl32(x / s)) with an IEEE division;
 *     a group whose scale is 0 (all zeros, or amax/448 underflowing in FP32)
 *     stores s = 0 and codes that keep only the sign of x.  Inputs are finite
 *     (NaN/Inf input gives unspecified codes).
 */
#ifndef FP8FG_H
#define FP8FG_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP8FG_OK = 0,
    FP8FG_ERR_INVALID_ARG = 1,        /* null pointer, bad enum, negative or non-tiling shape */
    FP8FG_ERR_MISALIGNED = 2,         /* a pointer breaks its alignment rule (16 bytes; 4 for scales) */
    FP8FG_ERR_UNSUPPORTED_DEVICE = 3, /* current device is not sm_103 */
    FP8FG_ERR_CUDA = 4,               /* a CUDA runtime/driver call or a launch failed */
    FP8FG_ERR_TIMEOUT = 5,            /* (device status) a bounded wait ran out */
    FP8FG_ERR_TEARDOWN = 6,           /* (device status) after a failed wait, the kernel's bounded wait for its
                                         own TMA copies or MMAs in flight ran out too before it freed shared
                                         and tensor memory; replaces an earlier FP8FG_ERR_TIMEOUT */
    FP8FG_ERR_TOO_LARGE = 7           /* the problem exceeds a fixed-size buffer of the library
                                         (fp8_gemm_quant_a_noalloc: M > 524288) */
} fp8fg_status;

typedef enum { FP8FG_OUT_F32 = 0, FP8FG_OUT_BF16 = 1 } fp8fg_out_dtype;

/* Grouping axis of the activation quantizer. */
typedef enum {
    FP8FG_AXIS_COLS = 0, /* 1x128: groups of 128 consecutive columns of one row */
    FP8FG_AXIS_ROWS = 1  /* 128x1: groups of 128 consecutive rows of one column; output transposed */
} fp8fg_axis;

/* How the GEMM's B operand is scaled. */
typedef enum {
    FP8FG_BSCALE_BLOCK128 = 0, /* one scale per 128 (N) x 128 (K) block */
    FP8FG_BSCALE_ROW = 1       /* one scale per row of B per 128-wide K chunk */
} fp8fg_bscale;

/*
 * fp8_quant_act_1x128 -- online E4M3 quantization of a BF16 activation or
 * gradient x[rows, cols] (row-major, 2-byte elements).
 *   axis FP8FG_AXIS_COLS (Fprop X, Dgrad dY; "per token per 128 channels",
 *   Figure 7 (a) of the DeepSeek-V3 FP8 post):
 *     requires cols % 128 == 0 (rows >= 0 arbitrary);
 *     q[rows, cols] uint8 E4M3 codes;
 *     scales[cols/128, rows] float32: scales[c*rows + i] belongs to the group
 *     x[i, 128c .. 128c+127].
 *   axis FP8FG_AXIS_ROWS (Wgrad operands, whose reduction runs over tokens:
 *   "DeepSeek FP8 Training", backward pass step 1):
 *     requires rows % 128 == 0 and cols % 8 == 0 (16-byte rows of x);
 *     q[cols, rows] uint8, i.e. the codes TRANSPOSED (K-major for the Wgrad GEMM);
 *     scales[rows/128, cols] float32: scales[t*cols + j] belongs to the group
 *     x[128t .. 128t+127, j].
 * x and q must be 16-byte aligned, scales 4-byte aligned.  rows == 0 or
 * cols == 0 is a no-op.
 */
int fp8_quant_act_1x128(const void *x_bf16, int64_t rows, int64_t cols, int axis,
                        uint8_t *q, float *scales, cudaStream_t stream);

/*
 * fp8_quant_act_dual -- both activation quantizations of one BF16 tensor
 * from a single read of it: the 1x128 row groups of fp8_quant_act_1x128
 * with axis FP8FG_AXIS_COLS and the 128x1 column groups (transposed output)
 * of axis FP8FG_AXIS_ROWS, bit for bit the same codes and scales.  The
 * forward pass caches the activation in FP8 for the backward pass (DeepSeek-V3
 * FP8 post, low-precision storage paragraph), which needs the 1x128 copy for
 * the next layer's GEMM and the token-axis copy for the weight gradient
 * ("DeepSeek FP8 Training", Wgrad step 1).
 *
 *   x_bf16  [rows, cols] BF16, row-major, 16-byte aligned.
 *   q_row   [rows, cols] E4M3 codes;       s_row [cols/128, rows] FP32.
 *   q_col_t [cols, rows] E4M3 codes;       s_col [rows/128, cols] FP32.
 *   rows and cols multiples of 128, cols/128 <= 65535; x and the codes
 *   16-byte aligned, the scales 4-byte aligned; all owned by the caller.
 *   rows == 0 or cols == 0 is a no-op.
 * Errors: FP8FG_ERR_INVALID_ARG (shape, NULL), FP8FG_ERR_MISALIGNED,
 * FP8FG_ERR_UNSUPPORTED_DEVICE, FP8FG_ERR_CUDA (launch).
 */
int fp8_quant_act_dual(const void *x_bf16, int64_t rows, int64_t cols, uint8_t *q_row, float *s_row,
                       uint8_t *q_col_t, float *s_col, cudaStream_t stream);

/*
 * fp8_quant_w_128x128 -- online E4M3 quantization of an FP32 master weight
 * w[rows, cols] in 128x128 blocks ("per 128 input channels per 128 output
 * channels", Figure 7 (a) of the DeepSeek-V3 FP8 post; the FP32 master is
 * cast to FP8 each step: "DeepSeek FP8 Training", forward step 2).
 *   requires rows % 128 == 0 and cols % 128 == 0;
 *   q[rows, cols] uint8 E4M3 codes;
 *   q_t: NULL, or q_t[cols, rows] uint8 receiving the same codes transposed
 *        (the K-major B operand of the Dgrad GEMM; a block's scale is the
 *        same in both orientations);
 *   scales[rows/128, cols/128] float32, row-major.
 * w, q and q_t 16-byte aligned, scales 4-byte aligned (so that experts can be
 * quantized one by one into slices of a [G, rows/128, cols/128] array).
 * rows == 0 or cols == 0 is a no-op.
 */
int fp8_quant_w_128x128(const float *w, int64_t rows, int64_t cols,
                        uint8_t *q, uint8_t *q_t, float *scales, cudaStream_t stream);

/*
 * fp8_gemm_blockscaled -- D[M, N] = A[M, K] . B[N, K]^T with per-group
 * scales, both operands K-major E4M3 ("DeepSeek FP8 Training": Fprop
 * Y = X W^T, Dgrad dX = dY W, Wgrad dW = dY^T X).  For every 128-wide K
 * chunk c the tensor cores form P = sum_{k in c} a[i,k] b[j,k] in FP32 and
 * the kernel adds P * (sa[c, i] * sb(j, c)) into FP32 accumulators (the
 * promotion at fixed intervals of "Unified E4M3 format in DeepSeek-V3",
 * Enhanced Numerical Stability; interval = one 128-wide group).
 *   a[M, K] uint8, sa[K/128, M] float32 (the layout fp8_quant_act_1x128 writes);
 *   b[N, K] uint8;
 *   bscale FP8FG_BSCALE_BLOCK128: sb(j, c) = sb[(j/128)*sb_stride_n + c*sb_stride_k]
 *     (a weight's [N/128, K/128] scales: strides (K/128, 1); Dgrad reads the
 *     same array transposed with strides (1, N_w/128));
 *   bscale FP8FG_BSCALE_ROW: sb(j, c) = sb[c*N + j], sb[K/128, N] (the
 *     layout of the 128x1 activation quantizer; Wgrad);
 *     sb_stride_n and sb_stride_k are ignored;
 *   d[M, N]: float32 (out_dtype FP8FG_OUT_F32) or bfloat16 rounded to
 *     nearest even (FP8FG_OUT_BF16).
 * Requires N % 128 == 0 and K % 128 == 0; with per-row B scales also
 * M % 128 == 0 (Wgrad: M = output channels, K = tokens, padded to 128 by
 * the caller), while block B scales take any M >= 0 (Fprop, Dgrad:
 * M = tokens; the last 128-row tile is then partial: its missing rows read
 * as zero codes and are not written); a, b and d 16-byte aligned; sa and sb
 * 4-byte aligned for block scales, both 16-byte aligned for per-row B
 * scales (the kernel reads B scales in 8-byte pairs there); sb strides >= 0.
 * K == 0 writes zeros.  M == 0 or N == 0 is a no-op.
 * Accuracy (tested): |d - o| <= 2^-16 * sum_k |a~ b~| for FP32 output, plus
 * one BF16 spacing of o for BF16 output, o being the exact sum of the
 * dequantized products.
 */
int fp8_gemm_blockscaled(const uint8_t *a, const float *sa,
                         const uint8_t *b, const float *sb, int bscale,
                         int64_t sb_stride_n, int64_t sb_stride_k,
                         void *d, int out_dtype, int64_t M, int64_t N, int64_t K,
                         cudaStream_t stream);

/*
 * fp8_gemm_quant_a -- the activation quantizer fused into the GEMM: one
 * launch computes what fp8_quant_act_1x128 (axis FP8FG_AXIS_COLS) on the BF16
 * A operand followed by fp8_gemm_blockscaled with 128x128 block B scales
 * computes, bit for bit (Fprop Y = X W^T and Dgrad dX = dY W of "DeepSeek
 * FP8 Training", with the 1x128 activation groups of the DeepSeek-V3 FP8
 * post's Figure 7 (a)).  A persistent kernel quantizes every 128-row band of
 * A once -- each CTA a share of the 128x128 tiles -- into q_a / s_a, then,
 * once every band is complete, runs the block-scaled GEMM on them; the
 * quantized A is not re-read by a second launch and usually still sits in
 * L2 when the GEMM's TMA loads it.
 *   a_bf16[M, K] BF16 (16-byte aligned);
 *   q_a[M, K] uint8 and s_a[K/128, M] float32: OUTPUTS, written with the
 *     codes and scales of fp8_quant_act_1x128 (q_a 16-byte, s_a 4-byte
 *     aligned);
 *   b[N, K], sb, sb_stride_n, sb_stride_k, d, out_dtype: as
 *     fp8_gemm_blockscaled with FP8FG_BSCALE_BLOCK128;
 *   band_flags: DEVICE int32[M/128] workspace owned by the caller (4-byte
 *     aligned), one counter per 128-row band of A; the call zeroes it on
 *     `stream` before the kernel, so its contents on entry do not matter and
 *     it must not be used by another call running at the same time.
 * Requires M, N, K multiples of 128.  The kernel is launched cooperatively
 * (every CTA resident at once, one per SM): a device or context that cannot
 * host that gives FP8FG_ERR_CUDA.  Its wait for the other CTAs' share of A
 * is bounded (fp8fg_set_wait_limit; FP8FG_ERR_TIMEOUT in the device status
 * word, nothing computed).  M == 0 is a no-op; N == 0 only quantizes A;
 * K == 0 writes D = 0.  Other errors as fp8_gemm_blockscaled.
 */
int fp8_gemm_quant_a(const void *a_bf16, uint8_t *q_a, float *s_a,
                     const uint8_t *b, const float *sb, int64_t sb_stride_n, int64_t sb_stride_k,
                     void *d, int out_dtype, int64_t M, int64_t N, int64_t K,
                     int32_t *band_flags, cudaStream_t stream);

/*
 * fp8_gemm_grouped -- grouped MoE-expert GEMM: rows [off[g], off[g+1]) of A
 * multiply expert weight g: D[r, :] = A[r, :] . B[g]^T with 128x128 block
 * scales (MoE training with FP8 activations, DeepSeek-V3 FP8 post; one
 * weight per expert, tokens grouped contiguously per expert).
 *   a[M_total, K] uint8, sa[K/128, M_total];
 *   b[G, N, K] uint8, sb[G, N/128, K/128] float32;
 *   group_offsets: DEVICE int32[G+1], non-decreasing, off[0] = 0,
 *     off[G] = M_total, every entry a multiple of 128 (groups padded with
 *     zero rows); empty groups allowed;
 *   d[M_total, N] float32 or bfloat16.
 * Requires M_total % 128 == 0, N % 128 == 0, K % 128 == 0, 1 <= G <= 4096;
 * a, b and d 16-byte aligned, sa and sb 4-byte aligned, group_offsets 4-byte
 * aligned.  Offsets that break these rules are detected on the device: the kernel
 * records FP8FG_ERR_INVALID_ARG in the device status word and writes nothing.
 */
int fp8_gemm_grouped(const uint8_t *a, const float *sa,
                     const uint8_t *b, const float *sb,
                     const int32_t *group_offsets, int G,
                     void *d, int out_dtype, int64_t M_total, int64_t N, int64_t K,
                     cudaStream_t stream);

/*
 * fp8_gemm_quant_a_noalloc -- fp8_gemm_quant_a for callers that cannot
 * allocate its band-counter workspace.  The pages have no counterpart: this
 * is a service of the library, not a step of the method.
 *
 * Who needs it: code that owns no device allocator (a host program or plugin
 * handed raw device pointers by another runtime, or whose host framework
 * forbids device allocations behind its own allocator) and code that must
 * not allocate in its steady state.  The call allocates nothing (no
 * cudaMalloc or cudaFree, no allocating library routine); instead the
 * counters live in a fixed array in the library's device memory: 4096 int32
 * counters (16 KB), held on every GPU that loads the library until the
 * process exits.
 *
 * Arguments, results and errors as fp8_gemm_quant_a (same kernel, same
 * output, bit for bit), without band_flags; additionally M > 4096 * 128 =
 * 524288 gives FP8FG_ERR_TOO_LARGE before anything is launched.
 * The first call on a device looks up the array's device address with
 * cudaGetSymbolAddress (a runtime call made once per device, with that
 * device current; FP8FG_ERR_CUDA if it fails): make the first call on each
 * device before any stream capture begins.
 * Every call on a device uses the same array, and each call zeroes it on
 * `stream` before its kernel runs.  Calls whose work overlaps on the GPU
 * (other streams, or other host threads, without ordering between them)
 * race on the array and may compute wrong results or fail: order such calls
 * one after another.
 */
int fp8_gemm_quant_a_noalloc(const void *a_bf16, uint8_t *q_a, float *s_a,
                             const uint8_t *b, const float *sb, int64_t sb_stride_n, int64_t sb_stride_k,
                             void *d, int out_dtype, int64_t M, int64_t N, int64_t K,
                             cudaStream_t stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char *fp8fg_status_string(int status);

/*
 * fp8fg_check_compute_capability -- the device rule every entry point
 * applies to the current device before any launch: FP8FG_OK for compute
 * capability 10.3 (sm_103: the kernels use tcgen05, TMEM and TMA as
 * compiled for that architecture only), FP8FG_ERR_UNSUPPORTED_DEVICE for
 * any other; there is no fallback path.  Pure function of its arguments
 * (touches no device), so the rule can be checked without such a device.
 */
int fp8fg_check_compute_capability(int major, int minor);

/*
 * fp8fg_last_device_status -- read and clear the device status word of the
 * current device (an asynchronous error recorded by a kernel: a bounded
 * wait that ran out, or invalid grouped offsets).  The word is one per
 * device, shared by every stream: the first error recorded since the last
 * read wins (FP8FG_ERR_TEARDOWN overrides it).  The read and the clear are
 * one atomic exchange on the device, ordered after the work already queued
 * on `stream`; kernels queued on other streams are included only if the
 * caller has ordered them before (synchronise those streams first).
 * Synchronises `stream`.  Returns FP8FG_OK when no kernel recorded anything
 * since the last read.
 */
int fp8fg_last_device_status(cudaStream_t stream);

/*
 * fp8fg_set_wait_limit -- limit, in nanoseconds, of the GEMM kernels' bounded
 * waits on their producer and consumer barriers (TMA data, scale ring, MMA
 * completion), for every later launch in this process on any device.
 * 0 restores the default of 2 s; allowed range 0 .. 10^10.  A wait that runs
 * out records FP8FG_ERR_TIMEOUT in the device status word and the kernel
 * winds down without computing (its output is then undefined) and returns.
 * A very short limit makes the waits run out on purpose (a test of those
 * paths).  The pages describe no such control: it belongs to this library's
 * failure detection.  Returns FP8FG_ERR_INVALID_ARG outside the range.
 */
int fp8fg_set_wait_limit(int64_t limit_ns);

/*
 * fp8fg_selftest_watchdog -- test hook for the kernels' bounded waits: runs a
 * one-warp kernel that waits on an mbarrier nobody arrives on, with a limit
 * of `timeout_ns` nanoseconds (1 .. 10^9).  The wait gives up, records
 * FP8FG_ERR_TIMEOUT in the device status word and the kernel returns.
 * The caller reads it with fp8fg_last_device_status().  No fault, no trap.
 */
int fp8fg_selftest_watchdog(int64_t timeout_ns, cudaStream_t stream);

/*
 * fp8fg_probe_mma_rate -- measurement hook: the tensor-core ceiling of the
 * GEMM's own MMA.  Launches one CTA per SM (their number is written to
 * *num_ctas), each issuing `chunks` (1 .. 2^24) x 4 back-to-back
 * tcgen05.mma.kind::f8f6f4 of 128 x 256 x 32 on a fixed pattern of E4M3
 * codes in shared memory, with no data movement, promotion or output.  The
 * caller times the launch on `stream`; its work is
 * *num_ctas * chunks * 2 * 128 * 256 * 128 FLOP.  The pages have no
 * counterpart: it gives the block-scaled GEMM a measured denominator.  Its
 * wait for the MMAs is bounded (fp8fg_set_wait_limit) and reports through
 * the device status word.
 */
int fp8fg_probe_mma_rate(int64_t chunks, int *num_ctas, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* FP8FG_H */
