/*
 * bnb_int8.h -- C ABI of the LLM.int8() mixed-precision decomposition linear
 * for NVIDIA B300 (sm_103a).
 *
 * The operation (Y = X W^T with outlier decomposition) is the one the pages
 * describe as LLM.int8(): feature dimensions of the activations whose values
 * are large ("outliers") are multiplied in 16-bit, every other value is
 * quantized vector-wise to int8, multiplied in int8 and converted back to
 * 16-bit at the end ("Hugging Face Quantization with bitsandbytes: 4-bit &
 * 8-bit Models Explained", section 2 "LLM.int8(): Quantizing Without
 * Degrading Large Models"; "bitsandbytes: GPU-Accelerated Inference and
 * Training at Lower Bit Depths", section "How LLM.int8() quantizes weights
 * and activations").  The outlier cut-off is llm_int8_threshold, default 6.0
 * (same Hugging Face page, section 3).  Weights are quantized once, when the
 * model is loaded ("bitsandbytes" glossary page, introduction).
 *
 * Definitions used by every call (T tokens, K features, N output channels):
 *   O       = { k : |X[t,k]| >= tau for some t }, ascending       (outliers)
 *   sx[t]   = max over k not in O of |X[t,k]|                     (row scale)
 *   sw[n]   = max over all k of |W[n,k]|                          (channel scale)
 *   Xq[t,k] = 0 for k in O, else rint(fl32(127 X[t,k]) / sx[t])    (ties to even;
 *             0 when sx[t] = 0); Wq likewise with sw[n]
 *   acc     = Xq Wq^T, exact int32
 *   Y[t,n]  = fp16( acc[t,n] * (sx[t]/127) * (sw[n]/127)
 *                   + sum_{k in O} X[t,k] * W16[n,k] )
 *
 * Conventions shared by all entry points:
 *   - Every data pointer is a DEVICE pointer to a dense row-major array; the
 *     caller allocates and owns all of them.  The library never allocates,
 *     frees or synchronises (except bnb_last_device_status, which syncs the
 *     given stream).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously on it.
 *   - fp16 data is IEEE binary16, passed as void*; the `_ex` entry points
 *     also take bfloat16 (bnb_dtype_t) for X, W16, the bias and Y.
 *   - Argument errors are detected on the host before anything is enqueued;
 *     in that case nothing is written.
 *   - Alignment: every pointer 16-byte aligned, K a multiple of 16.
 *   - Y must not alias X, W16, Wq or the workspace.
 *   - X must be finite.  tau may be +INFINITY (no outliers); tau NaN or
 *     negative is an argument error.
 *   - Calls on different streams with different workspaces may run
 *     concurrently; two calls that share a workspace must be ordered.
 */
#ifndef BNB_INT8_H
#define BNB_INT8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  BNB_OK = 0,
  BNB_ERR_INVALID_ARG = 1, /* NULL pointer, T/N/K <= 0, tau NaN or < 0,
                              workspace too small, aliasing output */
  BNB_ERR_UNSUPPORTED = 2, /* K % 16 != 0, pointer not 16-byte aligned,
                              size beyond the limits below, device is not
                              compute capability 10.3 */
  BNB_ERR_CUDA = 3,        /* a CUDA call or kernel launch failed */
  BNB_ERR_TIMEOUT = 4      /* a bounded device-side wait gave up; reported
                              through bnb_last_device_status */
} bnb_status_t;

/* The 16-bit element format of X, W16, the bias and Y (the codes, scales
 * and accumulators do not depend on it).  bf16 is the compute dtype the pages
 * prefer where the hardware supports it (Hugging Face page, section 5
 * "Storage Precision vs. Compute Precision"). */
typedef enum { BNB_DTYPE_FP16 = 0, BNB_DTYPE_BF16 = 1 } bnb_dtype_t;

/* Size limits of one call. */
#define BNB_MAX_K (1 << 20)
#define BNB_MAX_T (1 << 22)
#define BNB_MAX_N (1 << 22)

/*
 * Bytes of device workspace that bnb_int8_linear / bnb_int8_linear_debug
 * need for a call of this shape (0 for a non-positive dimension).  The
 * workspace holds the outlier column mask and index list, the row scales,
 * the activation codes, the fp16 outlier block of X and W16's outlier
 * columns for the GEMM path; it needs no initialisation and its contents
 * after a call are unspecified except the device status word read by
 * bnb_last_device_status.
 */
size_t bnb_int8_linear_workspace_bytes(int64_t T, int64_t N, int64_t K);

/*
 * Weight quantization, run once per weight (at load time).
 *   W16    [N x K] fp16, input.
 *   Wq     [N x K] int8, output: Wq[n,k] = rint(fl32(127 W16[n,k]) / sw[n]).
 *   Wscale [N] fp32, output: sw[n] = max_k |W16[n,k]| (absmax, not absmax/127).
 * Errors: BNB_ERR_INVALID_ARG (NULL, N<=0, K<=0), BNB_ERR_UNSUPPORTED
 * (alignment, K % 16, limits, device), BNB_ERR_CUDA (launch).
 */
bnb_status_t bnb_int8_quantize_weight(const void *W16, int64_t N, int64_t K,
                                      int8_t *Wq, float *Wscale, void *stream);

/*
 * The decomposition linear Y = X W^T (definitions above).
 *   X      [T x K] fp16 activations.
 *   Wq     [N x K] int8 and Wscale [N] fp32 from bnb_int8_quantize_weight.
 *   W16    [N x K] fp16 weight, source of the outlier columns.
 *   tau    outlier threshold (>= 0, may be +INFINITY).
 *   Y      [T x N] fp16 output, written once.
 *   workspace/workspace_bytes: at least bnb_int8_linear_workspace_bytes(T,N,K).
 * The outlier set is computed per call from all T rows and stays on the
 * device.  Errors as for bnb_int8_quantize_weight, plus BNB_ERR_INVALID_ARG
 * for a small workspace.  A device-side wait that gives up writes
 * BNB_ERR_TIMEOUT into the workspace status word.
 */
bnb_status_t bnb_int8_linear(const void *X, int64_t T, int64_t K, const int8_t *Wq,
                             const float *Wscale, const void *W16, int64_t N,
                             float tau, void *Y, void *workspace,
                             size_t workspace_bytes, void *stream);

/*
 * bnb_int8_linear with a bias: the layer is a drop-in replacement for
 * PyTorch's Linear (bitsandbytes GPU page, section "How LLM.int8() quantizes
 * weights and activations"), whose bias b is added to x W^T.  b[n] is added
 * in fp32 before the one rounding of Y to fp16:
 *   Y[t,n] = fp16(acc[t,n] sx[t] sw[n] / 127^2 + sum_{j in O} X[t,j] W16[n,j] + b[n]).
 *   bias   [N] fp16 on the device, 16-byte aligned, read only; NULL gives
 *          bnb_int8_linear.  It must not overlap Y.
 * Other arguments, errors and the device status word as for bnb_int8_linear.
 */
bnb_status_t bnb_int8_linear_bias(const void *X, int64_t T, int64_t K, const int8_t *Wq,
                                  const float *Wscale, const void *W16, const void *bias,
                                  int64_t N, float tau, void *Y, void *workspace,
                                  size_t workspace_bytes, void *stream);

/*
 * The layer with only the int8 weight resident: no fp16 copy of W is kept,
 * which halves the weight's bytes against fp16 (Hugging Face page, "Quick
 * Comparison" table; bitsandbytes GPU page, section "Why quantization matters
 * for LLM deployment").  The outlier columns then use the codes dequantized,
 * w[n,k] = Wq[n,k] sw[n] / 127, in the same 16-bit-input product:
 *   Y[t,n] = fp16( (acc[t,n] sx[t]/127 + sum_{j in O} X[t,j] Wq[n,j]) sw[n]/127 + b[n] ),
 * the sums in fp32 in any order, one rounding to fp16.  Arguments as for
 * bnb_int8_linear_bias without W16 (bias may be NULL); errors likewise.
 */
bnb_status_t bnb_int8_linear_wq_only(const void *X, int64_t T, int64_t K, const int8_t *Wq,
                                     const float *Wscale, const void *bias, int64_t N,
                                     float tau, void *Y, void *workspace,
                                     size_t workspace_bytes, void *stream);

/*
 * The general entry points, with the element format `dtype` (a bnb_dtype_t)
 * of W (quantize) or of X, W16, bias and Y (the layer).  With BNB_DTYPE_BF16
 * every fp16 array above is bf16 instead; the definitions are unchanged
 * except that Y is rounded to bf16 (nearest-even) and the codes of bf16
 * values are taken after scaling x and its absmax a by one power of two
 * 2^(1-e), a = f 2^e with f in [0.5, 1) -- the same code 127 x / a, computed
 * without leaving fp32's range (bf16 spans 2^-133 .. 2^128, where 127 x
 * would overflow).  W16 may be NULL (bnb_int8_linear_wq_only) and bias may
 * be NULL.  An unknown dtype is BNB_ERR_INVALID_ARG; other errors as for
 * the fp16 entry points.
 */
bnb_status_t bnb_int8_quantize_weight_ex(const void *W, int64_t N, int64_t K, int dtype,
                                         int8_t *Wq, float *Wscale, void *stream);
bnb_status_t bnb_int8_linear_ex(const void *X, int64_t T, int64_t K, const int8_t *Wq,
                                const float *Wscale, const void *W16, const void *bias, int64_t N,
                                float tau, int dtype, void *Y, void *workspace,
                                size_t workspace_bytes, void *stream);
bnb_status_t bnb_int8_linear_from_host_ex(const void *X_host, int64_t T, int64_t K,
                                          const int8_t *Wq, const float *Wscale, const void *W16,
                                          const void *bias, int64_t N, float tau, int dtype,
                                          void *Y_host, void *X_dev, void *Y_dev,
                                          void *workspace, size_t workspace_bytes,
                                          void *stream);
/* bnb_int8_linear_debug's intermediates (same meaning) for bnb_int8_linear_ex. */
bnb_status_t bnb_int8_linear_debug_ex(const void *X, int64_t T, int64_t K, const int8_t *Wq,
                                      const float *Wscale, const void *W16, const void *bias,
                                      int64_t N, float tau, int dtype, void *Y, void *workspace,
                                      size_t workspace_bytes, void *stream, int8_t *Xq,
                                      float *Xscale, int32_t *outlier_idx, int32_t *n_outliers,
                                      int32_t *acc);

/*
 * bnb_int8_linear that also exports its intermediates (for parity tests).
 * Same arguments as bnb_int8_linear, then (each may be NULL to skip):
 *   Xq          [T x K] int8 activation codes (0 in outlier columns)
 *   Xscale      [T] fp32 row scales sx
 *   outlier_idx [K] int32, entries [0, n_outliers) hold O ascending
 *   n_outliers  [1] int32, |O|
 *   acc         [T x N] int32 exact accumulators Xq Wq^T
 * Y is computed by the same kernels as bnb_int8_linear.
 */
bnb_status_t bnb_int8_linear_debug(const void *X, int64_t T, int64_t K,
                                   const int8_t *Wq, const float *Wscale,
                                   const void *W16, int64_t N, float tau, void *Y,
                                   void *workspace, size_t workspace_bytes,
                                   void *stream, int8_t *Xq, float *Xscale,
                                   int32_t *outlier_idx, int32_t *n_outliers,
                                   int32_t *acc);

/*
 * bnb_int8_linear with the activations and the result in host memory: on
 * `stream`, copies X from X_host into X_dev, runs bnb_int8_linear_bias(X_dev
 * -> Y_dev) and copies Y_dev back into Y_host, so that one call moves a
 * step's input in and its result out.  The pages have no counterpart to this
 * entry point; the layer itself is bnb_int8_linear_bias, unchanged.
 *   bias   [N] fp16 on the device or NULL, as for bnb_int8_linear_bias.
 *   W16    may be NULL: the layer is then bnb_int8_linear_wq_only.
 *   X_host [T x K] fp16 and Y_host [T x N] fp16: host memory.  Page-locked
 *          (pinned) memory makes both copies asynchronous; with pageable
 *          memory the CUDA runtime stages them and the call may block.  The
 *          caller keeps X_host unchanged and Y_host unread until the stream
 *          has passed this call.
 *   X_dev [T x K] and Y_dev [T x N]: device buffers the caller owns (the
 *          same rules as X and Y of bnb_int8_linear; they must not overlap).
 *   Other arguments and errors as for bnb_int8_linear, plus
 *   BNB_ERR_INVALID_ARG for a NULL host or device buffer.  Argument errors
 *   are detected before anything is enqueued.
 */
bnb_status_t bnb_int8_linear_from_host(const void *X_host, int64_t T, int64_t K,
                                       const int8_t *Wq, const float *Wscale, const void *W16,
                                       const void *bias, int64_t N, float tau, void *Y_host,
                                       void *X_dev,
                                       void *Y_dev, void *workspace, size_t workspace_bytes,
                                       void *stream);

/*
 * The blockwise 8-bit codec of optimizer states.  8-bit optimizers keep their
 * states quantized block-wise, each block with its own scaling factor
 * ("bitsandbytes: GPU-Accelerated Inference and Training at Lower Bit
 * Depths", section "8-bit optimizers for full-model training"; page
 * "bitsandbytes", section "What it provides").  Blocks are `block`
 * consecutive values (a power of two from 64 to 2048; the last block may be
 * short); a block's scale is its absmax a.
 *   bnb_int8_quantize_blockwise: x [n] fp32 -> codes [n] int8,
 *     codes[i] = rint(fl32(fl32(127 x[i]) / a)) (IEEE fp32, ties to even; 0
 *     when a = 0), and absmax [ceil(n / block)] fp32.
 *   bnb_int8_dequantize_blockwise: codes [n], absmax -> y [n] fp32,
 *     y[i] = fl32(fl32(codes[i] * a) / 127).
 *   Every finite fp32 input is accepted.  A block with a >= 2^120, where
 *   127 x and codes * a would overflow fp32, is coded as if x and a were
 *   multiplied by 2^-8 and decoded at that scale, the value multiplied back by
 *   2^8.  Both give the formulas above wherever those are finite, and the
 *   codes of such a block are still the integers nearest to 127 x / a.
 * Device pointers, 16-byte aligned, caller-owned; outputs must not overlap
 * inputs.  Errors: BNB_ERR_INVALID_ARG (NULL, n <= 0, overlap),
 * BNB_ERR_UNSUPPORTED (block size, alignment, n > BNB_MAX_BLOCKWISE_N,
 * device), BNB_ERR_CUDA (launch).  The pages give no block size: the
 * Python binding defaults to 256.
 */
#define BNB_MAX_BLOCKWISE_N (1LL << 40)
bnb_status_t bnb_int8_quantize_blockwise(const float *x, int64_t n, int64_t block, int8_t *codes,
                                         float *absmax, void *stream);
bnb_status_t bnb_int8_dequantize_blockwise(const int8_t *codes, const float *absmax, int64_t n,
                                           int64_t block, float *y, void *stream);

/*
 * Synchronises `stream`, then reads the device status word of `workspace`
 * into *out (BNB_OK, or BNB_ERR_TIMEOUT after a bounded wait gave up) and
 * clears it.  Returns BNB_ERR_CUDA if the synchronisation or copy failed.
 */
bnb_status_t bnb_last_device_status(const void *workspace, void *stream, int32_t *out);

/*
 * bnb_int8_linear without a caller-supplied workspace, for callers that
 * cannot allocate device memory: a runtime that plans all device memory
 * ahead of time and forbids allocation once it is serving, a
 * latency-critical loop in which cudaMalloc (which may synchronise the
 * device) is not allowed, or a host framework that owns the device memory
 * and hands out none.  The pages have no counterpart to this entry point; it
 * computes exactly what bnb_int8_linear computes, with the same kernels.
 *
 * The workspace is one static device array of BNB_NOALLOC_SCRATCH_BYTES
 * inside this library, held on every GPU that loads the library until the
 * process exits.  The call allocates nothing (no cudaMalloc, cudaFree or
 * allocating library routine).
 *   Arguments as for bnb_int8_linear, without workspace/workspace_bytes.
 *   Calls whose bnb_int8_linear_workspace_bytes(T, N, K) exceeds
 *   BNB_NOALLOC_SCRATCH_BYTES are rejected with BNB_ERR_UNSUPPORTED before
 *   anything is enqueued (at K = N = 4096 that admits T up to 382).
 *   The first call on a device looks up the array's device address with
 *   that device current (cudaGetSymbolAddress) and caches it; make that first
 *   call before any stream capture.  BNB_ERR_CUDA if the lookup fails.  The
 *   cache assumes that the device's primary context lives as long as the
 *   process uses this entry point: after cudaDeviceReset the cached address
 *   is stale, so do not call this entry point again after a reset.
 *   Every call, on every stream, shares the one array and leaves its contents
 *   behind; each call clears on the device what must start at zero.  Calls
 *   that may overlap on the GPU (different streams, or concurrent host
 *   threads without ordering) race on the array and give undefined results:
 *   order them on one stream.  The device status word of these calls is not
 *   readable through bnb_last_device_status.
 */
#define BNB_NOALLOC_SCRATCH_BYTES (8u << 20)
bnb_status_t bnb_int8_linear_noalloc(const void *X, int64_t T, int64_t K, const int8_t *Wq,
                                     const float *Wscale, const void *W16, int64_t N,
                                     float tau, void *Y, void *stream);

/* Static, human-readable name of a status code. */
const char *bnb_status_string(bnb_status_t s);

/*
 * Number of kernel launches this library has enqueued in this process
 * (memsets included), for accounting in benchmarks.
 */
uint64_t bnb_launch_count(void);

/*
 * Which kernel path bnb_int8_linear takes for a shape on the current device:
 * 1 = decode (T <= 16, K <= 4096 and N within what the decode kernels'
 * resident CTAs hold at up to 40 output channels each in at most three
 * launches: at K = 4096 on B300, 13860 for T > 8 and 17760 for T <= 8), 2 =
 * tensor-core GEMM (tcgen05; every other shape, decode-sized T included), 3 =
 * warp-level mma GEMM (only through bnb_int8_linear_opts with
 * BNB_OPT_LEGACY_MMA).
 */
int bnb_int8_linear_path(int64_t T, int64_t N, int64_t K);

/*
 * For a shape that takes the decode path (bnb_int8_linear_path == 1): the
 * form of the decode kernel bnb_int8_linear launches on the current device,
 * as a cluster size: 16, 8 or 4 (CTAs in thread-block clusters sharing one
 * activation pass) or 1 (no clusters: every CTA runs the whole activation
 * pass; by default T <= 5, and T <= 6 at K > 2048).  0 for any other shape.
 * For benchmarks and tests.
 */
int bnb_int8_decode_cluster(int64_t T, int64_t N, int64_t K);

/*
 * Per-call options for benchmarks and tests: bnb_int8_linear_opts is
 * bnb_int8_linear_debug_ex with a set of flags that change only that call.
 * The library keeps no switch of its own, so no option can change another
 * caller's results.
 *   BNB_OPT_MAIN_ONLY   enqueue only the main kernel of the path (the decode
 *                       kernel, or the GEMM on the activation-pass results
 *                       that the previous full call on the same workspace
 *                       left there).  Y is correct only if that call had the
 *                       same X and tau; the decode kernel recomputes its
 *                       activation pass and is unaffected.  For timing the
 *                       dominant kernel alone.
 *   BNB_OPT_ACT_ONLY    T > 16 path: enqueue only the activation pass (the
 *                       workspace clear, the column scan and the row pass);
 *                       Y is not written.
 *   BNB_OPT_NO_PDL      launch without programmatic dependent launch, so the
 *                       call's kernels start only after the stream's previous
 *                       work has completed.
 *   BNB_OPT_LEGACY_MMA  T > 16 path: the warp-level mma.sync GEMM (sm_80-style
 *                       tensor path, for comparison) instead of tcgen05.
 *   BNB_OPT_SINGLE_CTA  T > 32 on the tcgen05 GEMM: each 128 x 256 tile on
 *                       one CTA (cta_group::1) instead of 256 x 256 tiles on
 *                       CTA pairs (cta_group::2), for comparison.
 *   BNB_OPT_GEMM        T <= 16: the activation pass and the GEMM (path 2, or
 *                       3 with BNB_OPT_LEGACY_MMA) even where the decode
 *                       kernel holds the call, for comparison and tests.
 *   BNB_OPT_CLUSTER(c)  decode path: thread-block clusters of c CTAs (c = 4,
 *                       8 or 16) sharing one activation pass, or (c = 1, for
 *                       T <= 8) no clusters, every CTA running the whole
 *                       activation pass itself, instead of the form the
 *                       library picks, when that form holds the call in one
 *                       launch.
 *   BNB_OPT_FORCE_TIMEOUT  one thread of the call's main kernel waits, with a
 *                       limit of about 0.1 ms, on an mbarrier that nothing
 *                       completes, and then takes the kernel's timeout path
 *                       (BNB_ERR_TIMEOUT in the status word, Y unspecified).
 *                       Every other wait keeps its normal limit, and every copy
 *                       in flight lands before the kernel exits.  For testing
 *                       the timeout path; the next call on the workspace runs
 *                       normally.
 * Errors as for bnb_int8_linear_debug_ex, plus BNB_ERR_INVALID_ARG for an
 * unknown flag or cluster size.
 */
#define BNB_OPT_MAIN_ONLY 0x1u
#define BNB_OPT_ACT_ONLY 0x2u
#define BNB_OPT_NO_PDL 0x4u
#define BNB_OPT_LEGACY_MMA 0x8u
#define BNB_OPT_FORCE_TIMEOUT 0x10u
#define BNB_OPT_SINGLE_CTA 0x20u
#define BNB_OPT_GEMM 0x40u
#define BNB_OPT_CLUSTER(c) ((uint32_t)(c) << 8)
bnb_status_t bnb_int8_linear_opts(const void *X, int64_t T, int64_t K, const int8_t *Wq,
                                  const float *Wscale, const void *W16, const void *bias,
                                  int64_t N, float tau, int dtype, void *Y, void *workspace,
                                  size_t workspace_bytes, void *stream, int8_t *Xq,
                                  float *Xscale, int32_t *outlier_idx, int32_t *n_outliers,
                                  int32_t *acc, uint32_t opts);

#ifdef __cplusplus
}
#endif

#endif /* BNB_INT8_H */
