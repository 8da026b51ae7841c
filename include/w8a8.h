/*
 * w8a8.h -- C ABI of the GB300 (sm_103a) W8A8 INT8 Linear library.
 *
 * The method is the W8A8 Linear of "TurboDiffusion Integration Notes"
 * (TurboT2AV docs/acceleration.md):
 *   - section "Reused Components", bullet "W8A8 Linear": selected weights are
 *     quantized to INT8 once, at model initialization, and activations are
 *     quantized dynamically before every transformer Linear;
 *   - section "Differences From TurboDiffusion", row "W8A8 kernel" and the
 *     paragraph under that table: the post-scale kernel keeps the integer
 *     accumulation continuous across K and applies the activation and weight
 *     scales in the epilogue; TurboDiffusion's original kernel is
 *     blockwise-scaled.
 * The pages give no formulas.  This library computes:
 *   quantizer   s = absmax(group) / 127 (IEEE fp32 division),
 *               q = clamp(round_half_even(x / s), -127, 127) with x / s an
 *               IEEE fp32 division; a group whose absmax is 0 gets s = 0 and
 *               q = 0 everywhere.
 *   post-scale  acc[m,n] = sum_k Xq[m,k] * Wq[n,k] (exact int32),
 *               Y = bf16_rne(((float(acc) * sx[m]) * sw[n]) + bias[n]),
 *               every fp32 operation rounded on its own (no fused multiply-add),
 *               the bias add skipped when bias is NULL.
 *   blockwise   for each 128-wide K block kb, ascending, from acc = 0.0f:
 *               P = sum over the block of Xq * Wq (exact int32),
 *               acc = acc + ((float(P) * sx[m,kb]) * sw[n/128,kb]);
 *               Y = bf16_rne(acc + bias[n]) (add skipped when bias is NULL).
 *
 * Conventions for every entry point:
 *   - All matrices are row-major and dense (row stride = number of columns).
 *     X is [M,K] (tokens x input features), W is [N,K] (nn.Linear layout,
 *     Y = X * W^T), Y is [M,N].  bf16 arrays are passed as void pointers to
 *     IEEE bfloat16 values.
 *   - Every array pointer is a DEVICE pointer on the current CUDA device,
 *     16-byte aligned.  The caller owns all memory: the library allocates
 *     nothing and keeps no state between calls except cached device
 *     attributes and driver entry points.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream) and the call returns without synchronizing.
 *   - Argument checks are synchronous and happen before anything is
 *     enqueued: on any error nothing is launched and no output is touched.
 *   - M, N >= 0 (0 returns W8A8_OK and launches nothing).  K > 0, K % 16 == 0
 *     and K <= 131072 (so |acc| <= 127*127*K stays inside int32); the
 *     blockwise entry points also need K % 128 == 0.
 *   - Requires a device of compute capability 10.3 (GB300, sm_103a);
 *     otherwise W8A8_ERR_UNSUPPORTED_DEVICE.
 *   - Launch failures return W8A8_ERR_CUDA.  Faults found while a kernel
 *     runs (a bounded internal wait that ran out) are not returned by the
 *     call that enqueued it; read them with w8a8_get_device_error().
 */
#ifndef W8A8_GB300_H
#define W8A8_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define W8A8_API __attribute__((visibility("default")))
#else
#define W8A8_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    W8A8_OK = 0,
    W8A8_ERR_INVALID_ARG = 1,        /* NULL pointer, bad enum, negative size  */
    W8A8_ERR_ALIGNMENT = 2,          /* a pointer is not 16-byte aligned       */
    W8A8_ERR_SHAPE = 3,              /* K not a multiple of 16 (128), too large */
    W8A8_ERR_UNSUPPORTED_DEVICE = 4, /* current device is not sm_103           */
    W8A8_ERR_CUDA = 5,               /* a CUDA runtime / driver call failed    */
    W8A8_ERR_TIMEOUT = 6,            /* a device-side bounded wait ran out     */
    W8A8_ERR_WORKSPACE = 7           /* workspace missing or too small         */
} w8a8_status;

typedef enum {
    /* activations: one scale per token (row of X), sx[M];
     * weights: one scale per output channel (row of W), sw[N]. */
    W8A8_SCALE_PER_ROW = 0,
    /* activations: one scale per 1x128 block of a row, sx[M][K/128];
     * weights: one scale per 128x128 block, sw[ceil(N/128)][K/128]
     * (a last, partial row block uses the absmax over the rows it has). */
    W8A8_SCALE_BLOCK = 1
} w8a8_scale_mode;

/* Human-readable name of a status code (static string, never NULL). */
W8A8_API const char* w8a8_status_string(w8a8_status status);

/* One-line description of the last W8A8_ERR_CUDA returned on this host
 * thread (the CUDA call and its error string); "" if none.  The string is
 * owned by the library and valid until the next call on this thread. */
W8A8_API const char* w8a8_last_error_detail(void);

/*
 * Weight quantization, done once ("Reused Components", W8A8 Linear: weights
 * quantized to INT8 at model initialization).
 *   W   [N,K] bf16 in.
 *   Wq  [N,K] int8 out.
 *   sw  out: [N] (PER_ROW) or [ceil(N/128)][K/128] (BLOCK), fp32.
 */
W8A8_API w8a8_status w8a8_quantize_weight(const void* W, int64_t N, int64_t K, w8a8_scale_mode mode, int8_t* Wq,
                                 float* sw, void* stream);

/*
 * Dynamic activation quantization, done before every Linear ("Reused
 * Components", W8A8 Linear: activations dynamically quantized).
 *   X   [M,K] bf16 in.
 *   Xq  [M,K] int8 out.
 *   sx  out: [M] (PER_ROW, per token) or [M][K/128] (BLOCK), fp32.
 */
W8A8_API w8a8_status w8a8_quantize_act(const void* X, int64_t M, int64_t K, w8a8_scale_mode mode, int8_t* Xq,
                              float* sx, void* stream);

/*
 * Bytes of device workspace the GEMM entry points need for this shape.  The
 * tensor-core path runs the exact integer product on the bf16 tensor pipe
 * (GB300 has no 8-bit integer tcgen05 MMA); the workspace holds the bf16
 * images of Xq and Wq (every int8 value is exact in bf16) and, for few-token
 * post-scale shapes (M <= 256 with few 256-row weight tiles), the int32
 * partial sums of the K splits.  The same size serves both scale modes.
 * The post-scale entry points (w8a8_gemm_postscale, _s32, _noalloc) need less
 * for few tokens and accept it: with M <= 4 and M * K <= 131072 the GEMM is a
 * GEMV on the CUDA cores that needs no workspace; otherwise, with M <= 288,
 * it streams the int8 weight codes itself and needs the fp16 image of Xq
 * (M * K * 2 bytes, rounded up to 256) and, when N <= 76 * 128 and K > 384
 * (shapes whose K it may split), int32 sums (M * N * 4 bytes) and counters
 * (32 bytes per 128 rows of N), each rounded up to 256.
 */
W8A8_API size_t w8a8_gemm_workspace_size(int64_t M, int64_t N, int64_t K);

/*
 * Post-scale INT8 GEMM ("Differences From TurboDiffusion": the post-scale
 * kernel keeps the integer accumulation continuous across K and applies the
 * activation and weight scales in the epilogue).
 *   Xq [M,K] int8, sx [M] fp32 (per token), Wq [N,K] int8, sw [N] fp32
 *   (per output channel), bias [N] bf16 or NULL, Y [M,N] bf16 out.
 *   workspace: device buffer of at least w8a8_gemm_workspace_size(M,N,K)
 *   bytes, 256-byte aligned, owned by the caller, not read after the call's
 *   work completes on `stream`.  Few tokens need less (see
 *   w8a8_gemm_workspace_size): nothing with M <= 4 and M * K <= 131072
 *   (workspace may be NULL and workspace_bytes 0), the fp16 image of Xq plus,
 *   for shapes whose K may be split, int32 sums and counters with M <= 288;
 *   this also holds for w8a8_gemm_postscale_s32.
 */
W8A8_API w8a8_status w8a8_gemm_postscale(const int8_t* Xq, const float* sx, const int8_t* Wq, const float* sw,
                                const void* bias, void* Y, int64_t M, int64_t N, int64_t K, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * Blockwise-scaled INT8 GEMM ("Differences From TurboDiffusion": TurboDiffusion's
 * original W8A8 kernel is blockwise-scaled).  K % 128 == 0.
 *   Xq [M,K] int8, sx [M][K/128] fp32, Wq [N,K] int8,
 *   sw [ceil(N/128)][K/128] fp32, bias [N] bf16 or NULL, Y [M,N] bf16 out,
 *   workspace as for w8a8_gemm_postscale.
 */
W8A8_API w8a8_status w8a8_gemm_blockwise(const int8_t* Xq, const float* sx, const int8_t* Wq, const float* sw,
                                const void* bias, void* Y, int64_t M, int64_t N, int64_t K, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * Exact bf16 image of INT8 weight codes: Wimg[n,k] = (bf16) Wq[n,k], every
 * value in [-127, 127] exact.  The tensor-core GEMM consumes this image (GB300
 * has no 8-bit integer tcgen05 MMA), so packing it once, next to the weight
 * quantization at model initialization ("Reused Components", W8A8 Linear),
 * takes the per-call expansion out of the fused Linear below.  It occupies the
 * same 2 bytes per weight as the bf16 weight copy the pages keep.
 *   Wq [N,K] int8 in, Wimg [N,K] bf16 out.  K % 16 == 0.
 */
W8A8_API w8a8_status w8a8_pack_weight(const int8_t* Wq, int64_t N, int64_t K, void* Wimg, void* stream);

/* Device workspace bytes of the fused Linear entry points: the bf16 image of
 * the quantized activations (M * K * 2 bytes, rounded up to 256) plus, for
 * few-token post-scale shapes, the int32 partial sums of the K splits. */
W8A8_API size_t w8a8_linear_workspace_size(int64_t M, int64_t N, int64_t K);

/*
 * Fused W8A8 Linear, post-scale: dynamic per-token quantization of X ("Reused
 * Components": activations quantized before each Linear) followed by the
 * post-scale GEMM ("Differences From TurboDiffusion"), against a packed
 * weight image.  Results are identical to w8a8_quantize_act (PER_ROW) +
 * w8a8_gemm_postscale on the same inputs.
 *   X [M,K] bf16, Wimg [N,K] bf16 image from w8a8_pack_weight, sw [N] fp32,
 *   bias [N] bf16 or NULL, Y [M,N] bf16 out, sx [M] fp32 out (the per-token
 *   scales), Xq [M,K] int8 out or NULL (codes are written only if given),
 *   workspace of w8a8_linear_workspace_size(M,N,K) bytes, 256-byte aligned.
 */
W8A8_API w8a8_status w8a8_linear_postscale(const void* X, const void* Wimg, const float* sw, const void* bias,
                                           void* Y, int64_t M, int64_t N, int64_t K, float* sx, int8_t* Xq,
                                           void* workspace, size_t workspace_bytes, void* stream);

/* Device workspace bytes of w8a8_linear_postscale_codes: 0 when M <= 2 and
 * M * K <= 131072 (one kernel, no workspace); otherwise room for the int8
 * codes of X (M * K bytes, rounded up to 256; unused when the caller passes
 * Xq) plus what w8a8_gemm_postscale needs for the shape (nothing for the
 * GEMV, M <= 4; the int8 path's scratch with M <= 288; else
 * w8a8_gemm_workspace_size(M,N,K)). */
W8A8_API size_t w8a8_linear_codes_workspace_size(int64_t M, int64_t N, int64_t K);

/*
 * Fused W8A8 Linear, post-scale, against the int8 weight codes themselves
 * (no bf16 image): per-token quantization of X, then the post-scale GEMM of
 * w8a8_gemm_postscale, which reads each weight code once.  Meant for few
 * tokens (decoding): with M <= 2 and M * K <= 131072 it is one kernel, a
 * GEMV on the CUDA cores in which every CTA quantizes X into its shared
 * memory while its first weight loads are in flight; up to 4 tokens the
 * quantization kernel and the GEMV; up to 288 tokens the quantization kernel
 * and the int8-operand tensor-core GEMM.  Any M is accepted; for many
 * tokens w8a8_linear_postscale on a packed image is faster.
 * Results are identical to w8a8_quantize_act (PER_ROW) + w8a8_gemm_postscale
 * on the same inputs.
 *   X [M,K] bf16, Wq [N,K] int8 (w8a8_quantize_weight, PER_ROW), sw [N] fp32,
 *   bias [N] bf16 or NULL, Y [M,N] bf16 out, sx [M] fp32 out, Xq [M,K] int8
 *   out or NULL, workspace of w8a8_linear_codes_workspace_size(M,N,K) bytes,
 *   256-byte aligned (may be NULL when that size is 0).
 */
W8A8_API w8a8_status w8a8_linear_postscale_codes(const void* X, const int8_t* Wq, const float* sw, const void* bias,
                                                 void* Y, int64_t M, int64_t N, int64_t K, float* sx, int8_t* Xq,
                                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Fused W8A8 Linear, blockwise: 1x128 activation quantization followed by the
 * blockwise GEMM, against a packed weight image.  K % 128 == 0.  sx is
 * [M][K/128] out, sw is [ceil(N/128)][K/128]; other arguments as above.
 */
W8A8_API w8a8_status w8a8_linear_blockwise(const void* X, const void* Wimg, const float* sw, const void* bias,
                                           void* Y, int64_t M, int64_t N, int64_t K, float* sx, int8_t* Xq,
                                           void* workspace, size_t workspace_bytes, void* stream);

/*
 * Fused FFN up-projection as the blockwise down-projection consumes it.  The
 * pages tune the post-scale kernel for "LTX FFN shapes" ("Differences From
 * TurboDiffusion") and name no activation; the FFN's activation is taken to
 * be GELU in its erf form.  Computes, with the post-scale Linear of
 * w8a8_linear_postscale:
 *   y = bf16(((acc * sx) * sw) + bias),  g = bf16(gelu(y)),
 *   sg[m][j] = absmax(|g[m, 128j .. 128j+127]|) / 127,
 *   codes = clamp(rne(g / sg), -127, 127) per 1x128 block,
 * and writes the exact bf16 image of the codes, which w8a8_gemm_blockwise_images
 * takes as its activation operand (1x128 activation scales sg).  gelu(x) =
 * x * Phi(x), Phi(x) = erfc(-x / sqrt 2) / 2 = (1 + erf(x / sqrt 2)) / 2, with
 * erfc from the Chebyshev-fitted formula of Numerical Recipes in C (2nd ed.,
 * section 6.2, fractional error < 1.2e-7) evaluated in binary32; g is within
 * 1 bf16 ulp of the bf16 of the exact GELU for every bf16 input
 * (w8a8_gelu_bf16 exports the same function for testing).
 *   X [M,K] bf16, Wimg [N,K] bf16 image (w8a8_pack_weight), sw [N] fp32,
 *   bias [N] bf16 or NULL, Gimg [M,N] bf16 out, sg [M][N/128] fp32 out,
 *   sx [M] fp32 out, Xq [M,K] int8 out or NULL, workspace of
 *   w8a8_linear_workspace_size(M,N,K) bytes, 256-byte aligned.
 *   N % 128 == 0 (else W8A8_ERR_SHAPE).
 */
W8A8_API w8a8_status w8a8_linear_postscale_gelu_quant(const void* X, const void* Wimg, const float* sw,
                                                      const void* bias, void* Gimg, float* sg, int64_t M, int64_t N,
                                                      int64_t K, float* sx, int8_t* Xq, void* workspace,
                                                      size_t workspace_bytes, void* stream);

/*
 * Blockwise GEMM on operand images: Ximg [M,K] and Wimg [N,K] are exact bf16
 * images of int8 codes (from w8a8_linear_postscale_gelu_quant and
 * w8a8_pack_weight), sx [M][K/128], sw [ceil(N/128)][K/128], bias [N] bf16 or
 * NULL, Y [M,N] bf16 out.  Same arithmetic as w8a8_gemm_blockwise.  K % 128
 * == 0.  Needs no workspace.
 */
W8A8_API w8a8_status w8a8_gemm_blockwise_images(const void* Ximg, const float* sx, const void* Wimg, const float* sw,
                                                const void* bias, void* Y, int64_t M, int64_t N, int64_t K,
                                                void* stream);

/* Normalization of the fused normalization + quantization entry point. */
typedef enum {
    W8A8_NORM_RMS = 0,   /* y = (x * r) * gamma,             r = 1 / sqrt(S(x*x)/K + eps)  */
    W8A8_NORM_LAYER = 1  /* y = ((d * r) * gamma) + beta,    d = x - S(x)/K, r = 1 / sqrt(S(d*d)/K + eps) */
} w8a8_norm_kind;

/*
 * RMSNorm or LayerNorm fused with per-token activation quantization
 * ("TurboDiffusion Integration Notes", section "Reused Components": FastNorm
 * replaces RMSNorm/LayerNorm with fused implementations; W8A8 and FastNorm
 * form one combined stage in section "End-to-End Result").  One read of X:
 * y = bf16(normalized row, formulas above; a NULL gamma or beta skips that
 * operation), then sx[m] = absmax(y[m,:]) / 127 and q = clamp(rne(y / sx),
 * -127, 127).  S() is summed in a fixed order independent of the launch:
 * chunks of 8 consecutive elements left to right, then the chunk sums
 * (zero-padded to a power of two) pairwise level by level.  Every operation
 * is IEEE binary32, rounded on its own.
 *   X [M,K] bf16, gamma / beta [K] bf16 or NULL (beta only for LAYER), eps >= 0,
 *   Y [M,K] bf16 out or NULL (the normalized row), Xq [M,K] int8 out or NULL,
 *   Ximg [M,K] bf16 out or NULL (exact image of Xq, the GEMM's operand),
 *   sx [M] fp32 out.  K % 8 == 0 and K <= 16384 (else W8A8_ERR_SHAPE).
 */
W8A8_API w8a8_status w8a8_norm_quant(const void* X, const void* gamma, const void* beta, float eps,
                                     w8a8_norm_kind kind, int64_t M, int64_t K, void* Y, int8_t* Xq, void* Ximg,
                                     float* sx, void* stream);

/* Device workspace bytes of w8a8_gemm_postscale_images (the int32 partial
 * sums of the K splits of few-token shapes; 0 when the shape is not split). */
W8A8_API size_t w8a8_splitk_workspace_size(int64_t M, int64_t N, int64_t K);

/*
 * Post-scale GEMM on operand images: Ximg [M,K] and Wimg [N,K] are exact
 * bf16 images of int8 codes (from w8a8_norm_quant and w8a8_pack_weight), sx
 * [M], sw [N], bias [N] bf16 or NULL, Y [M,N] bf16 out.  Same arithmetic as
 * w8a8_gemm_postscale.  workspace: w8a8_splitk_workspace_size(M,N,K) bytes,
 * 256-byte aligned (may be NULL when that size is 0).
 */
W8A8_API w8a8_status w8a8_gemm_postscale_images(const void* Ximg, const float* sx, const void* Wimg, const float* sw,
                                                const void* bias, void* Y, int64_t M, int64_t N, int64_t K,
                                                void* workspace, size_t workspace_bytes, void* stream);

/*
 * Allocation-free variant of w8a8_gemm_postscale (the pages have no
 * counterpart: this is a library convenience).  Same arguments, results and
 * checks, minus the workspace: the scratch lives in a fixed 64 MiB device
 * array inside the library, so the shape's scratch need must fit in it, else
 * W8A8_ERR_WORKSPACE and nothing is launched.  The need is that of
 * w8a8_gemm_postscale: nothing with M <= 4 and M * K <= 131072 (the
 * few-token GEMV), the fp16 image of Xq plus any K-split sums with M <= 288
 * (a few MB: for example M = 77, N = 13824, K = 5120 needs 788 KB), else
 * w8a8_gemm_workspace_size(M,N,K) (for example M = N = K = 4096 fits
 * exactly).
 *
 * For callers that cannot allocate device memory at the call site, for
 * example code running inside a host callback or a real-time loop where
 * cudaMalloc's implicit synchronization is not allowed, or a plugin whose
 * host framework owns the device allocator and offers it no hook.
 *
 * The array is created when the library is loaded on a device and held by
 * every device that loads the library until the process exits.  The first
 * call on each device looks up the array's device address (once, with that
 * device current); make that first call before any stream capture.  Every
 * call shares the one array and leaves its contents behind (nothing in it
 * needs to start at zero): calls whose work overlaps on the GPU, on
 * different streams or threads, race on it and must be serialized by the
 * caller.  Calls no cudaMalloc, cudaFree or allocating library routine.
 */
W8A8_API w8a8_status w8a8_gemm_postscale_noalloc(const int8_t* Xq, const float* sx, const int8_t* Wq,
                                                 const float* sw, const void* bias, void* Y, int64_t M, int64_t N,
                                                 int64_t K, void* stream);

/*
 * Test and debug exports of the same mainloops, stopping before the bf16
 * epilogue.
 *   w8a8_gemm_postscale_s32: acc [M,N] int32 = sum_k Xq[m,k] * Wq[n,k].
 *   w8a8_gemm_blockwise_f32: acc [M,N] fp32, the blockwise accumulator before
 *   the bias add and bf16 rounding.
 */
W8A8_API w8a8_status w8a8_gemm_postscale_s32(const int8_t* Xq, const int8_t* Wq, int32_t* acc, int64_t M, int64_t N,
                                    int64_t K, void* workspace, size_t workspace_bytes, void* stream);
W8A8_API w8a8_status w8a8_gemm_blockwise_f32(const int8_t* Xq, const float* sx, const int8_t* Wq, const float* sw,
                                    float* acc, int64_t M, int64_t N, int64_t K, void* workspace,
                                    size_t workspace_bytes, void* stream);

/*
 * Test export of the FFN up-projection's activation (not part of the
 * Linear): G[i] = bf16(gelu(Y[i])) for n bf16 values, computed by the same
 * device function as the epilogue of w8a8_linear_postscale_gelu_quant, so
 * that its values can be checked on every bf16 input.  Y and G are device
 * pointers, 16-byte aligned; n % 8 == 0 (else W8A8_ERR_SHAPE).  Asynchronous
 * on `stream`.
 */
W8A8_API w8a8_status w8a8_gelu_bf16(const void* Y, int64_t n, void* G, void* stream);

/*
 * Reads and clears the device-side error word of the current device.
 * Synchronizes the device.  *code receives 0 when no kernel has recorded a
 * fault, else the first recorded code (0x100 + n: internal bounded wait n ran
 * out).  Returns W8A8_ERR_TIMEOUT when a wait ran out, W8A8_OK otherwise (or
 * W8A8_ERR_CUDA if the readback itself failed).
 */
W8A8_API w8a8_status w8a8_get_device_error(int* code);

/*
 * Failure-detection check (not part of the Linear): launches one CTA whose
 * thread waits on an mbarrier that nothing arrives on.  The wait is bounded
 * like every wait in the library's kernels (2 s of device time); when it
 * runs out the kernel records a timeout in the device error word and returns
 * normally, so the context stays usable.  A following w8a8_get_device_error
 * reports W8A8_ERR_TIMEOUT with code 0x100 + 30.  Asynchronous on `stream`.
 */
W8A8_API w8a8_status w8a8_probe_wait_timeout(void* stream);

/*
 * Measurement hook (not part of the Linear): while set, every GEMM entry
 * point called from this host thread records `start` immediately before and
 * `end` immediately after its tensor-core kernel launch, on the call's
 * stream.  Both are cudaEvent_t handles created by the caller (with timing
 * enabled); pass NULL, NULL to stop.  This is the only per-thread state the
 * library keeps.  Returns W8A8_ERR_INVALID_ARG if exactly one is NULL.
 */
W8A8_API w8a8_status w8a8_set_gemm_timing_events(void* start, void* end);

/*
 * Measurement helper (not part of the Linear): runs a throughput kernel of
 * warp-level INT8 MMAs (mma.sync m16n8k32 s8 x s8 -> s32) on every SM and
 * returns the achieved tera-operations per second (2 ops per multiply-add)
 * in *tops.  Used as the measured dense INT8 roofline of this GPU.
 * Synchronizes `stream`.
 */
W8A8_API w8a8_status w8a8_measure_imma_peak(double* tops, void* stream);

/*
 * Measurement helper (not part of the Linear): moves the bytes of an
 * activation quantization -- reads n bf16 values from src, writes n bytes to
 * dst (the high byte of each value) -- as a plain grid-stride stream.  Timed
 * under the same conditions as w8a8_quantize_act on the same shape it gives
 * the memory floor of that quantization.  n % 8 == 0; both pointers 16-byte
 * aligned; asynchronous on `stream`.
 */
W8A8_API w8a8_status w8a8_stream_floor(const void* src, int64_t n, void* dst, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* W8A8_GB300_H */
