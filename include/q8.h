/*
 * q8.h -- C ABI of the GB300 W8A8 quantized linear layer.
 *
 * The layer is the datapath the pages describe as "dequantize after integer
 * accumulation": activations are quantized at run time, weights offline, the
 * dot products are exact integer arithmetic accumulated in INT32, and the
 * scales (and the zero-point correction) are applied once per output element
 * in the epilogue:
 *
 *   y[m][n] = (float)(acc[m][n] - z_a[m] * colsum[n]) * (s_a[m] * s_w[n]),
 *   acc[m][n] = sum_k qa[m][k] * qw[n][k],   colsum[n] = sum_k qw[n][k].
 *
 * ("100 Days of GPU, Day 98: Quantization and sparsity", sections "What a
 * scale actually promises" and "The program, and the gate that has to be per
 * column"; "Activation Quantization Architecture", section "The integer GEMM,
 * written out"; "Write Int8 Quantized Kernel", reasoning steps 1, 2 and 4.)
 *
 * Conventions for every entry point:
 *  - All array arguments are DEVICE pointers (memory the caller allocated on
 *    the current CUDA device) unless stated otherwise. The caller owns every
 *    buffer; the library keeps no pointer after a call returns and allocates
 *    no device memory (the fixed array behind q8_linear_host_static is part of
 *    the loaded library, not an allocation).
 *  - Matrices are row-major and dense. A is [M, K]; the weight is stored
 *    K-major as W[N, K] (row n holds output channel n), the (N, K) layout of
 *    "Write Int8 Quantized Kernel" (Common failure modes); y is [M, N].
 *  - Every array base must be 16-byte aligned and K must be a multiple of 16
 *    (rows are then 16-byte aligned for vector loads and TMA tiles).
 *  - Calls are asynchronous and ordered on `stream` (NULL = the legacy default
 *    stream). A returned Q8_OK means the work was enqueued; errors that
 *    happen on the device surface at the next synchronising call.
 *  - Arguments are validated on the host before anything is enqueued; a
 *    rejected call enqueues nothing and touches no memory.
 *  - Inputs must be finite: NaN and Inf are not checked and give unspecified
 *    codes (the pages do not define them).
 *  - M, N or K equal to 0 are valid empty problems.
 */
#ifndef Q8_H_
#define Q8_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared here so the header needs no CUDA include. */
typedef struct CUstream_st* q8_stream_t;

typedef enum q8_status {
    Q8_OK = 0,
    Q8_ERR_INVALID_ARG = 1,  /* null pointer, negative size, bad enum, misaligned base */
    Q8_ERR_UNSUPPORTED = 2,  /* K not a multiple of 16, or K beyond the INT32 range limit */
    Q8_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
    Q8_ERR_TIMEOUT = 4       /* a bounded device-side wait gave up (see q8_device_error) */
} q8_status;

/* One scale for the whole tensor, or one per row: per token for A (rows of
 * A), per output channel for W (rows of the K-major W[N, K]). Day 98, "What
 * a scale actually promises"; "Write Int8 Quantized Kernel", inputs to gather. */
typedef enum q8_granularity { Q8_PER_TENSOR = 0, Q8_PER_ROW = 1 } q8_granularity;

typedef enum q8_symmetry { Q8_SYMMETRIC = 0, Q8_ASYMMETRIC = 1 } q8_symmetry;

/* GEMM kernel choice for q8_gemm_dequant_ex / q8_gemm_s32_ex. */
typedef enum q8_gemm_kernel {
    Q8_GEMM_AUTO = 0,     /* pick by shape (what q8_gemm_dequant does) */
    Q8_GEMM_TCGEN05 = 1,  /* tcgen05 tensor-core kernel (fp32 TMEM chunks drained to INT32) */
    Q8_GEMM_MMA_S8 = 2,   /* warp-level mma.sync s8 kernel, 128x128 tiles */
    Q8_GEMM_SKINNY = 3,   /* warp-level mma.sync s8 kernel, 16x64 tiles */
    Q8_GEMM_DECODE = 4,   /* M <= 16: TMA weight stream, in-register int8->fp16, mma.sync f16 */
    Q8_GEMM_DECODE_TC = 5, /* M <= 16 on tcgen05: weights as the MMA M side, tokens as N = 16 */
    Q8_GEMM_TCGEN05_PAIR = 6 /* tcgen05 on CTA pairs (cta_group::2), 256 x 256 tiles */
} q8_gemm_kernel;

/*
 * Dynamic activation quantization (one call per forward pass).
 *
 * Symmetric: s = max(amax, 1e-8) / 127 with amax = max|a| over the row (or
 * tensor), q = clamp(rint(a / s), -127, 127), z not used. ("Activation
 * Quantization Architecture", The quantizer itself and the Fusion pseudocode;
 * Day 98, What a scale actually promises.)
 * Asymmetric: lo = min(min a, 0), hi = max(max a, 0), s = max(hi - lo, 1e-8)
 * / 255, z = clamp(-128 - rint(lo / s), -128, 127), q = clamp(rint(a / s) + z,
 * -128, 127): the uint8 codes 0..255 of "Write Int8 Quantized Kernel" step 1
 * stored as int8 (code - 128), with z the code that dequantizes to zero (Day 98).
 * Divisions are IEEE fp32, rint is round-half-to-even.
 *
 * a   : fp32 [M, K], read only.
 * qa  : int8 [M, K], written.
 * s_a : fp32 [M] (Q8_PER_ROW) or [1] (Q8_PER_TENSOR), written.
 * z_a : int32 [M] or [1], written; must be NULL for Q8_SYMMETRIC and non-NULL
 *       for Q8_ASYMMETRIC.
 * Per-tensor granularity uses s_a[0] (and z_a[0]) as its reduction cell, so no
 * extra workspace is needed; their contents on entry are ignored.
 */
q8_status q8_quantize_act(const float* a, int64_t M, int64_t K, q8_granularity g,
                          q8_symmetry sym, int8_t* qa, float* s_a, int32_t* z_a,
                          q8_stream_t stream);

/*
 * Fused RMSNorm + per-token symmetric activation quantization, the step before
 * the GEMM when the layer input comes out of a normalisation ("Activation
 * Quantization Architecture", Fusion: the kernel pseudocode for the fused norm
 * and quantize step). Per row m of a:
 *   rms = sqrt(mean_k a[m,k]^2 + eps),  y[m,k] = a[m,k] / rms * gamma[k],
 *   then s_a[m] and qa[m,:] from y exactly as q8_quantize_act(Q8_PER_ROW,
 *   Q8_SYMMETRIC) would compute them from y.
 * Arithmetic: the sum of squares is the exact sum rounded once to fp32 (any
 * order of summation gives it, up to sums within ~2^-40 of an fp32 rounding
 * midpoint, where either neighbour is returned); then fp32 IEEE operations in
 * the order written: mean = sum / K, rms = sqrt(mean + eps), y = (a / rms) *
 * gamma. y itself is not stored: one pass reads a and writes the codes.
 *
 * a     : fp32 [M, K], read only, 16-byte aligned.
 * gamma : fp32 [K], read only, 16-byte aligned.
 * eps   : > 0 and finite.
 * qa    : int8 [M, K], written, 16-byte aligned.
 * s_a   : fp32 [M], written.
 * Errors: Q8_ERR_INVALID_ARG for null or misaligned pointers (M > 0), M < 0,
 * K <= 0 with M > 0, or eps not > 0; Q8_ERR_UNSUPPORTED for K % 16 != 0 or
 * K > 2^24 (K must convert to fp32 exactly for the mean).
 * M == 0 returns Q8_OK without touching the device.
 */
q8_status q8_rmsnorm_quantize_act(const float* a, const float* gamma, int64_t M, int64_t K, float eps,
                                  int8_t* qa, float* s_a, q8_stream_t stream);

/*
 * Offline int4 weight quantization for W4A8, per output channel: TileLang tutorial
 * ch. 27 (low-precision quantization), 2.4 int8 / int4 with qmax = 7:
 *   s_w[n] = max(absmax_n, 1e-8) / 7,  q = clamp(rint(w / s_w[n]), -8, 7),
 * packed two codes per byte along K, low nibble first: byte i of row n holds
 * (q[n][2i] & 0xF) | (q[n][2i+1] & 0xF) << 4 (the int4 GEMM example's packing;
 * decoders sign-extend each nibble).
 *
 * w    : fp32 W[N, K], read only, 16-byte aligned.
 * qw4  : uint8 [N, K / 2], written, 16-byte aligned.
 * s_w  : fp32 [N], written.
 * Errors: Q8_ERR_INVALID_ARG for null or misaligned pointers (N, K > 0) or N, K < 0;
 * Q8_ERR_UNSUPPORTED for K % 32 != 0 (whole 16-byte packed rows).
 */
q8_status q8_quantize_weight_int4(const float* w, int64_t N, int64_t K, uint8_t* qw4, float* s_w,
                                  q8_stream_t stream);

/* Column sums of int4 weights, colsum[n] = sum_k q[n][k] (for asymmetric
 * activations in W4A8): qw4 uint8 [N, K / 2] as written by q8_quantize_weight_int4. */
q8_status q8_colsum_int4(const uint8_t* qw4, int64_t N, int64_t K, int32_t* colsum,
                         q8_stream_t stream);

/*
 * Offline symmetric weight quantization, per output channel or per tensor,
 * with the symmetric rule above ("Activation Quantization Architecture", the
 * numpy reference quantize_per_channel; Day 98, one scale per column of B).
 *
 * w   : fp32 W[N, K] (K-major), read only.
 * qw  : int8 [N, K], written.
 * s_w : fp32 [N] (Q8_PER_ROW) or [1] (Q8_PER_TENSOR), written.
 */
q8_status q8_quantize_weight(const float* w, int64_t N, int64_t K, q8_granularity g,
                             int8_t* qw, float* s_w, q8_stream_t stream);

/*
 * Column sums of the quantized weights, colsum[n] = sum_k qw[n][k] (exact
 * int32; |colsum| <= 128 K). Computed once, offline, next to the weights; the
 * epilogue needs them only when A is asymmetric (Day 98, the paragraph after
 * the kernel listing).
 *
 * qw     : int8 [N, K], read only.
 * colsum : int32 [N], written.
 */
q8_status q8_colsum(const int8_t* qw, int64_t N, int64_t K, int32_t* colsum,
                    q8_stream_t stream);

/*
 * Integer GEMM with the fused dequantization epilogue:
 *   acc  = sum_k qa[m][k] * qw[n][k]                  (exact, INT32)
 *   corr = acc - z_a[m] * colsum[n]                   (INT32; 0 when z_a == NULL)
 *   y    = (float)corr * (s_a[m] * s_w[n])            (two fp32 roundings)
 * The multiply order is that of the Day 98 epilogue listing; the zero-point
 * correction is applied before the scales ("Write Int8 Quantized Kernel",
 * correctness requirements).
 *
 * qa, qw   : int8 [M, K], int8 [N, K]; any codes in [-128, 127] are accepted.
 * s_a      : fp32 [M] if ga == Q8_PER_ROW, else [1].
 * z_a      : NULL (symmetric A) or int32 [M] / [1] following ga.
 * s_w      : fp32 [N] if gw == Q8_PER_ROW, else [1].
 * colsum   : int32 [N]; required iff z_a != NULL (ignored otherwise).
 * y        : fp32 [M, N], written.
 * Limits   : K <= 131056 when z_a == NULL (128*128*K < 2^31) and K <= 65792
 *            otherwise (255*128*K < 2^31), so acc and corr never leave INT32;
 *            larger K returns Q8_ERR_UNSUPPORTED.
 */
q8_status q8_gemm_dequant(const int8_t* qa, const float* s_a, const int32_t* z_a,
                          q8_granularity ga, const int8_t* qw, const float* s_w,
                          q8_granularity gw, const int32_t* colsum, int64_t M, int64_t N,
                          int64_t K, float* y, q8_stream_t stream);

/*
 * The layer on device buffers in one call: q8_quantize_act(a, ga, sym) into the
 * caller's qa / s_a / z_a, then q8_gemm_dequant (kernel by shape) into y. The
 * results are those of the two calls made one after the other ("Activation
 * Quantization Architecture", the quantizer itself and the integer GEMM written
 * out; Day 98's epilogue).
 *
 * Both halves are validated before either is enqueued; arguments, limits and
 * errors are those of q8_quantize_act and q8_gemm_dequant (qa, s_a, z_a are
 * outputs of the first and inputs of the second). For M <= 16 the decode kernel
 * streams the weights while the quantizer is still running (the two are launched
 * back to back on `stream`); it does so only when qa, s_a and z_a share no byte
 * with qw, s_w or colsum, and otherwise starts after the quantizer completes.
 * A standalone q8_gemm_dequant always waits for the kernel before it on the
 * stream before reading any operand.
 */
q8_status q8_linear(const float* a, int64_t M, int64_t K, q8_granularity ga, q8_symmetry sym,
                    int8_t* qa, float* s_a, int32_t* z_a, const int8_t* qw, const float* s_w,
                    q8_granularity gw, const int32_t* colsum, int64_t N, float* y,
                    q8_stream_t stream);

/*
 * q8_gemm_dequant with a caller-owned device workspace, same results bit for
 * bit. For shapes that run on the CTA-pair tensor-core kernel (prefill: more than
 * 16 tokens and a layer above the small-layer cut), the call first writes the
 * activation codes once as the fp16 numbers of equal value into the workspace (a
 * stream through HBM: M K bytes read, 2 M K written) and the kernel then loads
 * them by TMA straight into its operand stages. Without the workspace the kernel
 * converts every activation code in shared memory once per 256-column output tile
 * it enters (N / 256 times), and that shared-memory traffic bounds it. The
 * stored activation format stays int8; the fp16 copy is scratch.
 *
 * q8_gemm_workspace(M, N, K): the bytes this shape can use (2 M K, or 0 when the
 * shape takes another kernel). workspace: NULL or smaller than that runs
 * q8_gemm_dequant; otherwise 16-byte aligned device memory, overwritten; the caller
 * owns it and may reuse it once the call's work on `stream` has completed; it must
 * not overlap any operand or y.
 * Other arguments, limits and errors as q8_gemm_dequant; a misaligned workspace
 * returns Q8_ERR_INVALID_ARG.
 */
size_t q8_gemm_workspace(int64_t M, int64_t N, int64_t K);
q8_status q8_gemm_dequant_ws(const int8_t* qa, const float* s_a, const int32_t* z_a,
                             q8_granularity ga, const int8_t* qw, const float* s_w,
                             q8_granularity gw, const int32_t* colsum, int64_t M, int64_t N,
                             int64_t K, float* y, void* workspace, size_t workspace_bytes,
                             q8_stream_t stream);

/* q8_gemm_dequant with an explicit kernel choice. A kernel that cannot run
 * the given shape returns Q8_ERR_UNSUPPORTED (Q8_GEMM_AUTO never does). */
q8_status q8_gemm_dequant_ex(const int8_t* qa, const float* s_a, const int32_t* z_a,
                             q8_granularity ga, const int8_t* qw, const float* s_w,
                             q8_granularity gw, const int32_t* colsum, int64_t M, int64_t N,
                             int64_t K, float* y, q8_gemm_kernel kernel, q8_stream_t stream);

/* Output type of q8_gemm_epilogue_ex. */
typedef enum q8_out_type {
    Q8_OUT_F32 = 0,   /* fp32 y */
    Q8_OUT_BF16 = 1,  /* bf16 y (uint16 bit patterns), round to nearest even */
    Q8_OUT_I8 = 2     /* int8 codes clamp(rint(y / out_scale), -127, 127) for the next GEMM */
} q8_out_type;

/*
 * q8_gemm_dequant_ex with the epilogue variants of "Activation Quantization
 * Architecture" (Fusion: after the int32 accumulation the epilogue multiplies
 * by the per-token and per-channel scales, adds the bias and writes bf16; some
 * kernels quantize the output for the next GEMM directly):
 *   y[m][n] = fl((float)corr * (s_a * s_w)) + bias[n]   (one fp32 add; no bias: + 0 skipped)
 * then written as out_type. The output quantization uses a static per-tensor
 * scale (out_scale, e.g. from calibration): a per-token output scale would need
 * each row's maximum over all N before any code could be written.
 *
 * bias      : fp32 [N] or NULL, 4-byte aligned.
 * out       : fp32 / bf16 / int8 [M, N] by out_type, written, 16-byte aligned.
 * out_scale : Q8_OUT_I8 only: > 0 and finite.
 * Other arguments, limits and errors as q8_gemm_dequant_ex. With K == 0 the
 * output is bias (or zeros) in the requested type.
 */
q8_status q8_gemm_epilogue_ex(const int8_t* qa, const float* s_a, const int32_t* z_a,
                              q8_granularity ga, const int8_t* qw, const float* s_w,
                              q8_granularity gw, const int32_t* colsum, const float* bias,
                              int64_t M, int64_t N, int64_t K, q8_out_type out_type, void* out,
                              float out_scale, q8_gemm_kernel kernel, q8_stream_t stream);

/*
 * W4A8: the quantized linear layer with int4 weights (TileLang tutorial ch. 27,
 * low-precision quantization: 2.4 int8 / int4 and the int4 / dequantize GEMM
 * examples): acc[m][n] = sum_k qa[m][k] * q4[n][k] (exact int32; |acc| <= K *
 * 128 * 8), then the epilogue of q8_gemm_epilogue_ex with per-channel s_w.
 *
 * qw4    : uint8 [N, K / 2], two sign-extended int4 codes per byte, low nibble
 *          first (as written by q8_quantize_weight_int4), 16-byte aligned.
 * s_w    : fp32 [N] (per output channel).
 * colsum : int32 [N] from q8_colsum_int4, required iff z_a is given.
 * kernel : Q8_GEMM_AUTO (decode kernel for M <= 16, else the CTA-pair kernel),
 *          Q8_GEMM_DECODE or Q8_GEMM_TCGEN05_PAIR; other kernels return
 *          Q8_ERR_UNSUPPORTED.
 * Other arguments and errors as q8_gemm_epilogue_ex; K % 32 != 0 returns
 * Q8_ERR_UNSUPPORTED.
 */
q8_status q8_gemm_w4a8_ex(const int8_t* qa, const float* s_a, const int32_t* z_a, q8_granularity ga,
                          const uint8_t* qw4, const float* s_w, const int32_t* colsum,
                          const float* bias, int64_t M, int64_t N, int64_t K, q8_out_type out_type,
                          void* out, float out_scale, q8_gemm_kernel kernel, q8_stream_t stream);

/*
 * q8_gemm_w4a8_ex (kernel Q8_GEMM_AUTO) with a caller workspace: where the call
 * runs the CTA-pair kernel (M > 16, or a shape the decode kernel does not take),
 * the activation codes are first written once into the workspace as fp16 values,
 * each group of four K in the order 0, 2, 1, 3 in which the kernel converts the
 * packed weight codes, and the kernel loads them by TMA straight into its operand
 * stages; its converter warps then handle the weights only. The result is that of
 * q8_gemm_w4a8_ex, bit for bit (the same exact INT32 sums).
 *
 * workspace : NULL, or 16-byte aligned device memory of workspace_bytes bytes; used
 *             iff workspace_bytes >= 2 M K and the CTA-pair kernel runs, then
 *             overwritten. The caller owns it, may reuse it once the call's work on
 *             `stream` has completed, and must not let it overlap any operand or out.
 * Other arguments and errors as q8_gemm_w4a8_ex; a misaligned workspace returns
 * Q8_ERR_INVALID_ARG.
 */
q8_status q8_gemm_w4a8_ws(const int8_t* qa, const float* s_a, const int32_t* z_a, q8_granularity ga,
                          const uint8_t* qw4, const float* s_w, const int32_t* colsum,
                          const float* bias, int64_t M, int64_t N, int64_t K, q8_out_type out_type,
                          void* out, float out_scale, void* workspace, size_t workspace_bytes,
                          q8_stream_t stream);

/* Raw INT32 accumulators of the W4A8 product (diagnostic export, for bit-exact checks). */
q8_status q8_gemm_w4a8_s32_ex(const int8_t* qa, const uint8_t* qw4, int64_t M, int64_t N, int64_t K,
                              int32_t* acc, q8_gemm_kernel kernel, q8_stream_t stream);

/*
 * Block-scaled (MX-style) int8 weights (TileLang tutorial ch. 27, low-precision
 * quantization, 2.3 MX / block-scaled: block granularity + E8M0).
 *
 * Every `group` consecutive K elements of a weight row share one scale
 * s = 2^(e - 127), stored as the E8M0 byte e: x = amax / 127 (fp32 division)
 * rounded up to a power of two (the exponent field of x, plus one when its
 * mantissa is not zero), e clamped to [103, 136] (s = 2^-24 .. 2^9: every
 * dequantized q * s is then an exact fp16 value; weights with |w| > 127 * 2^9
 * saturate at +-127). Codes q = clamp(rint(w / s), -127, 127).
 *
 * w     : fp32 [N, K] row-major, 16-byte aligned, finite.
 * group : 32 (the native MX block) or 128; K % group != 0 -> Q8_ERR_UNSUPPORTED.
 * qw    : int8 [N, K], written, 16-byte aligned.
 * sf    : uint32 [ceil(K / group / 4), N], written, 4-byte aligned: four scale
 *         bytes per word, byte b (bits 8b .. 8b + 7) of word w holding group
 *         4w + b, words group-major (word w of row n at sf[w * N + n]); bytes
 *         past the last group are 0.
 * Errors: Q8_ERR_INVALID_ARG (negative sizes, group not 32 / 128, null or
 * misaligned pointers), Q8_ERR_CUDA.
 */
q8_status q8_quantize_weight_mx(const float* w, int64_t N, int64_t K, int group, int8_t* qw,
                                uint32_t* sf, q8_stream_t stream);

/*
 * The layer with block-scaled weights and symmetric int8 activations:
 *   T[m][n] = sum_k qa[m][k] * (qw[n][k] * s[n][k / group]),
 *   y[m][n] = fl(T[m][n] * s_a[m]) (+ bias[n]), then the output type.
 * The weights are dequantized to fp16 before the product (exact), T is summed
 * by the tensor core in fp32 over the whole K: not bit-reproducible against an
 * exactly rounded sum, its error bounded by the fp32 accumulation (the products
 * are exact); the same inputs give the same bits on every run.
 *
 * qa, s_a, ga : as q8_gemm_dequant_ex (symmetric activations only).
 * qw, sf      : from q8_quantize_weight_mx with the same group.
 * bias, out_type, out, out_scale : as q8_gemm_epilogue_ex.
 * kernel      : Q8_GEMM_AUTO (the decode kernel where it applies, else the pair
 *               kernel), Q8_GEMM_DECODE (M <= 16, N % 4 == 0, sf 16-byte aligned),
 *               Q8_GEMM_TCGEN05_PAIR (any M); others -> Q8_ERR_UNSUPPORTED.
 * Errors: as q8_gemm_epilogue_ex; group not 32 / 128 -> Q8_ERR_INVALID_ARG;
 * K % group != 0 -> Q8_ERR_UNSUPPORTED.
 */
q8_status q8_gemm_mx_ex(const int8_t* qa, const float* s_a, q8_granularity ga, const int8_t* qw,
                        const uint32_t* sf, int group, const float* bias, int64_t M, int64_t N,
                        int64_t K, q8_out_type out_type, void* out, float out_scale,
                        q8_gemm_kernel kernel, q8_stream_t stream);

/*
 * q8_gemm_mx_ex (kernel Q8_GEMM_AUTO) with a caller workspace, as q8_gemm_w4a8_ws:
 * where the CTA-pair kernel runs, the activation codes go once into the workspace
 * as fp16 values (each group of four K as K 0, 2, 1, 3) and are loaded by TMA; the
 * converter warps dequantize the weights only. The tensor core then sees the same
 * operands in the same order as without the workspace: y is bit-identical to that
 * of q8_gemm_mx_ex.
 * workspace, workspace_bytes : as q8_gemm_w4a8_ws (used iff >= 2 M K bytes and the
 * CTA-pair kernel runs). Other arguments and errors as q8_gemm_mx_ex.
 */
q8_status q8_gemm_mx_ws(const int8_t* qa, const float* s_a, q8_granularity ga, const int8_t* qw,
                        const uint32_t* sf, int group, const float* bias, int64_t M, int64_t N,
                        int64_t K, q8_out_type out_type, void* out, float out_scale,
                        void* workspace, size_t workspace_bytes, q8_stream_t stream);

/*
 * Activation codes stored as fp16 values. The quantization is that of
 * q8_quantize_act (the same scales, zero points and codes: rint of the IEEE
 * quotient, clamped), but each code is written as the fp16 number of equal value
 * (exact, |code| <= 128), two bytes per element. The pages store the codes as
 * int8; the fp16 form is the operand type of this library's tensor-core GEMM,
 * which otherwise converts every activation code once per 256-column output tile
 * it enters. Written once per code here, it is converted once in all. The
 * weights stay int8.
 *
 * qa16 : fp16 bit patterns [M, K], written, 16-byte aligned. Other arguments and
 * errors as q8_quantize_act.
 */
q8_status q8_quantize_act_f16(const float* a, int64_t M, int64_t K, q8_granularity g,
                              q8_symmetry sym, uint16_t* qa16, float* s_a, int32_t* z_a,
                              q8_stream_t stream);

/*
 * q8_quantize_act that also writes the codes as fp16 values (in K order, the
 * format of q8_quantize_act_f16) into qa16: the int8 codes stay the stored
 * activation format, and qa16 is the operand q8_gemm_f16a_ex loads by TMA.
 * Per-token rows of up to 32768 elements take one pass over a (both formats from
 * the row held in registers); otherwise q8_quantize_act runs, then a copy kernel.
 *
 * qa16 : fp16 bit patterns [M, K], written, 16-byte aligned, not overlapping the
 *        other buffers. Other arguments and errors as q8_quantize_act.
 */
q8_status q8_quantize_act_dual(const float* a, int64_t M, int64_t K, q8_granularity g,
                               q8_symmetry sym, int8_t* qa, uint16_t* qa16, float* s_a,
                               int32_t* z_a, q8_stream_t stream);

/*
 * q8_linear with a caller workspace: where q8_gemm_workspace(M, N, K) is nonzero
 * and workspace_bytes reaches it, the quantizer writes the codes both to qa (int8)
 * and into the workspace (fp16 values, q8_quantize_act_dual) in one pass, and the
 * CTA-pair kernel loads the fp16 copy by TMA (q8_gemm_f16a_ex). y, qa, s_a and z_a
 * are those of q8_linear, bit for bit. Otherwise (workspace NULL or too small, or
 * a shape on another kernel) the call is q8_linear.
 *
 * workspace : NULL, or 16-byte aligned device memory, overwritten when used; the
 *             caller owns it and may reuse it once the call's work on `stream` has
 *             completed; it must not overlap any other buffer of the call.
 * Other arguments and errors as q8_linear; a misaligned workspace returns
 * Q8_ERR_INVALID_ARG.
 */
q8_status q8_linear_ws(const float* a, int64_t M, int64_t K, q8_granularity ga, q8_symmetry sym,
                       int8_t* qa, float* s_a, int32_t* z_a, const int8_t* qw, const float* s_w,
                       q8_granularity gw, const int32_t* colsum, int64_t N, float* y,
                       void* workspace, size_t workspace_bytes, q8_stream_t stream);

/*
 * q8_gemm_epilogue_ex on activation codes from q8_quantize_act_f16: the same
 * INT8 x INT8 -> INT32 products and sums (the fp16 values are the int8 codes),
 * the same epilogue and output types, on the CTA-pair tcgen05 kernel (TMA loads
 * the fp16 codes straight into its operand stages). qa16 values must be integers
 * in [-128, 127]; other values give unspecified results.
 * Errors as q8_gemm_epilogue_ex.
 */
q8_status q8_gemm_f16a_ex(const uint16_t* qa16, const float* s_a, const int32_t* z_a,
                          q8_granularity ga, const int8_t* qw, const float* s_w,
                          q8_granularity gw, const int32_t* colsum, const float* bias, int64_t M,
                          int64_t N, int64_t K, q8_out_type out_type, void* out, float out_scale,
                          q8_stream_t stream);

/* The raw INT32 accumulators of q8_gemm_f16a_ex (as q8_gemm_s32_ex). */
q8_status q8_gemm_f16a_s32(const uint16_t* qa16, const int8_t* qw, int64_t M, int64_t N, int64_t K,
                           int32_t* acc, q8_stream_t stream);

/*
 * The whole layer on host buffers ("Activation Quantization Architecture", the
 * quantizer itself and the integer GEMM; Day 98's epilogue): A fp32 [M, K] in host
 * memory -> per-token quantization (symmetric, or asymmetric with colsum) -> the
 * INT32 GEMM against device-resident weights -> y fp32 [M, N] in host memory. The
 * token rows go through in slices of chunk_rows rows (0: about a sixteenth of M,
 * whole 256-row tiles): the copy of one slice in, the device work on the previous
 * one and the copy out of the one before overlap. y is the same as that of
 * q8_quantize_act (Q8_PER_ROW) + q8_gemm_dequant over all rows.
 *
 * a_host, y_host : host memory; page-locked (cudaHostAlloc / pinned) for the copies
 *                  to overlap, else they run synchronously. a_host may be NULL iff K == 0.
 * qw, s_w, gw, colsum : device buffers as q8_gemm_dequant (colsum iff asymmetric).
 * workspace      : device memory of at least q8_linear_host_workspace(M, N, K,
 *                  chunk_rows) bytes, 256-byte aligned, owned by the caller; not
 *                  touched after the call's work on `stream` completes.
 * stream         : the device work runs on it; the call returns once everything is
 *                  queued, and `stream` completes only after the last slice of y has
 *                  reached the host. The first call on a device creates two copy
 *                  streams and seven events, kept until the process exits; calls from
 *                  several host threads are queued one after another.
 * Errors: Q8_ERR_INVALID_ARG (sizes, pointers, alignment, a workspace too small),
 * Q8_ERR_UNSUPPORTED (K % 16, K above the int32 bound), Q8_ERR_CUDA.
 */
size_t q8_linear_host_workspace(int64_t M, int64_t N, int64_t K, int64_t chunk_rows);
q8_status q8_linear_host(const float* a_host, int64_t M, int64_t K, q8_symmetry sym, const int8_t* qw,
                         const float* s_w, q8_granularity gw, const int32_t* colsum, int64_t N,
                         float* y_host, int64_t chunk_rows, void* workspace, size_t workspace_bytes,
                         q8_stream_t stream);

/*
 * q8_linear_host without a caller-supplied workspace: the same layer, the same result,
 * for callers that cannot allocate device memory themselves. Examples: a plugin inside an
 * inference server or framework whose device memory all belongs to the host
 * application's pool (allocating outside it breaks the pool's accounting and limits),
 * and code on a latency-critical path, where cudaMalloc/cudaFree are off limits because
 * they can synchronize the whole device. No counterpart in the source material: this is
 * a packaging of the layer, not a step of the method.
 *
 * The workspace is a fixed device array of q8_linear_host_static_limit() bytes
 * (64 MiB) inside this library. Every device that loads the library holds it until the
 * process exits, and every call on that device uses the same array; nothing in it has to
 * start at zero, and it keeps whatever the last call left. Calls whose device work
 * overlaps (on different streams, or from different host threads onto different
 * streams) race on the array; calls on one stream run one after another and do not.
 * The call allocates no device memory (no cudaMalloc / cudaFree, no allocating library
 * routine). Every call looks up the array's device address with the device current (the
 * first lookup on a device loads the library's device code there). The first call on a
 * device also does set-up: it creates the two copy streams and seven events that
 * q8_linear_host keeps per device; make that first call before any stream capture.
 *
 * Arguments as q8_linear_host. chunk_rows = 0 picks the largest slice whose two
 * workspace slots fit the array (whole 256-row tiles when one fits). Errors: as
 * q8_linear_host, checked first and in the same order; then Q8_ERR_UNSUPPORTED when
 * q8_linear_host_workspace(M, N, K, chunk_rows) (or, for chunk_rows = 0, that of a
 * one-row slice) exceeds the array.
 */
size_t q8_linear_host_static_limit(void);
q8_status q8_linear_host_static(const float* a_host, int64_t M, int64_t K, q8_symmetry sym, const int8_t* qw,
                                const float* s_w, q8_granularity gw, const int32_t* colsum, int64_t N,
                                float* y_host, int64_t chunk_rows, q8_stream_t stream);

/*
 * Diagnostic export of the raw INT32 accumulators acc[m][n] (no epilogue),
 * computed by the same main loop as q8_gemm_dequant_ex with the same kernel
 * choice. Used to check the integer GEMM bit for bit.
 * acc : int32 [M, N], written. K <= 131056.
 */
q8_status q8_gemm_s32_ex(const int8_t* qa, const int8_t* qw, int64_t M, int64_t N, int64_t K,
                         int32_t* acc, q8_gemm_kernel kernel, q8_stream_t stream);

/*
 * Self-test of the device-side failure path behind Q8_ERR_TIMEOUT (the bounded
 * waits of the tensor-core and decode kernels). No counterpart in the pages:
 * it exercises this library's own error handling.
 *
 * Runs `kernel` (Q8_GEMM_DECODE, M <= 16, or Q8_GEMM_TCGEN05) on the given
 * operands with its TMA producer issuing no load and the wait of its converter
 * (decode: compute) warps on the first loaded stage limited to wait_cycles SM
 * clock cycles. That wait runs out with no copy and no MMA in flight; the kernel
 * records it in the device error word, its other roles leave on the kernel's
 * abort flag, tensor memory is released, and acc is not written. Afterwards
 * q8_device_error returns Q8_ERR_TIMEOUT with code 2 << 16 (decode kernel: its
 * compute warps' wait) or 2 (tcgen05 kernel: its converters' wait), and later
 * calls run normally.
 *
 * qa, qw, M, N, K, acc : as q8_gemm_s32_ex (M, N, K > 0; acc is not written).
 * wait_cycles          : 1 .. 2^31.
 * Errors: Q8_ERR_INVALID_ARG for another kernel, wait_cycles out of range, or
 * the argument errors of q8_gemm_s32_ex; Q8_ERR_UNSUPPORTED when the kernel
 * cannot run the shape.
 */
q8_status q8_selftest_wait_timeout(q8_gemm_kernel kernel, const int8_t* qa, const int8_t* qw,
                                   int64_t M, int64_t N, int64_t K, int32_t* acc,
                                   int64_t wait_cycles, q8_stream_t stream);

/* The kernel q8_gemm_dequant would run for this shape (never Q8_GEMM_AUTO). */
q8_gemm_kernel q8_gemm_pick(int64_t M, int64_t N, int64_t K);

/* Static description of a status code. Never NULL. */
const char* q8_status_string(q8_status status);

/*
 * Device-side error word of the current device: 0 if every bounded wait of a
 * tensor-core kernel completed, otherwise a nonzero code naming the wait that
 * gave up: one byte per kernel family (bits 0..7: the single-CTA tcgen05 kernel,
 * and bit 7 the fused RMSNorm quantizer's wait for a row copy; bits 8..15: the
 * tcgen05 decode kernel; bits 16..23: the warp-MMA decode kernels; bits 24..31:
 * the CTA-pair kernel), within a byte one bit per role (1 TMA producer,
 * 2 converters / compute warps waiting for loaded data, 4 converters waiting
 * for a free stage, 8 MMA issuer waiting for converted data, 16 MMA issuer
 * waiting for a free accumulator, 32 accumulator drain, 64 the odd CTA's relay).
 * Synchronises the device. Reading it resets it to 0. A nonzero value means the
 * outputs of the kernel that set it are invalid.
 */
q8_status q8_device_error(uint32_t* code_out);

/* Number of kernels this library has launched in this process (all devices). */
uint64_t q8_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* Q8_H_ */
