/*
 * q8_oracle.c -- plain, slow CPU oracle for the W8A8 quantized linear layer.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the independent reference that the
 * CUDA path is checked against. It shares no code, header, table or helper
 * with the library under int8_quantized_gemm_gb300/. Only tests/, the smoke
 * check in __graft_entry__.py and the cpu_baseline leg of bench.py may load
 * it. The product never calls it.
 *
 * Build: gcc -O2 -ffp-contract=off (no -ffast-math) so that every fp32
 * operation below is one IEEE-754 single-precision operation, rounded to
 * nearest-even, in exactly the order written. Integer dot products
 * accumulate in int64, so they cannot overflow for any K this file accepts.
 *
 * Steps and the passages they follow:
 *  - symmetric scale s = max|x| / 127, codes clamp(rint(x/s), -127, 127):
 *      "100 Days of GPU, Day 98" (What a scale actually promises);
 *      "Write Int8 Quantized Kernel" (Required reasoning process, step 1);
 *      "Activation Quantization Architecture" (The quantizer itself, and the
 *      numpy reference quantize_per_token / quantize_per_channel).
 *    The zero-row guard is applied to amax before the divide, as in the fused
 *    norm+quantize pseudocode of "Activation Quantization Architecture"
 *    (Fusion): s = max(amax, 1e-8) / 127.
 *  - asymmetric scale and zero point: Day 98 (z is the code that dequantizes
 *    to zero) and "Write Int8 Quantized Kernel" step 1 (s = (max-min)/255,
 *    z = round(-min/s)), stored in the int8 range [-128, 127]:
 *      lo = min(min x, 0), hi = max(max x, 0), s = max(hi - lo, 1e-8) / 255,
 *      z  = clamp(-128 - rint(lo / s), -128, 127),
 *      q  = clamp(rint(x / s) + z, -128, 127).
 *  - integer dot product acc[m][n] = sum_k qa[m][k] * qw[n][k] (Day 98, the
 *    accumulate loop; "Activation Quantization Architecture", The integer
 *    GEMM, written out), here in int64.
 *  - column sums colsum[n] = sum_k qw[n][k] (Day 98, the zero-point paragraph
 *    after the kernel listing).
 *  - epilogue corr = acc - z * colsum, y = (float)corr * (s_a * s_w), the
 *    multiply order of the Day 98 epilogue listing.
 *  - epilogue variants ("Activation Quantization Architecture", Fusion: the
 *    epilogue multiplies by the per-token and per-channel scales, adds the bias
 *    and writes bf16; some kernels quantize the output for the next GEMM):
 *      y = fl(corr * scale) + bias[n] (one fp32 add), then either fp32, bf16
 *    rounded to nearest-even, or int8 codes clamp(rint(y / s_out), -127, 127)
 *    with a static per-tensor output scale s_out.
 *  - int4 weights for W4A8 (TileLang tutorial ch. 27, low-precision quantization:
 *    2.4 int8 / int4, qmax = 7, s = absmax / qmax, q = clip(round(x / s), -qmax-1,
 *    qmax); its int4 GEMM and dequantize-GEMM examples: two codes per byte,
 *    (a & 0x0F) | ((b & 0x0F) << 4), decoded by shifting left 4 and then right 4
 *    arithmetically to sign-extend).
 *  - MX-style block-scaled int8 weights (TileLang tutorial ch. 27, low-precision
 *    quantization, 2.3 MX / block-scaled: block granularity + E8M0): every G
 *    consecutive K elements of a weight row share one scale 2^(e - 127) stored
 *    as its biased exponent byte e, amax / qmax rounded up to a power of two;
 *    four scale bytes per 32-bit word, words laid out group-major (see
 *    q8o_quantize_weight_mx). The product is accumulated exactly and rounded
 *    once (q8o_gemm_mx).
 *  - fused RMSNorm + per-token quantization ("Activation Quantization
 *    Architecture", Fusion: the fused norm-and-quantize pseudocode):
 *      rms = sqrt(mean(x * x) + eps), y = x / rms * gamma, then the symmetric
 *    per-token quantizer above on y (see q8o_rmsnorm for the summation reading).
 * rint() is round-half-to-even in the default rounding mode, matching np.rint
 * in the numpy reference of "Activation Quantization Architecture".
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>

#define Q8O_ZERO_GUARD 1e-8f

/* Status codes of the oracle (not the library's). */
enum { Q8O_OK = 0, Q8O_BAD_ARG = 1, Q8O_INT32_OVERFLOW = 2 };

static float q8o_absf(float v) { return v < 0.0f ? -v : v; }

static int q8o_clampi(long v, int lo, int hi) {
    if (v < lo) return lo;
    if (v > hi) return hi;
    return (int)v;
}

/* amax over n values (exact: comparisons only). */
static float q8o_amax(const float* x, int64_t n) {
    float m = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = q8o_absf(x[i]);
        if (a > m) m = a;
    }
    return m;
}

float q8o_sym_scale(float amax) {
    float g = amax > Q8O_ZERO_GUARD ? amax : Q8O_ZERO_GUARD;
    return g / 127.0f;
}

int q8o_sym_code(float x, float s) {
    float r = rintf(x / s);
    return q8o_clampi((long)r, -127, 127);
}

/*
 * Symmetric quantization of a rows x cols fp32 matrix (row-major).
 * per_row != 0: one scale per row (per token for A, per output channel for a
 * K-major W[N, K]); s has `rows` entries. per_row == 0: one scale for the
 * whole tensor; s has one entry.
 */
int q8o_quantize_sym(const float* x, int64_t rows, int64_t cols, int per_row,
                     int8_t* q, float* s) {
    if (rows < 0 || cols < 0) return Q8O_BAD_ARG;
    if (!per_row) {
        float amax = q8o_amax(x, rows * cols);
        float sc = q8o_sym_scale(amax);
        s[0] = sc;
        for (int64_t i = 0; i < rows * cols; ++i) q[i] = (int8_t)q8o_sym_code(x[i], sc);
        return Q8O_OK;
    }
    for (int64_t r = 0; r < rows; ++r) {
        const float* xr = x + r * cols;
        float sc = q8o_sym_scale(q8o_amax(xr, cols));
        s[r] = sc;
        for (int64_t c = 0; c < cols; ++c) q[r * cols + c] = (int8_t)q8o_sym_code(xr[c], sc);
    }
    return Q8O_OK;
}

/* Range of a set of values, widened to include 0 so that 0 has a code. */
static void q8o_range0(const float* x, int64_t n, float* lo, float* hi) {
    float a = 0.0f, b = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        if (x[i] < a) a = x[i];
        if (x[i] > b) b = x[i];
    }
    *lo = a;
    *hi = b;
}

void q8o_asym_params(float lo, float hi, float* s, int* z) {
    float span = hi - lo;
    float g = span > Q8O_ZERO_GUARD ? span : Q8O_ZERO_GUARD;
    float sc = g / 255.0f;
    float r = rintf(lo / sc);
    *s = sc;
    *z = q8o_clampi(-128L - (long)r, -128, 127);
}

int q8o_asym_code(float x, float s, int z) {
    float r = rintf(x / s);
    return q8o_clampi((long)r + (long)z, -128, 127);
}

/* Asymmetric quantization; s and z have `rows` entries (per_row) or one. */
int q8o_quantize_asym(const float* x, int64_t rows, int64_t cols, int per_row,
                      int8_t* q, float* s, int32_t* z) {
    if (rows < 0 || cols < 0) return Q8O_BAD_ARG;
    if (!per_row) {
        float lo, hi, sc;
        int zp;
        q8o_range0(x, rows * cols, &lo, &hi);
        q8o_asym_params(lo, hi, &sc, &zp);
        s[0] = sc;
        z[0] = zp;
        for (int64_t i = 0; i < rows * cols; ++i) q[i] = (int8_t)q8o_asym_code(x[i], sc, zp);
        return Q8O_OK;
    }
    for (int64_t r = 0; r < rows; ++r) {
        const float* xr = x + r * cols;
        float lo, hi, sc;
        int zp;
        q8o_range0(xr, cols, &lo, &hi);
        q8o_asym_params(lo, hi, &sc, &zp);
        s[r] = sc;
        z[r] = zp;
        for (int64_t c = 0; c < cols; ++c) q[r * cols + c] = (int8_t)q8o_asym_code(xr[c], sc, zp);
    }
    return Q8O_OK;
}

/* colsum[n] = sum_k qw[n][k], in int64. */
void q8o_colsum(const int8_t* qw, int64_t N, int64_t K, int64_t* colsum) {
    for (int64_t n = 0; n < N; ++n) {
        int64_t t = 0;
        for (int64_t k = 0; k < K; ++k) t += qw[n * K + k];
        colsum[n] = t;
    }
}

/* One integer dot product of length K, in int64. */
int64_t q8o_dot(const int8_t* a, const int8_t* b, int64_t K) {
    int64_t t = 0;
    for (int64_t k = 0; k < K; ++k) t += (int64_t)a[k] * (int64_t)b[k];
    return t;
}

/* acc[m][n] = sum_k qa[m][k] * qw[n][k] for all m, n (int64 out). */
void q8o_gemm_acc(const int8_t* qa, const int8_t* qw, int64_t M, int64_t N, int64_t K,
                  int64_t* acc, int threads) {
    (void)threads;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads > 0 ? threads : 1)
#endif
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) acc[m * N + n] = q8o_dot(qa + m * K, qw + n * K, K);
}

/*
 * Epilogue for one element: corr = acc - z * colsum (int64), must fit int32;
 * y = (float)corr * (s_a * s_w). Returns Q8O_INT32_OVERFLOW if corr or acc
 * leaves the int32 range (the value is still written).
 */
int q8o_epilogue_one(int64_t acc, int32_t z, int64_t colsum, float sa, float sw, float* y) {
    int64_t corr = acc - (int64_t)z * colsum;
    float scale = sa * sw;
    *y = (float)corr * scale;
    if (acc > INT32_MAX || acc < INT32_MIN || corr > INT32_MAX || corr < INT32_MIN)
        return Q8O_INT32_OVERFLOW;
    return Q8O_OK;
}

/*
 * Full linear layer on codes already quantized: y[m][n] for all m, n.
 * sa has M entries if a_per_row else 1; za is NULL (symmetric) or has M / 1
 * entries; sw has N entries if w_per_row else 1. Returns the worst status.
 */
int q8o_linear_codes(const int8_t* qa, const float* sa, const int32_t* za, int a_per_row,
                     const int8_t* qw, const float* sw, int w_per_row,
                     int64_t M, int64_t N, int64_t K, float* y, int threads) {
    int status = Q8O_OK;
    (void)threads;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads > 0 ? threads : 1) reduction(max : status)
#endif
    for (int64_t m = 0; m < M; ++m) {
        float a_s = sa[a_per_row ? m : 0];
        int32_t a_z = za ? za[a_per_row ? m : 0] : 0;
        for (int64_t n = 0; n < N; ++n) {
            int64_t acc = q8o_dot(qa + m * K, qw + n * K, K);
            int64_t cs = 0;
            if (za) {
                for (int64_t k = 0; k < K; ++k) cs += qw[n * K + k];
            }
            int st = q8o_epilogue_one(acc, a_z, cs, a_s, sw[w_per_row ? n : 0], &y[m * N + n]);
            if (st > status) status = st;
        }
    }
    return status;
}

/* y at a list of (m, n) pairs; same arguments as q8o_linear_codes. */
/*
 * The linear layer from codes with the epilogue variants of "Activation
 * Quantization Architecture" (Fusion): y = fl((float)corr * (s_a * s_w)) as in
 * q8o_linear_codes, then y + bias[n] in fp32 when bias is given.
 */
int q8o_linear_codes_bias(const int8_t* qa, const float* sa, const int32_t* za, int a_per_row,
                          const int8_t* qw, const float* sw, int w_per_row, const float* bias,
                          int64_t M, int64_t N, int64_t K, float* y, int threads) {
    int status = q8o_linear_codes(qa, sa, za, a_per_row, qw, sw, w_per_row, M, N, K, y, threads);
    if (bias) {
        for (int64_t m = 0; m < M; ++m)
            for (int64_t n = 0; n < N; ++n) y[m * N + n] = y[m * N + n] + bias[n];
    }
    return status;
}

/*
 * fp32 -> bf16 with round-to-nearest-even on the bit pattern: keep the high 16
 * bits after adding 0x7FFF plus the lowest kept bit (finite inputs; the pages
 * name bf16 as the epilogue's output type).
 */
void q8o_to_bf16(const float* y, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) {
        uint32_t u;
        memcpy(&u, &y[i], sizeof u);
        u += 0x7FFFu + ((u >> 16) & 1u);
        out[i] = (uint16_t)(u >> 16);
    }
}

/* Static output quantization for the next GEMM: clamp(rint(y / s_out), -127, 127). */
void q8o_quantize_static(const float* y, int64_t n, float s_out, int8_t* q) {
    for (int64_t i = 0; i < n; ++i) q[i] = (int8_t)q8o_sym_code(y[i], s_out);
}

int q8o_linear_codes_at(const int8_t* qa, const float* sa, const int32_t* za, int a_per_row,
                        const int8_t* qw, const float* sw, int w_per_row, int64_t K,
                        const int64_t* ms, const int64_t* ns, int64_t count,
                        float* y, int64_t* acc_out) {
    int status = Q8O_OK;
    for (int64_t i = 0; i < count; ++i) {
        int64_t m = ms[i], n = ns[i];
        int64_t acc = q8o_dot(qa + m * K, qw + n * K, K);
        int64_t cs = 0;
        if (za) {
            for (int64_t k = 0; k < K; ++k) cs += qw[n * K + k];
        }
        if (acc_out) acc_out[i] = acc;
        int st = q8o_epilogue_one(acc, za ? za[a_per_row ? m : 0] : 0, cs,
                                  sa[a_per_row ? m : 0], sw[w_per_row ? n : 0], &y[i]);
        if (st > status) status = st;
    }
    return status;
}

/*
 * Symmetric int4 quantization of each row of w[rows][cols] (per output channel):
 * s = max(absmax, 1e-8) / 7, q = clamp(rint(w / s), -8, 7) (-8 is reachable only
 * through rounding, as |w / s| <= 7 up to one ulp). Codes are returned one per
 * int8 element; q8o_pack_int4 packs them.
 */
int q8o_quantize_int4(const float* w, int64_t rows, int64_t cols, int8_t* q, float* s) {
    if (rows < 0 || cols < 0) return Q8O_BAD_ARG;
    for (int64_t r = 0; r < rows; ++r) {
        const float* wr = w + r * cols;
        const float amax = q8o_amax(wr, cols);
        const float sc = (amax > Q8O_ZERO_GUARD ? amax : Q8O_ZERO_GUARD) / 7.0f;
        s[r] = sc;
        for (int64_t k = 0; k < cols; ++k) q[r * cols + k] = (int8_t)q8o_clampi((long)rintf(wr[k] / sc), -8, 7);
    }
    return Q8O_OK;
}

/* Two int4 codes per byte along each row: byte i = (q[2i] & 0x0F) | ((q[2i+1] & 0x0F) << 4). */
int q8o_pack_int4(const int8_t* q, int64_t rows, int64_t cols, uint8_t* packed) {
    if (rows < 0 || cols < 0 || (cols & 1)) return Q8O_BAD_ARG;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t i = 0; i < cols / 2; ++i) {
            const uint8_t lo = (uint8_t)(q[r * cols + 2 * i] & 0x0F);
            const uint8_t hi = (uint8_t)(q[r * cols + 2 * i + 1] & 0x0F);
            packed[r * (cols / 2) + i] = (uint8_t)(lo | (hi << 4));
        }
    return Q8O_OK;
}

/* Inverse of q8o_pack_int4: each nibble sign-extended (shift left 4, arithmetic right 4). */
int q8o_unpack_int4(const uint8_t* packed, int64_t rows, int64_t cols, int8_t* q) {
    if (rows < 0 || cols < 0 || (cols & 1)) return Q8O_BAD_ARG;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t i = 0; i < cols / 2; ++i) {
            const int b = packed[r * (cols / 2) + i];
            const int lo = ((int)(int8_t)(uint8_t)(b << 4)) >> 4;
            const int hi = ((int)(int8_t)(uint8_t)b) >> 4;
            q[r * cols + 2 * i] = (int8_t)lo;
            q[r * cols + 2 * i + 1] = (int8_t)hi;
        }
    return Q8O_OK;
}

/*
 * RMSNorm of each row of x[rows][cols] with per-column weights gamma[cols]
 * ("Activation Quantization Architecture", Fusion pseudocode):
 *   rms = sqrt(mean(x * x) + eps),  y = x / rms * gamma.
 * The pages do not fix the order of the sum in mean(x * x). Reading taken: the
 * sum S of the exact squares x_k^2 is formed exactly and rounded once to fp32,
 * so that the value does not depend on any order. Here each square is exact in
 * long double (a 24-bit significand squared needs 48 bits) and the running sum
 * keeps at least 64 significand bits, far below one fp32 ulp of S for any row
 * length this file is used with. After that every step is one fp32 operation in
 * the order written: mean = fl(fl(S) / cols), r = sqrtf(fl(mean + eps)),
 * y_k = fl(fl(x_k / r) * gamma_k). sumsq[row] (optional) receives S as a double.
 */
int q8o_rmsnorm(const float* x, const float* gamma, int64_t rows, int64_t cols, float eps, float* y,
                double* sumsq) {
    if (rows < 0 || cols <= 0 || !(eps >= 0.0f)) return Q8O_BAD_ARG;
    for (int64_t r = 0; r < rows; ++r) {
        const float* xr = x + r * cols;
        long double acc = 0.0L;
        for (int64_t k = 0; k < cols; ++k) {
            const long double v = (long double)xr[k];
            acc += v * v;
        }
        if (sumsq) sumsq[r] = (double)acc;
        const float ms = (float)acc;                 /* one rounding of the exact sum */
        const float mean = ms / (float)cols;
        const float rms = sqrtf(mean + eps);
        float* yr = y + r * cols;
        for (int64_t k = 0; k < cols; ++k) yr[k] = (xr[k] / rms) * gamma[k];
    }
    return Q8O_OK;
}

/*
 * MX-style block-scaled int8 weights (TileLang tutorial ch. 27, low-precision
 * quantization, 2.3 MX / block-scaled: block granularity + E8M0).
 *
 * Each row n of w[N][K] is cut into groups of G consecutive K elements. A group's
 * scale is a bare power of two s = 2^(e - 127), stored as the E8M0 byte e: the
 * pages form it from x = amax / qmax by taking the biased exponent field of x and
 * adding one when x's 23 mantissa bits are not all zero (x rounded up to a power of
 * two, so every |w / s| <= qmax). Here qmax = 127 (the int8 rule of 2.4) and the
 * codes are clamp(rint(w / s), -127, 127); dividing by a power of two is exact.
 * Reading: e is clamped to [103, 136] (s from 2^-24 to 2^9) where the pages clamp
 * to [1, 254]; in that range every q * s is an exact fp16 value. A zero group gets
 * e = 103 and codes 0.
 * Layout (2.3 (c)): four scale bytes are packed into one 32-bit word, byte b
 * (bits 8b .. 8b + 7) holding group 4w + b of word w, and the words are stored
 * group-major: word w of row n at sf[w * N + n]. Bytes past the last group are 0.
 */
#define Q8O_MX_EMIN 103
#define Q8O_MX_EMAX 136

int q8o_e8m0_ceil(float x) {
    uint32_t bits;
    memcpy(&bits, &x, sizeof bits);
    bits &= 0x7FFFFFFFu;
    const int e = (int)(bits >> 23) + ((bits & 0x7FFFFFu) != 0 ? 1 : 0);
    return q8o_clampi(e, Q8O_MX_EMIN, Q8O_MX_EMAX);
}

int q8o_quantize_weight_mx(const float* w, int64_t N, int64_t K, int G, int8_t* q, uint32_t* sf) {
    if (N < 0 || K < 0 || G <= 0 || K % G != 0) return Q8O_BAD_ARG;
    const int64_t groups = K / G, words = (groups + 3) / 4;
    for (int64_t i = 0; i < words * N; ++i) sf[i] = 0;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t g = 0; g < groups; ++g) {
            const float* wg = w + n * K + g * G;
            const float x = q8o_amax(wg, G) / 127.0f;
            const int e = q8o_e8m0_ceil(x);
            const float s = ldexpf(1.0f, e - 127);
            sf[(g / 4) * N + n] |= (uint32_t)e << (8 * (g % 4));
            for (int64_t k = 0; k < G; ++k)
                q[n * K + g * G + k] = (int8_t)q8o_clampi((long)rintf(wg[k] / s), -127, 127);
        }
    return Q8O_OK;
}

/* Nearest fp32 to v * 2^-24 (ties to even), for an exact 128-bit integer v. */
static float q8o_round_i128_unit24(__int128 v) {
    const int neg = v < 0;
    unsigned __int128 u = neg ? (unsigned __int128)0 - (unsigned __int128)v : (unsigned __int128)v;
    int top = 0;
    while (top < 127 && (u >> (top + 1)) != 0) ++top;
    int shift = top - 23;
    if (shift > 0) {
        const unsigned __int128 rem = u & (((unsigned __int128)1 << shift) - 1);
        const unsigned __int128 half = (unsigned __int128)1 << (shift - 1);
        u >>= shift;
        if (rem > half || (rem == half && (u & 1))) ++u;
    } else {
        shift = 0;
    }
    const float r = ldexpf((float)(uint32_t)u, shift - 24);   /* u < 2^25: exact */
    return neg ? -r : r;
}

/*
 * T[m][n] = sum_k qa[m][k] * q[n][k] * s[n][k / G] with the scales of
 * q8o_quantize_weight_mx, formed exactly and rounded once to fp32. Each group's
 * integer dot product is exact in int64; a group term is that integer times
 * 2^(e - 103) in units of 2^-24 (e >= 103), summed exactly in a 128-bit integer.
 * absum[m][n] (optional) receives sum_k |qa * q * s| in double (for error bounds).
 */
int q8o_gemm_mx(const int8_t* qa, const int8_t* q, const uint32_t* sf, int64_t M, int64_t N, int64_t K, int G,
                float* t, double* absum, int threads) {
    if (M < 0 || N < 0 || K < 0 || G <= 0 || K % G != 0) return Q8O_BAD_ARG;
    const int64_t groups = K / G;
    (void)threads;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads > 0 ? threads : 1)
#endif
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            __int128 sum = 0;
            double abs_acc = 0.0;
            for (int64_t g = 0; g < groups; ++g) {
                const int e = (int)((sf[(g / 4) * N + n] >> (8 * (g % 4))) & 0xFFu);
                if (e < Q8O_MX_EMIN || e > Q8O_MX_EMAX) continue;   /* not produced by the quantizer */
                int64_t dot = 0, adot = 0;
                for (int64_t k = g * G; k < (g + 1) * G; ++k) {
                    const int64_t p = (int64_t)qa[m * K + k] * (int64_t)q[n * K + k];
                    dot += p;
                    adot += p < 0 ? -p : p;
                }
                sum += (__int128)dot << (e - Q8O_MX_EMIN);
                abs_acc += ldexp((double)adot, e - 127);
            }
            t[m * N + n] = q8o_round_i128_unit24(sum);
            if (absum) absum[m * N + n] = abs_acc;
        }
    return Q8O_OK;
}

/* y[m][n] = fl(T[m][n] * s_a[m]) (+ bias[n], one fp32 add): the block-scaled layer. */
int q8o_linear_mx(const int8_t* qa, const float* sa, int a_per_row, const int8_t* q, const uint32_t* sf,
                  const float* bias, int64_t M, int64_t N, int64_t K, int G, float* y, int threads) {
    const int st = q8o_gemm_mx(qa, q, sf, M, N, K, G, y, NULL, threads);
    if (st != Q8O_OK) return st;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            float v = y[m * N + n] * sa[a_per_row ? m : 0];
            if (bias) v = v + bias[n];
            y[m * N + n] = v;
        }
    return Q8O_OK;
}

int q8o_openmp_max_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
