// Activation / weight quantizers and weight column sums.
//
// These kernels are HBM-bound streams: each fp32 element is read once from
// HBM (4 bytes) and its code written once (1 byte). Per-row quantization keeps
// the whole row in registers between the range reduction and the code pass,
// so the row is never re-read. Results follow the rules in q8.h exactly: the
// codes are those of the IEEE fp32 quotient rounded half to even, and no multiply
// is contracted into an FMA unless written as one (the file is built with
// -fmad=false). Where a cheaper form than one division and one conversion per
// element gives the same bits, the argument is written beside it.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "q8_internal.h"
#include "q8_tc_ptx.cuh"

namespace q8 {

// Device error word of this file: bit 0x80 (reported in the lowest byte of q8_device_error) is
// set when the streaming RMSNorm quantizer's bounded wait for a row copy gave up.
static __device__ unsigned int g_quant_error;

namespace {

constexpr int kWarp = 32;

__device__ __forceinline__ int clampi(int v, int lo, int hi) { return min(max(v, lo), hi); }

// Symmetric scale from the absolute maximum.
__device__ __forceinline__ float sym_scale(float amax) {
    return __fdiv_rn(fmaxf(amax, kZeroGuard), 127.0f);
}

__device__ __forceinline__ void asym_params(float lo, float hi, float* s, int* z) {
    float span = __fsub_rn(hi, lo);
    float sc = __fdiv_rn(fmaxf(span, kZeroGuard), 255.0f);
    *s = sc;
    *z = clampi(-128 - __float2int_rn(__fdiv_rn(lo, sc)), -128, 127);
}

// 1.5 * 2^23: for |t| < 2^22, RN(t + kMagic) = kMagic + rint(t) (the addition rounds to the
// integer grid, half to even), so the low bits of its encoding hold rint(t) in two's complement
// (kMagicBits + rint(t)); no conversion instruction is needed.
constexpr float kMagic = 12582912.0f;
constexpr uint32_t kMagicBits = 0x4B400000u;

// rint(RN(x / s)), the code of the IEEE quotient rounded half to even, for |x / s| <= 256, from the
// row's reciprocal r = RN(1 / s). t = RN(x r) carries two roundings of relative size <= 2^-24 each,
// RN(x / s) one, so |t - RN(x / s)| <= 256 (1.5 2^-23 + 2^-48) < 2^-14. Unless t lies within 2^-14
// of a half-integer, no half-integer separates the two and they round to the same integer; near a
// half-integer (exact ties included) the IEEE quotient itself is rounded. t is rounded by the
// kMagic addition, and t - rint(t) is exact. Returns a word whose value minus kMagicBits is the
// integer (so its low byte is the int8 code).
__device__ __forceinline__ uint32_t rint_quot_bits(float x, float s, float r) {
    const float t = __fmul_rn(x, r);
    const float u = __fadd_rn(t, kMagic);
    if (fabsf(__fsub_rn(t, __fsub_rn(u, kMagic))) >= 0.5f - 0x1p-14f)
        return kMagicBits + (uint32_t)__float2int_rn(__fdiv_rn(x, s));
    return __float_as_uint(u);
}

// The symmetric clamp to [-127, 127] never binds: every x of the row (or tensor) has |x| <= amax
// and s = RN(max(amax, 1e-8) / 127) >= (amax / 127)(1 - 2^-24), so |RN(x / s)| < 127.0001 and its
// rint is at most 127 in magnitude (t above is within 2^-14 of it). The code is rint_quot_bits
// itself: its low byte.
__device__ __forceinline__ uint32_t sym_code(float x, float s, float r) {
    return rint_quot_bits(x, s, r);
}

// Asymmetric: clamp(rint(x / s) + z, -128, 127); zoff = z - kMagicBits (mod 2^32).
__device__ __forceinline__ uint32_t asym_code(float x, float s, float r, int zoff) {
    return (uint32_t)clampi((int)rint_quot_bits(x, s, r) + zoff, -128, 127);
}

// The low bytes of four words as one word, a's in the lowest byte.
__device__ __forceinline__ uint32_t pack4(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    return __byte_perm(__byte_perm(a, b, 0x0040u), __byte_perm(c, d, 0x0040u), 0x5410u);
}

// rint_quot_bits without its per-element branch: the word kMagicBits + rint(RN(x r)), and
// dmax = max(dmax, |t - rint(t)|). When dmax stays below 0.5 - 2^-14 for every element of a
// thread, each of its codes equals rint_quot_bits' (no t was near a half-integer); otherwise the
// thread recomputes its codes with rint_quot_bits (rare: about 2^-13 of the quotients).
__device__ __forceinline__ uint32_t rint_bits_tracked(float x, float r, float& dmax) {
    const float t = __fmul_rn(x, r);
    const float u = __fadd_rn(t, kMagic);
    dmax = fmaxf(dmax, fabsf(__fsub_rn(t, __fsub_rn(u, kMagic))));
    return __float_as_uint(u);
}
constexpr float kNearHalf = 0.5f - 0x1p-14f;

// The same from the exact product x r: u = RN(x r + kMagic) holds kMagicBits + rint(x r) (one
// rounding of the exact product to the integer grid), and d = RN(x r - rint(x r)) (one FMA) is
// within 2^-25 of the exact distance. x r (r = RN(1 / s), |x / s| <= 256) is within
// 256 * 2^-24 = 2^-16 of x / s, and RN(x / s) within 2^-16 of it too, so when |d| stays below
// kNearHalf no half-integer separates x r from RN(x / s) and both have the same rint.
__device__ __forceinline__ uint32_t rint_bits_fma_tracked(float x, float r, float& dmax) {
    const float u = __fmaf_rn(x, r, kMagic);
    dmax = fmaxf(dmax, fabsf(__fmaf_rn(x, r, -__fsub_rn(u, kMagic))));
    return __float_as_uint(u);
}

__device__ __forceinline__ uint32_t sym_codes4_tracked(float4 v, float r, float& dmax) {
    return pack4(rint_bits_fma_tracked(v.x, r, dmax), rint_bits_fma_tracked(v.y, r, dmax),
                 rint_bits_fma_tracked(v.z, r, dmax), rint_bits_fma_tracked(v.w, r, dmax));
}

// Codes of elements 4i .. 4i + 3 (the low bytes of a .. d) of a row (or tensor) whose codes start
// at q: int8 (one 32-bit word) or, for H, fp16 values (8 bytes). fp16: the half with bits
// 0x6400 | (byte ^ 0x80) is 1024 + (code + 128) exactly, and subtracting 1152 leaves the code.
template <bool H>
__device__ __forceinline__ void store_codes4(void* q, int64_t i, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    const uint32_t w = pack4(a, b, c, d);
    if constexpr (H) {
        uint32_t lo, hi;
        asm("sub.rn.f16x2 %0, %1, %2;\n" : "=r"(lo) : "r"(__byte_perm(w, 0x6464u, 0x5140u) ^ 0x00800080u),
            "r"(0x64806480u));
        asm("sub.rn.f16x2 %0, %1, %2;\n" : "=r"(hi) : "r"(__byte_perm(w, 0x6464u, 0x5342u) ^ 0x00800080u),
            "r"(0x64806480u));
        reinterpret_cast<uint2*>(q)[i] = make_uint2(lo, hi);
    } else {
        reinterpret_cast<uint32_t*>(q)[i] = w;
    }
}

// Codes of four elements into store_codes4 (the low byte of each word): symmetric, or asymmetric
// clamp(rint + z, -128, 127) with zoff = z - kMagicBits; tracked as rint_bits_tracked.
template <bool ASYM, bool H>
__device__ __forceinline__ void store_codes4_tracked(void* q, int64_t i, float4 v, float r, int zoff, float& dmax) {
    uint32_t c[4] = {rint_bits_tracked(v.x, r, dmax), rint_bits_tracked(v.y, r, dmax), rint_bits_tracked(v.z, r, dmax),
                     rint_bits_tracked(v.w, r, dmax)};
    if constexpr (ASYM) {
#pragma unroll
        for (int k = 0; k < 4; ++k) c[k] = (uint32_t)clampi((int)c[k] + zoff, -128, 127);
    }
    store_codes4<H>(q, i, c[0], c[1], c[2], c[3]);
}

// The same four codes with rint_quot_bits' near-half check (the exact path). DUAL: int8 codes to q
// and the same codes as fp16 values to q16 (both in K order).
template <bool ASYM, bool H, bool DUAL = false>
__device__ __forceinline__ void store_codes4_exact(void* q, int64_t i, float4 v, float s, float r, int zoff,
                                                   uint16_t* q16 = nullptr) {
    uint32_t c[4];
    if constexpr (ASYM) {
        c[0] = asym_code(v.x, s, r, zoff), c[1] = asym_code(v.y, s, r, zoff);
        c[2] = asym_code(v.z, s, r, zoff), c[3] = asym_code(v.w, s, r, zoff);
    } else {
        c[0] = sym_code(v.x, s, r), c[1] = sym_code(v.y, s, r), c[2] = sym_code(v.z, s, r), c[3] = sym_code(v.w, s, r);
    }
    store_codes4<H>(q, i, c[0], c[1], c[2], c[3]);
    if constexpr (DUAL) store_codes4<true>(q16, i, c[0], c[1], c[2], c[3]);
}

// Block-wide max of two values (hi, and nlo = -lo for the asymmetric range).
// All threads receive the results.
template <bool ASYM>
__device__ __forceinline__ void block_max2(float& hi, float& nlo, float* red) {
#pragma unroll
    for (int o = kWarp / 2; o > 0; o >>= 1) {
        hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
        if (ASYM) nlo = fmaxf(nlo, __shfl_xor_sync(0xffffffffu, nlo, o));
    }
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int nwarps = blockDim.x / kWarp;
    if (lane == 0) {
        red[warp] = hi;
        if (ASYM) red[32 + warp] = nlo;
    }
    __syncthreads();
    hi = lane < nwarps ? red[lane] : 0.0f;
    if (ASYM) nlo = lane < nwarps ? red[32 + lane] : 0.0f;
#pragma unroll
    for (int o = kWarp / 2; o > 0; o >>= 1) {
        hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
        if (ASYM) nlo = fmaxf(nlo, __shfl_xor_sync(0xffffffffu, nlo, o));
    }
}

// One CTA per row; each thread keeps up to VPT float4 of the row in registers.
// Requires cols % 4 == 0 and cols / 4 <= VPT * blockDim.x. DUAL: the int8 codes and, in q16, the
// same codes as fp16 values.
template <int VPT, bool ASYM, bool H = false, bool DUAL = false>
__global__ void __launch_bounds__(1024, (VPT <= 4 ? 2 : 1)) quantize_rows_kernel(const float* __restrict__ x, int64_t cols,
                                                            void* __restrict__ q,
                                                            float* __restrict__ s,
                                                            int32_t* __restrict__ z,
                                                            uint16_t* __restrict__ q16) {
    __shared__ float red[64];
    // A decode GEMM launched after this kernel with programmatic stream serialization may start
    // its weight stream now; it reads the codes and scales only after waiting for this grid.
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    const int64_t row = blockIdx.x;
    const int64_t n4 = cols / 4;
    const float4* xr = reinterpret_cast<const float4*>(x + row * cols);
    float4 v[VPT];
    float hi = 0.0f, nlo = 0.0f;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int64_t i = threadIdx.x + (int64_t)j * blockDim.x;
        if (i < n4) {
            v[j] = __ldcs(xr + i);   // streamed once: evict-first
            if (ASYM) {
                hi = fmaxf(hi, fmaxf(fmaxf(v[j].x, v[j].y), fmaxf(v[j].z, v[j].w)));
                nlo = fmaxf(nlo, -fminf(fminf(v[j].x, v[j].y), fminf(v[j].z, v[j].w)));
            } else {
                hi = fmaxf(hi, fmaxf(fmaxf(fabsf(v[j].x), fabsf(v[j].y)),
                                     fmaxf(fabsf(v[j].z), fabsf(v[j].w))));
            }
        }
    }
    block_max2<ASYM>(hi, nlo, red);
    float sc;
    int zp = 0;
    if (ASYM) {
        asym_params(-nlo, hi, &sc, &zp);
    } else {
        sc = sym_scale(hi);
    }
    if (threadIdx.x == 0) {
        s[row] = sc;
        if (ASYM) z[row] = zp;
    }
    const float rc = __fdiv_rn(1.0f, sc);
    const int zoff = zp - (int)kMagicBits;
    void* qr = static_cast<uint8_t*>(q) + row * cols * (H ? 2 : 1);
    uint16_t* q16r = DUAL ? q16 + row * cols : nullptr;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int64_t i = threadIdx.x + (int64_t)j * blockDim.x;
        if (i < n4) store_codes4_exact<ASYM, H, DUAL>(qr, i, v[j], sc, rc, zoff, q16r);
    }
}

// Rows longer than the register budget: reduce in one sweep, code in a second
// sweep (the second read of the row is served mostly by L2).
template <bool ASYM, bool H = false>
__global__ void __launch_bounds__(1024) quantize_long_rows_kernel(const float* __restrict__ x, int64_t cols,
                                                                 void* __restrict__ q,
                                                                 float* __restrict__ s,
                                                                 int32_t* __restrict__ z) {
    __shared__ float red[64];
    const int64_t row = blockIdx.x;
    const int64_t n4 = cols / 4;
    const float4* xr = reinterpret_cast<const float4*>(x + row * cols);
    float hi = 0.0f, nlo = 0.0f;
    for (int64_t i = threadIdx.x; i < n4; i += blockDim.x) {
        float4 v = xr[i];
        if (ASYM) {
            hi = fmaxf(hi, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
            nlo = fmaxf(nlo, -fminf(fminf(v.x, v.y), fminf(v.z, v.w)));
        } else {
            hi = fmaxf(hi, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
    }
    block_max2<ASYM>(hi, nlo, red);
    float sc;
    int zp = 0;
    if (ASYM) {
        asym_params(-nlo, hi, &sc, &zp);
    } else {
        sc = sym_scale(hi);
    }
    if (threadIdx.x == 0) {
        s[row] = sc;
        if (ASYM) z[row] = zp;
    }
    const float rc = __fdiv_rn(1.0f, sc);
    const int zoff = zp - (int)kMagicBits;
    void* qr = static_cast<uint8_t*>(q) + row * cols * (H ? 2 : 1);
    for (int64_t i = threadIdx.x; i < n4; i += blockDim.x) {
        const float4 v = __ldcs(xr + i);
        float dmax = 0.0f;
        store_codes4_tracked<ASYM, H>(qr, i, v, rc, zoff, dmax);
        if (dmax >= kNearHalf) store_codes4_exact<ASYM, H>(qr, i, v, sc, rc, zoff);
    }
}

// Per-tensor range: every block reduces its share and folds it into the cells
// with an integer atomic max on the fp32 bit pattern (non-negative floats
// order like their bits, so the result does not depend on block order).
// cell_hi holds max|x| (symmetric) or max(max x, 0); cell_nlo holds -min(min x, 0).
template <bool ASYM>
__global__ void __launch_bounds__(512) tensor_range_kernel(const float* __restrict__ x, int64_t n4,
                                                           unsigned int* cell_hi,
                                                           unsigned int* cell_nlo) {
    __shared__ float red[64];
    const float4* x4 = reinterpret_cast<const float4*>(x);
    float hi = 0.0f, nlo = 0.0f;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4;
         i += (int64_t)gridDim.x * blockDim.x) {
        float4 v = x4[i];
        if (ASYM) {
            hi = fmaxf(hi, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
            nlo = fmaxf(nlo, -fminf(fminf(v.x, v.y), fminf(v.z, v.w)));
        } else {
            hi = fmaxf(hi, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
    }
    block_max2<ASYM>(hi, nlo, red);
    if (threadIdx.x == 0) {
        atomicMax(cell_hi, __float_as_uint(hi));
        if (ASYM) atomicMax(cell_nlo, __float_as_uint(nlo));
    }
}

// Turns the reduced range in the cells into the tensor's scale (and zero point),
// written over the same cells.
template <bool ASYM>
__global__ void tensor_params_kernel(float* s, int32_t* z) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    const float hi = __uint_as_float(*reinterpret_cast<unsigned int*>(s));
    if (ASYM) {
        const float nlo = __uint_as_float(*reinterpret_cast<unsigned int*>(z));
        float sc;
        int zp;
        asym_params(-nlo, hi, &sc, &zp);
        s[0] = sc;
        z[0] = zp;
    } else {
        s[0] = sym_scale(hi);
    }
}

template <bool ASYM, bool H = false>
__global__ void __launch_bounds__(512) tensor_codes_kernel(const float* __restrict__ x, int64_t n4,
                                                           const float* __restrict__ s,
                                                           const int32_t* __restrict__ z,
                                                           void* __restrict__ q) {
    const float sc = s[0];
    const float rc = __fdiv_rn(1.0f, sc);
    const int zoff = (ASYM ? z[0] : 0) - (int)kMagicBits;
    const float4* x4 = reinterpret_cast<const float4*>(x);
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float4 v = __ldcs(x4 + i);
        float dmax = 0.0f;
        store_codes4_tracked<ASYM, H>(q, i, v, rc, zoff, dmax);
        if (dmax >= kNearHalf) store_codes4_exact<ASYM, H>(q, i, v, sc, rc, zoff);
    }
}

// A small tensor (per-tensor granularity) in one CTA: the range over all elements (block maximum,
// the same values as the grid-wide range kernel's), the scale (and zero point) computed by every
// thread from it, then the codes with the tensor's second read served by L1 / L2. The same
// operations as the three-kernel path, without its two memsets and three launches.
template <bool ASYM, bool H>
__global__ void __launch_bounds__(1024) tensor_small_kernel(const float* __restrict__ x, int64_t n4,
                                                            float* __restrict__ s, int32_t* __restrict__ z,
                                                            void* __restrict__ q) {
    __shared__ float red[64];
    const float4* x4 = reinterpret_cast<const float4*>(x);
    float hi = 0.0f, nlo = 0.0f;
    for (int64_t i = threadIdx.x; i < n4; i += blockDim.x) {
        const float4 v = x4[i];
        if (ASYM) {
            hi = fmaxf(hi, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
            nlo = fmaxf(nlo, -fminf(fminf(v.x, v.y), fminf(v.z, v.w)));
        } else {
            hi = fmaxf(hi, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
    }
    block_max2<ASYM>(hi, nlo, red);
    float sc;
    int zp = 0;
    if (ASYM) {
        asym_params(-nlo, hi, &sc, &zp);
    } else {
        sc = sym_scale(hi);
    }
    if (threadIdx.x == 0) {
        s[0] = sc;
        if (ASYM) z[0] = zp;
    }
    const float rc = __fdiv_rn(1.0f, sc);
    const int zoff = zp - (int)kMagicBits;
    for (int64_t i = threadIdx.x; i < n4; i += blockDim.x) {
        const float4 v = x4[i];
        float dmax = 0.0f;
        store_codes4_tracked<ASYM, H>(q, i, v, rc, zoff, dmax);
        if (dmax >= kNearHalf) store_codes4_exact<ASYM, H>(q, i, v, sc, rc, zoff);
    }
}

// colsum[n] = sum_k qw[n][k]: one warp per weight row, 16-byte loads, dp4a
// against ones (four signed bytes summed into an int32 per instruction).
__global__ void __launch_bounds__(256) colsum_kernel(const int8_t* __restrict__ qw, int64_t N,
                                                     int64_t K, int32_t* __restrict__ colsum) {
    const int64_t n = blockIdx.x * (int64_t)(blockDim.x / kWarp) + threadIdx.x / kWarp;
    const int lane = threadIdx.x % kWarp;
    if (n >= N) return;
    const int4* r = reinterpret_cast<const int4*>(qw + n * K);
    const int64_t n16 = K / 16;
    int acc = 0;
    for (int64_t i = lane; i < n16; i += kWarp) {
        int4 v = r[i];
        acc = __dp4a(v.x, 0x01010101, acc);
        acc = __dp4a(v.y, 0x01010101, acc);
        acc = __dp4a(v.z, 0x01010101, acc);
        acc = __dp4a(v.w, 0x01010101, acc);
    }
#pragma unroll
    for (int o = kWarp / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) colsum[n] = acc;
}

// ------------------------------------------------------------------ fused RMSNorm + quantize
// rms = sqrt(mean(x * x) + eps), y = x / rms * gamma, then the per-token symmetric quantizer
// on y. The sum of squares is the exact sum rounded once to fp32: every square is split into
// its fp32 product and the exact remainder (one FMA), and the running sums are kept as
// unevaluated pairs (hi, lo) combined with TwoSum (Knuth), about twice fp32's precision, so
// the single final rounding fl(hi + lo) is the exactly rounded sum unless that sum lies
// within ~2^-40 of an fp32 rounding midpoint (where either neighbour is a correct rounding).

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

__device__ __forceinline__ void pair_add(float& hi, float& lo, float h2, float l2) {
    float s, e;
    two_sum(hi, h2, s, e);
    hi = s;
    lo = __fadd_rn(lo, __fadd_rn(l2, e));
}

// hi + lo += v * v for a running pair of non-negative parts: the square is split into its fp32
// product and the exact remainder (one FMA), and the product is added by Fast2Sum (Dekker 1971)
// on the larger and the smaller operand (both >= 0), whose error term is exact.
__device__ __forceinline__ void pair_add_square(float& hi, float& lo, float v) {
    const float p = __fmul_rn(v, v);
    const float e = __fmaf_rn(v, v, -p);   // v * v == p + e exactly
    const float a = fmaxf(hi, p), b = fminf(hi, p);
    const float s = __fadd_rn(a, b);
    hi = s;
    lo = __fadd_rn(lo, __fadd_rn(__fsub_rn(b, __fsub_rn(s, a)), e));
}

// Block-wide sum of the pairs; every thread receives lane 0's fl(hi + lo), so the whole
// row uses the same bits (lanes of a butterfly may differ in the last bit of lo).
__device__ __forceinline__ float block_sum_pairs(float hi, float lo, float* red) {
#pragma unroll
    for (int o = kWarp / 2; o > 0; o >>= 1)
        pair_add(hi, lo, __shfl_xor_sync(0xffffffffu, hi, o), __shfl_xor_sync(0xffffffffu, lo, o));
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int nwarps = blockDim.x / kWarp;
    hi = __shfl_sync(0xffffffffu, hi, 0);
    lo = __shfl_sync(0xffffffffu, lo, 0);
    if (lane == 0) {
        red[warp] = hi;
        red[32 + warp] = lo;
    }
    __syncthreads();
    hi = lane < nwarps ? red[lane] : 0.0f;
    lo = lane < nwarps ? red[32 + lane] : 0.0f;
#pragma unroll
    for (int o = kWarp / 2; o > 0; o >>= 1)
        pair_add(hi, lo, __shfl_xor_sync(0xffffffffu, hi, o), __shfl_xor_sync(0xffffffffu, lo, o));
    return __shfl_sync(0xffffffffu, __fadd_rn(hi, lo), 0);
}

__device__ __forceinline__ float rms_of(float sumsq, int64_t cols, float eps) {
    const float mean = __fdiv_rn(sumsq, (float)cols);
    return __fsqrt_rn(__fadd_rn(mean, eps));
}

// RN(x / d) from r = RN(1 / d) by Markstein's correction (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Develop. 34(1), 1990): with
// q0 = RN(x r), the remainder x - q0 d is formed in one FMA and q1 = RN(q0 + (x - q0 d) r). q1 is
// the correctly rounded quotient for every pair of significands: checked against CUDA's IEEE
// division over all 2^23 x 2^23 pairs x, d in [1, 2). Scaling x or d by a power of two scales
// every intermediate exactly while all of them stay normal, so the check covers every x and d
// for which they do: d in [2^-60, 2^60] and |x| >= 2^-60 (x / d, the remainder and the
// correction are then normal); the caller checks both. x = -0 gives +0 (IEEE: -0); the sign of
// a zero y changes neither the row maximum nor its code.
constexpr uint32_t kDivTinyBits = 0x21800000u;   // 2^-60
__device__ __forceinline__ float div_markstein(float x, float d, float r) {
    const float q0 = __fmul_rn(x, r);
    return __fmaf_rn(__fmaf_rn(-q0, d, x), r, q0);
}

// The row's normaliser: rms, its reciprocal and whether Markstein's quotient applies to the row.
struct RowNorm {
    float rms, rr;
    bool fast;
    __device__ __forceinline__ explicit RowNorm(float rms_) : rms(rms_) {
        fast = rms_ >= 0x1p-60f && rms_ <= 0x1p60f;
        rr = __fdiv_rn(1.0f, rms_);
    }
    // y = RN(RN(x / rms) * g): the quotient by Markstein's correction where it is exact, else IEEE.
    __device__ __forceinline__ float operator()(float x, float g) const {
        const uint32_t ax = __float_as_uint(x) & 0x7FFFFFFFu;
        const float q = (fast && ax - 1u >= kDivTinyBits - 1u) ? div_markstein(x, rms, rr) : __fdiv_rn(x, rms);
        return __fmul_rn(q, g);
    }
};

// The IEEE quotient out of line, for paths that are rarely taken (keeps the registers of an
// inlined division sequence out of the callers' main paths).
__device__ __noinline__ float fdiv_rare(float a, float b) { return __fdiv_rn(a, b); }

// The codes of a thread's elements i = t, t + stride, ... (< n4) on the exact path, y recomputed
// from x with the same operations as the kernel's (Markstein's quotient when fast, else IEEE).
// Out of line: it runs only for a thread with a quotient near a half-integer, and keeps its
// registers out of the kernel's main path.
__device__ __noinline__ void rmsnorm_codes_exact(const float4* __restrict__ xr, const float4* __restrict__ g4,
                                                 uint32_t* __restrict__ qr, int64_t t, int64_t stride, int64_t n4,
                                                 float rms, float rr, bool fast, float sc, float rc) {
    for (int64_t i = t; i < n4; i += stride) {
        const float4 a = xr[i], g = __ldg(g4 + i);
        float4 y;
        if (fast)
            y = make_float4(__fmul_rn(div_markstein(a.x, rms, rr), g.x), __fmul_rn(div_markstein(a.y, rms, rr), g.y),
                            __fmul_rn(div_markstein(a.z, rms, rr), g.z), __fmul_rn(div_markstein(a.w, rms, rr), g.w));
        else
            y = make_float4(__fmul_rn(__fdiv_rn(a.x, rms), g.x), __fmul_rn(__fdiv_rn(a.y, rms), g.y),
                            __fmul_rn(__fdiv_rn(a.z, rms), g.z), __fmul_rn(__fdiv_rn(a.w, rms), g.w));
        qr[i] = pack4(sym_code(y.x, sc, rc), sym_code(y.y, sc, rc), sym_code(y.z, sc, rc), sym_code(y.w, sc, rc));
    }
}

// One CTA per row, the row in registers (VPT float4 per thread): one HBM read of x. Up to
// four float4 per thread the kernel fits 32 registers, so two 1024-thread CTAs share an SM
// (the row phases - load, reduce, normalise, reduce, store - of one CTA overlap the other's).
// Per element: the exact square sum (Fast2Sum pair), Markstein's quotient, the gamma product,
// the row maximum and the code by the kMagic FMA, with no per-element branch (elements below
// 2^-60 and quotients near a half-integer are flagged per thread, and that thread takes the
// exact path). The block reductions are cheap for the many warps: every thread stores its pair
// (or its maximum) to shared memory and one warp reduces them and computes the row's scalars
// (rms and its reciprocal; the scale and its reciprocal) once, for all threads to read.
template <int VPT>
__global__ void __launch_bounds__(1024, (VPT <= 4 ? 2 : 1))
    rmsnorm_quantize_rows_kernel(const float* __restrict__ x, const float* __restrict__ gamma, int64_t cols,
                                 float eps, int8_t* __restrict__ q, float* __restrict__ s) {
    __shared__ float2 part[1024];
    __shared__ float wmax[32];
    __shared__ float bc[4];   // rms, 1 / rms, s, 1 / s
    const int64_t row = blockIdx.x;
    const int64_t n4 = cols / 4;
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int nthreads = blockDim.x;
    const float4* xr = reinterpret_cast<const float4*>(x + row * cols);
    const float4* g4 = reinterpret_cast<const float4*>(gamma);
    float4 v[VPT];
    float h0 = 0.0f, l0 = 0.0f;
    uint32_t tmin = 0xFFFFFFFFu;   // min over the thread's elements of 2 |x|bits - 2 (zeros: huge)
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int64_t i = threadIdx.x + (int64_t)j * nthreads;
        if (i < n4) {
            v[j] = __ldcs(xr + i);
            pair_add_square(h0, l0, v[j].x);
            pair_add_square(h0, l0, v[j].y);
            pair_add_square(h0, l0, v[j].z);
            pair_add_square(h0, l0, v[j].w);
            tmin = min(min(tmin, (__float_as_uint(v[j].x) << 1) - 2u), (__float_as_uint(v[j].y) << 1) - 2u);
            tmin = min(min(tmin, (__float_as_uint(v[j].z) << 1) - 2u), (__float_as_uint(v[j].w) << 1) - 2u);
        }
    }
    part[threadIdx.x] = make_float2(h0, l0);
    __syncthreads();
    if (warp == 0) {
        float hi = 0.0f, lo = 0.0f;
        for (int t = lane; t < nthreads; t += kWarp) {
            const float2 pr = part[t];
            pair_add(hi, lo, pr.x, pr.y);
        }
#pragma unroll
        for (int o = kWarp / 2; o > 0; o >>= 1)
            pair_add(hi, lo, __shfl_xor_sync(0xffffffffu, hi, o), __shfl_xor_sync(0xffffffffu, lo, o));
        if (lane == 0) {
            // lane 0's pair (lanes of a butterfly may differ in the last bit of lo)
            const float rms = rms_of(__fadd_rn(hi, lo), cols, eps);
            bc[0] = rms;
            bc[1] = __fdiv_rn(1.0f, rms);
        }
    }
    __syncthreads();
    const float rms = bc[0], rr = bc[1];
    // y = RN(RN(x / rms) * g): Markstein's quotient where it is exact, else the IEEE quotient
    const bool fast = rms >= 0x1p-60f && rms <= 0x1p60f && tmin >= 2u * kDivTinyBits - 2u;
    float amax = 0.0f;
    if (fast) {
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int64_t i = threadIdx.x + (int64_t)j * nthreads;
            if (i < n4) {
                const float4 g = __ldg(g4 + i);
                v[j] = make_float4(__fmul_rn(div_markstein(v[j].x, rms, rr), g.x),
                                   __fmul_rn(div_markstein(v[j].y, rms, rr), g.y),
                                   __fmul_rn(div_markstein(v[j].z, rms, rr), g.z),
                                   __fmul_rn(div_markstein(v[j].w, rms, rr), g.w));
                amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[j].x), fabsf(v[j].y)), fmaxf(fabsf(v[j].z), fabsf(v[j].w))));
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int64_t i = threadIdx.x + (int64_t)j * nthreads;
            if (i < n4) {
                const float4 g = __ldg(g4 + i);
                v[j] = make_float4(__fmul_rn(fdiv_rare(v[j].x, rms), g.x), __fmul_rn(fdiv_rare(v[j].y, rms), g.y),
                                   __fmul_rn(fdiv_rare(v[j].z, rms), g.z), __fmul_rn(fdiv_rare(v[j].w, rms), g.w));
                amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[j].x), fabsf(v[j].y)), fmaxf(fabsf(v[j].z), fabsf(v[j].w))));
            }
        }
    }
#pragma unroll
    for (int o = kWarp / 2; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) wmax[warp] = amax;
    __syncthreads();
    if (warp == 0) {
        float m = lane < nthreads / kWarp ? wmax[lane] : 0.0f;
#pragma unroll
        for (int o = kWarp / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) {
            const float sc = sym_scale(m);
            s[row] = sc;
            bc[2] = sc;
            bc[3] = __fdiv_rn(1.0f, sc);
        }
    }
    __syncthreads();
    const float sc = bc[2], rc = bc[3];
    uint32_t* qr = reinterpret_cast<uint32_t*>(q + row * cols);
    float dmax = 0.0f;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int64_t i = threadIdx.x + (int64_t)j * nthreads;
        if (i < n4) qr[i] = sym_codes4_tracked(v[j], rc, dmax);
    }
    if (dmax >= kNearHalf)   // some quotient near a half-integer (rare): this thread's codes exactly
        rmsnorm_codes_exact(xr, g4, qr, threadIdx.x, nthreads, n4, rms, rr, fast, sc, rc);
}

// Rows longer than the register budget: three sweeps (sum of squares; y and its maximum;
// codes), the later ones served mostly from L2.
__global__ void __launch_bounds__(1024)
    rmsnorm_quantize_long_rows_kernel(const float* __restrict__ x, const float* __restrict__ gamma,
                                      int64_t cols, float eps, int8_t* __restrict__ q, float* __restrict__ s) {
    __shared__ float red[64];
    __shared__ float red2[64];
    const int64_t row = blockIdx.x;
    const int64_t n4 = cols / 4;
    const float4* xr = reinterpret_cast<const float4*>(x + row * cols);
    const float4* g4 = reinterpret_cast<const float4*>(gamma);
    float hi = 0.0f, lo = 0.0f;
    for (int64_t i = threadIdx.x; i < n4; i += blockDim.x) {
        const float4 v = xr[i];
        pair_add_square(hi, lo, v.x);
        pair_add_square(hi, lo, v.y);
        pair_add_square(hi, lo, v.z);
        pair_add_square(hi, lo, v.w);
    }
    const RowNorm nrm(rms_of(block_sum_pairs(hi, lo, red), cols, eps));
    float amax = 0.0f, unused = 0.0f;
    for (int64_t i = threadIdx.x; i < n4; i += blockDim.x) {
        const float4 v = xr[i];
        const float4 g = __ldg(g4 + i);
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(nrm(v.x, g.x)), fabsf(nrm(v.y, g.y))),
                                 fmaxf(fabsf(nrm(v.z, g.z)), fabsf(nrm(v.w, g.w)))));
    }
    block_max2<false>(amax, unused, red2);
    const float sc = sym_scale(amax);
    if (threadIdx.x == 0) s[row] = sc;
    const float rc = __fdiv_rn(1.0f, sc);
    uint32_t* qr = reinterpret_cast<uint32_t*>(q + row * cols);
    for (int64_t i = threadIdx.x; i < n4; i += blockDim.x) {
        const float4 v = __ldcs(xr + i);
        const float4 g = __ldg(g4 + i);
        qr[i] = pack4(sym_code(nrm(v.x, g.x), sc, rc), sym_code(nrm(v.y, g.y), sc, rc),
                      sym_code(nrm(v.z, g.z), sc, rc), sym_code(nrm(v.w, g.w), sc, rc));
    }
}

// Streaming form for rows of up to 1024 * VPT float4 whose three copies fit in shared memory
// (K <= 16384): a persistent grid of one 1024-thread CTA per SM takes rows blockIdx.x,
// blockIdx.x + grid, ...; each row arrives in one of three shared-memory buffers by one bulk copy
// (cp.async.bulk, completing on that buffer's mbarrier), issued three rows ahead, so the SM's HBM
// stream continues through the block reductions of the row it is working on. The row is read
// into registers (VPT float4 per thread), then: the exact square sum (Fast2Sum pair), Markstein's
// quotient, the gamma product, the row maximum and the codes by the kMagic FMA, with no
// per-element branch (elements below 2^-60 in magnitude and quotients near a half-integer are
// flagged per thread and that thread takes the exact path).
// Block reductions of the streaming kernel: every warp reduces its lanes by a butterfly and one
// lane per warp stores the result; after a barrier warp 0 alone reduces the warps' results and
// computes the row's scalars from them, which it stores for all threads to read after a second
// barrier (the other warps spend no issue slots on the second level or the scalar math).
// bc[0], bc[1]: rms and RN(1 / rms); bc[2], bc[3]: the row's scale s and RN(1 / s).
// Returns whether `ok` holds in every thread (the vote rides on the first barrier); the row's
// scalars are computed only when it does.
__device__ __forceinline__ bool stream_sum_to_rms(float hi, float lo, bool ok, float2* red, float* bc, int64_t cols,
                                                  float eps) {
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
#pragma unroll
    for (int o = kWarp / 2; o > 0; o >>= 1)
        pair_add(hi, lo, __shfl_xor_sync(0xffffffffu, hi, o), __shfl_xor_sync(0xffffffffu, lo, o));
    if (lane == 0) red[warp] = make_float2(hi, lo);
    if (!__syncthreads_and(ok)) return false;
    if (warp == 0) {
        const float2 pr = lane < (int)(blockDim.x / kWarp) ? red[lane] : make_float2(0.0f, 0.0f);
        hi = pr.x;
        lo = pr.y;
#pragma unroll
        for (int o = kWarp / 2; o > 0; o >>= 1)
            pair_add(hi, lo, __shfl_xor_sync(0xffffffffu, hi, o), __shfl_xor_sync(0xffffffffu, lo, o));
        if (lane == 0) {   // lane 0's pair (lanes of a butterfly may differ in the last bit of lo)
            const float rms = rms_of(__fadd_rn(hi, lo), cols, eps);
            bc[0] = rms;
            bc[1] = __fdiv_rn(1.0f, rms);
        }
    }
    __syncthreads();
    return true;
}

__device__ __forceinline__ void stream_max_to_scale(float amax, float* red, float* bc) {
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
#pragma unroll
    for (int o = kWarp / 2; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) red[warp] = amax;
    __syncthreads();
    if (warp == 0) {
        float m = lane < (int)(blockDim.x / kWarp) ? red[lane] : 0.0f;
#pragma unroll
        for (int o = kWarp / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) {
            const float sc = sym_scale(m);
            bc[2] = sc;
            bc[3] = __fdiv_rn(1.0f, sc);
        }
    }
    __syncthreads();
}

constexpr int kStreamThreads = 1024;
constexpr int kStreamBufs = 3;
int num_sms();

__device__ __forceinline__ void bulk_row_load(uint32_t dst, const float* src, uint32_t bytes, uint32_t bar) {
    tc::mbar_expect_tx(bar, bytes);
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// THREADS threads per CTA, VPT float4 per thread; FULL: every row is exactly VPT * THREADS float4
// (no bounds checks). With THREADS <= 512 each thread keeps its gamma float4s in registers for all
// its rows (the persistent grid gives a thread the same columns in every row).
template <int VPT, int THREADS, bool FULL>
__global__ void __launch_bounds__(THREADS, 1)
    rmsnorm_quantize_stream_kernel(const float* __restrict__ x, const float* __restrict__ gamma, int64_t rows,
                                   int64_t cols, float eps, int8_t* __restrict__ q, float* __restrict__ s) {
    constexpr bool kGammaRegs = THREADS <= 512 && VPT <= 8;
    extern __shared__ __align__(128) uint8_t rowbuf[];
    __shared__ __align__(8) uint64_t bar_cells[kStreamBufs];
    __shared__ float2 red[32];
    __shared__ float red2[32];
    __shared__ float bc[4];
    __shared__ int abort_cell;
    const uint32_t bytes = (uint32_t)(cols * 4);
    const int n4 = (int)(cols / 4);
    const float4* g4 = reinterpret_cast<const float4*>(gamma);
    volatile int* abort_flag = &abort_cell;
    auto live = [&](int j) { return FULL || (int)threadIdx.x + j * THREADS < n4; };
    float4 gv[kGammaRegs ? VPT : 1];
    if constexpr (kGammaRegs) {
#pragma unroll
        for (int j = 0; j < VPT; ++j)
            gv[j] = live(j) ? __ldg(g4 + threadIdx.x + j * THREADS) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
    if (threadIdx.x == 0) {
        for (int b = 0; b < kStreamBufs; ++b) tc::mbar_init(tc::smem_u32(&bar_cells[b]), 1);
        abort_cell = 0;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int b = 0; b < kStreamBufs; ++b) {
            const int64_t r = blockIdx.x + (int64_t)b * gridDim.x;
            if (r < rows)
                bulk_row_load(tc::smem_u32(rowbuf) + b * bytes, x + r * cols, bytes, tc::smem_u32(&bar_cells[b]));
        }
    }
    int64_t row = blockIdx.x;
    for (uint32_t it = 0; row < rows; row += gridDim.x, ++it) {
        const uint32_t b = it % kStreamBufs;
        const uint32_t buf = tc::smem_u32(rowbuf) + b * bytes;
        // every thread waits for the copy itself (bounded); the block votes on the outcome at the
        // first reduction's barrier and leaves together if any thread's wait gave up (a thread
        // whose wait gave up sums stale shared memory, which the vote then discards)
        const bool arrived = tc::mbar_wait(tc::smem_u32(&bar_cells[b]), (it / kStreamBufs) & 1u, abort_flag, 0x80u,
                                           &g_quant_error);
        float4 v[VPT];
        float hi = 0.0f, lo = 0.0f;
        uint32_t tmin = 0xFFFFFFFFu;   // min over the thread's elements of 2 |x|bits - 2 (zeros: huge)
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            if (live(j)) {
                const uint4 r = tc::lds128(buf + 16u * (threadIdx.x + (uint32_t)(j * THREADS)));
                v[j] = make_float4(__uint_as_float(r.x), __uint_as_float(r.y), __uint_as_float(r.z), __uint_as_float(r.w));
                pair_add_square(hi, lo, v[j].x);
                pair_add_square(hi, lo, v[j].y);
                pair_add_square(hi, lo, v[j].z);
                pair_add_square(hi, lo, v[j].w);
                tmin = min(min(tmin, (__float_as_uint(v[j].x) << 1) - 2u), (__float_as_uint(v[j].y) << 1) - 2u);
                tmin = min(min(tmin, (__float_as_uint(v[j].z) << 1) - 2u), (__float_as_uint(v[j].w) << 1) - 2u);
            }
        }
        if (!stream_sum_to_rms(hi, lo, arrived, red, bc, cols, eps)) break;
        // every thread has summed its values from buffer b: it takes the row kStreamBufs ahead
        const int64_t ahead = row + (int64_t)kStreamBufs * gridDim.x;
        if (threadIdx.x == 0 && ahead < rows) {
            tc::fence_proxy_async_smem();
            bulk_row_load(buf, x + ahead * cols, bytes, tc::smem_u32(&bar_cells[b]));
        }
        const float rms = bc[0], rr = bc[1];
        const bool fast = rms >= 0x1p-60f && rms <= 0x1p60f && tmin >= 2u * kDivTinyBits - 2u;
        float amax = 0.0f;
        auto gamma_of = [&](int j) { return kGammaRegs ? gv[kGammaRegs ? j : 0] : __ldg(g4 + threadIdx.x + j * THREADS); };
        if (fast) {
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                if (live(j)) {
                    const float4 g = gamma_of(j);
                    v[j] = make_float4(__fmul_rn(div_markstein(v[j].x, rms, rr), g.x),
                                       __fmul_rn(div_markstein(v[j].y, rms, rr), g.y),
                                       __fmul_rn(div_markstein(v[j].z, rms, rr), g.z),
                                       __fmul_rn(div_markstein(v[j].w, rms, rr), g.w));
                    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[j].x), fabsf(v[j].y)), fmaxf(fabsf(v[j].z), fabsf(v[j].w))));
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                if (live(j)) {
                    const float4 g = gamma_of(j);
                    v[j] = make_float4(__fmul_rn(__fdiv_rn(v[j].x, rms), g.x), __fmul_rn(__fdiv_rn(v[j].y, rms), g.y),
                                       __fmul_rn(__fdiv_rn(v[j].z, rms), g.z), __fmul_rn(__fdiv_rn(v[j].w, rms), g.w));
                    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[j].x), fabsf(v[j].y)), fmaxf(fabsf(v[j].z), fabsf(v[j].w))));
                }
            }
        }
        stream_max_to_scale(amax, red2, bc);
        const float sc = bc[2], rc = bc[3];
        if (threadIdx.x == 0) s[row] = sc;
        uint32_t* qr = reinterpret_cast<uint32_t*>(q + row * cols);
        float dmax = 0.0f;
#pragma unroll
        for (int j = 0; j < VPT; ++j)
            if (live(j)) qr[threadIdx.x + j * THREADS] = sym_codes4_tracked(v[j], rc, dmax);
        if (dmax >= kNearHalf) {   // some quotient near a half-integer (rare): this thread's codes exactly
#pragma unroll
            for (int j = 0; j < VPT; ++j)
                if (live(j))
                    qr[threadIdx.x + j * THREADS] = pack4(sym_code(v[j].x, sc, rc), sym_code(v[j].y, sc, rc),
                                                          sym_code(v[j].z, sc, rc), sym_code(v[j].w, sc, rc));
        }
        // (the reductions' shared cells: red is written again by the next row before its first
        // barrier, after every thread has passed this row's second barrier, which follows the
        // last read of red; red2 and bc likewise after the next row's barriers)
    }
    if (*abort_flag) {   // a row copy did not arrive: give copies in flight a bounded time to land
        const long long t0 = clock64();
        while (clock64() - t0 < (1LL << 22)) __nanosleep(1000);
    }
}

template <int VPT, int THREADS, bool FULL>
cudaError_t launch_rms_stream(const float* x, const float* gamma, int64_t rows, int64_t cols, float eps, int8_t* q,
                              float* s, cudaStream_t st) {
    const int smem = (int)(cols * 4) * kStreamBufs;
    auto kern = rmsnorm_quantize_stream_kernel<VPT, THREADS, FULL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int64_t cap = num_sms();
    const unsigned grid = (unsigned)(rows < cap ? rows : cap);
    kern<<<grid, THREADS, smem, st>>>(x, gamma, rows, cols, eps, q, s);
    note_launch();
    return cudaGetLastError();
}

template <int VPT>
cudaError_t launch_rms_rows(const float* x, const float* gamma, int64_t rows, int64_t cols, float eps, int threads,
                            int8_t* q, float* s, cudaStream_t st) {
    rmsnorm_quantize_rows_kernel<VPT><<<(unsigned)rows, threads, 0, st>>>(x, gamma, cols, eps, q, s);
    note_launch();
    return cudaGetLastError();
}

// ------------------------------------------------------------------ int4 weights (W4A8)
// Per-row symmetric int4 codes: s = max(absmax, 1e-8) / 7, q = clamp(rint(w / s), -8, 7),
// two codes per byte along the row, low nibble first ((q0 & 0xF) | (q1 & 0xF) << 4).
__device__ __forceinline__ uint32_t int4_code(float x, float s) {
    return (uint32_t)clampi(__float2int_rn(__fdiv_rn(x, s)), -8, 7) & 0xFu;
}

template <int VPT>
__global__ void __launch_bounds__(1024, (VPT <= 4 ? 2 : 1))
    quantize_int4_rows_kernel(const float* __restrict__ w, int64_t cols, uint8_t* __restrict__ q,
                              float* __restrict__ s) {
    __shared__ float red[64];
    const int64_t row = blockIdx.x;
    const int64_t n4 = cols / 4;
    const float4* wr = reinterpret_cast<const float4*>(w + row * cols);
    float4 v[VPT];
    float hi = 0.0f, unused = 0.0f;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int64_t i = threadIdx.x + (int64_t)j * blockDim.x;
        if (i < n4) {
            v[j] = wr[i];
            hi = fmaxf(hi, fmaxf(fmaxf(fabsf(v[j].x), fabsf(v[j].y)), fmaxf(fabsf(v[j].z), fabsf(v[j].w))));
        }
    }
    block_max2<false>(hi, unused, red);
    const float sc = __fdiv_rn(fmaxf(hi, kZeroGuard), 7.0f);
    if (threadIdx.x == 0) s[row] = sc;
    uint16_t* qr = reinterpret_cast<uint16_t*>(q + row * (cols / 2));
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int64_t i = threadIdx.x + (int64_t)j * blockDim.x;
        if (i < n4)
            qr[i] = (uint16_t)(int4_code(v[j].x, sc) | (int4_code(v[j].y, sc) << 4) | (int4_code(v[j].z, sc) << 8) |
                               (int4_code(v[j].w, sc) << 12));
    }
}

// Rows longer than the register budget: range sweep, then code sweep.
__global__ void __launch_bounds__(1024) quantize_int4_long_rows_kernel(const float* __restrict__ w, int64_t cols,
                                                                     uint8_t* __restrict__ q,
                                                                     float* __restrict__ s) {
    __shared__ float red[64];
    const int64_t row = blockIdx.x;
    const int64_t n4 = cols / 4;
    const float4* wr = reinterpret_cast<const float4*>(w + row * cols);
    float hi = 0.0f, unused = 0.0f;
    for (int64_t i = threadIdx.x; i < n4; i += blockDim.x) {
        const float4 v = wr[i];
        hi = fmaxf(hi, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    block_max2<false>(hi, unused, red);
    const float sc = __fdiv_rn(fmaxf(hi, kZeroGuard), 7.0f);
    if (threadIdx.x == 0) s[row] = sc;
    uint16_t* qr = reinterpret_cast<uint16_t*>(q + row * (cols / 2));
    for (int64_t i = threadIdx.x; i < n4; i += blockDim.x) {
        const float4 v = wr[i];
        qr[i] = (uint16_t)(int4_code(v.x, sc) | (int4_code(v.y, sc) << 4) | (int4_code(v.z, sc) << 8) |
                           (int4_code(v.w, sc) << 12));
    }
}

// colsum[n] = sum_k q[n][k] over sign-extended nibbles: for the low (or high) nibbles of a
// word, u = nibble value 0..15 in each byte, and (u ^ 8) - 8 is the signed code, so a dp4a of
// (u ^ 8) against ones minus 32 sums the four codes.
__global__ void __launch_bounds__(256) colsum_int4_kernel(const uint8_t* __restrict__ q, int64_t N, int64_t K,
                                                          int32_t* __restrict__ colsum) {
    const int64_t n = blockIdx.x * (int64_t)(blockDim.x / kWarp) + threadIdx.x / kWarp;
    const int lane = threadIdx.x % kWarp;
    if (n >= N) return;
    const uint4* r = reinterpret_cast<const uint4*>(q + n * (K / 2));
    const int64_t n16 = K / 32;
    int acc = 0;
    for (int64_t i = lane; i < n16; i += kWarp) {
        const uint4 v = r[i];
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            acc = __dp4a((int)((w4[t] & 0x0F0F0F0Fu) ^ 0x08080808u), 0x01010101, acc) - 32;
            acc = __dp4a((int)(((w4[t] >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u), 0x01010101, acc) - 32;
        }
    }
#pragma unroll
    for (int o = kWarp / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) colsum[n] = acc;
}

// Block-scaled int8 weights, one warp per (row, group of G K elements). The scale is
// x = amax / 127 rounded up to a power of two as an E8M0 byte: the exponent field of x, plus
// one when its mantissa is not zero, clamped to [kMxEmin, kMxEmax] (2^-24 .. 2^9, where every
// q * s is exact in fp16); s = 2^(e - 127); codes clamp(rint(w / s), -127, 127) with an IEEE
// division (exact for a power of two). Lane 0 writes the scale byte: byte g % 4 of word g / 4
// of the row, words group-major (word w of row n at index w * N + n); the last group of a row
// also zeroes the bytes after it in its word.
__global__ void __launch_bounds__(256) quantize_weight_mx_kernel(const float* __restrict__ w, int64_t N, int64_t K,
                                                                 int G, int8_t* __restrict__ q,
                                                                 uint8_t* __restrict__ sf_bytes) {
    const int64_t groups = K / G;
    const int64_t item = blockIdx.x * (int64_t)(blockDim.x / kWarp) + threadIdx.x / kWarp;
    const int lane = threadIdx.x % kWarp;
    if (item >= N * groups) return;
    const int64_t n = item / groups, g = item - n * groups;
    const float* wg = w + n * K + g * G;
    uint32_t amax_bits = 0;
    for (int k = lane; k < G; k += kWarp) amax_bits = max(amax_bits, __float_as_uint(fabsf(wg[k])));
    amax_bits = __reduce_max_sync(0xffffffffu, amax_bits);
    const uint32_t xb = __float_as_uint(__fdiv_rn(__uint_as_float(amax_bits), 127.0f));
    const int e = min(max((int)(xb >> 23) + ((xb & 0x7FFFFFu) != 0 ? 1 : 0), kMxEmin), kMxEmax);
    const float s = __uint_as_float((uint32_t)e << 23);
    int8_t* qg = q + n * K + g * G;
    for (int k = lane; k < G; k += kWarp) qg[k] = (int8_t)min(max(__float2int_rn(__fdiv_rn(wg[k], s)), -127), 127);
    if (lane == 0) {
        uint8_t* word = sf_bytes + ((g / 4) * N + n) * 4;
        word[g % 4] = (uint8_t)e;
        if (g == groups - 1)
            for (int b = (int)(g % 4) + 1; b < 4; ++b) word[b] = 0;
    }
}

// SM count of the current device, cached per device.
int num_sms() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) dev = 0;
    int* slot = dev < 64 ? &cached[dev] : nullptr;
    if (slot && *slot > 0) return *slot;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
        (void)cudaGetLastError();
        return 1;
    }
    if (slot) *slot = sms;
    return sms;
}

template <int VPT, bool ASYM, bool H, bool DUAL = false>
cudaError_t launch_rows(const float* x, int64_t rows, int64_t cols, int threads, void* q, float* s,
                        int32_t* z, cudaStream_t st, uint16_t* q16 = nullptr) {
    quantize_rows_kernel<VPT, ASYM, H, DUAL><<<(unsigned)rows, threads, 0, st>>>(x, cols, q, s, z, q16);
    note_launch();
    return cudaGetLastError();
}

// Both code formats from one pass (rows held in registers, up to 8 float4 per thread); longer
// rows return cudaErrorNotSupported.
template <bool ASYM>
cudaError_t dispatch_rows_dual(const float* x, int64_t rows, int64_t cols, int8_t* q, uint16_t* q16, float* s,
                               int32_t* z, cudaStream_t st) {
    const int64_t n4 = cols / 4;
    auto threads_for = [&](int vpt) {
        int64_t t = (n4 + vpt - 1) / vpt;
        t = ((t + kWarp - 1) / kWarp) * kWarp;
        return (int)(t < kWarp ? kWarp : t);
    };
    if (n4 <= 256) return launch_rows<1, ASYM, false, true>(x, rows, cols, threads_for(1), q, s, z, st, q16);
    if (n4 <= 1024 * 4) return launch_rows<4, ASYM, false, true>(x, rows, cols, threads_for(4), q, s, z, st, q16);
    if (n4 <= 1024 * 8) return launch_rows<8, ASYM, false, true>(x, rows, cols, threads_for(8), q, s, z, st, q16);
    return cudaErrorNotSupported;
}

template <bool ASYM, bool H>
cudaError_t dispatch_rows(const float* x, int64_t rows, int64_t cols, void* q, float* s, int32_t* z,
                          cudaStream_t st) {
    const int64_t n4 = cols / 4;
    // Smallest block that covers the row with the per-thread register budget.
    auto threads_for = [&](int vpt) {
        int64_t t = (n4 + vpt - 1) / vpt;
        t = ((t + kWarp - 1) / kWarp) * kWarp;
        return (int)(t < kWarp ? kWarp : t);
    };
    // Up to 1024 threads per row and at most 4 float4 per thread keeps the kernel at
    // <= 32 registers, so a full SM of threads stays resident. Rows of more than 256 float4 take
    // four per thread (several independent loads in flight per thread, and for rows up to 1024
    // float4 blocks of at most 256 threads, several rows per SM).
    if (n4 <= 256) return launch_rows<1, ASYM, H>(x, rows, cols, threads_for(1), q, s, z, st);
    if (n4 <= 1024 * 4) return launch_rows<4, ASYM, H>(x, rows, cols, threads_for(4), q, s, z, st);
    if (n4 <= 1024 * 8) return launch_rows<8, ASYM, H>(x, rows, cols, threads_for(8), q, s, z, st);
    quantize_long_rows_kernel<ASYM, H><<<(unsigned)rows, 1024, 0, st>>>(x, cols, q, s, z);
    note_launch();
    return cudaGetLastError();
}

template <bool ASYM, bool H>
cudaError_t dispatch_tensor(const float* x, int64_t n, void* q, float* s, int32_t* z, cudaStream_t st) {
    const int64_t n4 = n / 4;
    if (n4 <= 8192) {   // up to 128 KB of fp32: one CTA, one launch
        tensor_small_kernel<ASYM, H><<<1, 1024, 0, st>>>(x, n4, s, z, q);
        note_launch();
        return cudaGetLastError();
    }
    cudaError_t e = cudaMemsetAsync(s, 0, sizeof(float), st);
    if (e == cudaSuccess && ASYM) e = cudaMemsetAsync(z, 0, sizeof(int32_t), st);
    if (e != cudaSuccess) return e;
    int64_t blocks = (n4 + 511) / 512;
    const int64_t cap = (int64_t)num_sms() * 4;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    tensor_range_kernel<ASYM><<<(unsigned)blocks, 512, 0, st>>>(
        x, n4, reinterpret_cast<unsigned int*>(s), reinterpret_cast<unsigned int*>(z));
    tensor_params_kernel<ASYM><<<1, 32, 0, st>>>(s, z);
    tensor_codes_kernel<ASYM, H><<<(unsigned)blocks, 512, 0, st>>>(x, n4, s, z, q);
    note_launch(3);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize(const float* x, int64_t rows, int64_t cols, bool per_row, int8_t* q,
                            float* s, int32_t* z, cudaStream_t stream) {
    if (per_row) {
        if (rows == 0) return cudaSuccess;
        return z ? dispatch_rows<true, false>(x, rows, cols, q, s, z, stream)
                 : dispatch_rows<false, false>(x, rows, cols, q, s, z, stream);
    }
    return z ? dispatch_tensor<true, false>(x, rows * cols, q, s, z, stream)
             : dispatch_tensor<false, false>(x, rows * cols, q, s, z, stream);
}

cudaError_t launch_quantize_dual(const float* x, int64_t rows, int64_t cols, int8_t* q, uint16_t* q16, float* s,
                                 int32_t* z, cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    return z ? dispatch_rows_dual<true>(x, rows, cols, q, q16, s, z, stream)
             : dispatch_rows_dual<false>(x, rows, cols, q, q16, s, z, stream);
}

cudaError_t launch_quantize_f16(const float* x, int64_t rows, int64_t cols, bool per_row, uint16_t* q,
                                float* s, int32_t* z, cudaStream_t stream) {
    if (per_row) {
        if (rows == 0) return cudaSuccess;
        return z ? dispatch_rows<true, true>(x, rows, cols, q, s, z, stream)
                 : dispatch_rows<false, true>(x, rows, cols, q, s, z, stream);
    }
    return z ? dispatch_tensor<true, true>(x, rows * cols, q, s, z, stream)
             : dispatch_tensor<false, true>(x, rows * cols, q, s, z, stream);
}

cudaError_t launch_rmsnorm_quantize(const float* x, const float* gamma, int64_t rows, int64_t cols, float eps,
                                   int8_t* q, float* s, cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    const int64_t n4 = cols / 4;
    auto threads_for = [&](int vpt) {
        int64_t t = (n4 + vpt - 1) / vpt;
        t = ((t + kWarp - 1) / kWarp) * kWarp;
        return (int)(t < kWarp ? kWarp : t);
    };
    if (n4 <= 256) return launch_rms_rows<1>(x, gamma, rows, cols, eps, threads_for(1), q, s, stream);
    // rows of 1024 .. 16384 elements with many rows: the streaming kernel (three rows in flight
    // per SM through shared memory)
    if (n4 > 256 && n4 <= kStreamThreads * 4 && rows >= 2 * (int64_t)num_sms()) {
        // rows of exactly 16384 elements: 512 threads of eight float4 each, no bounds checks, gamma
        // in registers (fewer warps per row: half the reduction work per element)
        if (n4 == 512 * 8) return launch_rms_stream<8, 512, true>(x, gamma, rows, cols, eps, q, s, stream);
        return launch_rms_stream<4, kStreamThreads, false>(x, gamma, rows, cols, eps, q, s, stream);
    }
    if (n4 <= 1024 * 4) return launch_rms_rows<4>(x, gamma, rows, cols, eps, threads_for(4), q, s, stream);
    if (n4 <= 1024 * 8) return launch_rms_rows<8>(x, gamma, rows, cols, eps, threads_for(8), q, s, stream);
    rmsnorm_quantize_long_rows_kernel<<<(unsigned)rows, 1024, 0, stream>>>(x, gamma, cols, eps, q, s);
    note_launch();
    return cudaGetLastError();
}

// The layer output when K == 0 (every dot product empty, corr = 0): y = fl(0 * scale) + bias[n]
// written in the requested output type.
__global__ void epilogue_fill_kernel(Epilogue ep, int64_t M, int64_t N) {
    const int64_t total = M * N;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x)
        epi_store(ep, i, epi_bias(ep, 0.0f, i % N));
}

cudaError_t launch_epilogue_fill(const Epilogue& ep, int64_t M, int64_t N, cudaStream_t stream) {
    const int64_t total = M * N;
    if (total == 0) return cudaSuccess;
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    epilogue_fill_kernel<<<(unsigned)blocks, 256, 0, stream>>>(ep, M, N);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_quantize_int4(const float* w, int64_t rows, int64_t cols, uint8_t* q, float* s,
                                 cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    const int64_t n4 = cols / 4;
    auto threads_for = [&](int vpt) {
        int64_t t = (n4 + vpt - 1) / vpt;
        t = ((t + kWarp - 1) / kWarp) * kWarp;
        return (int)(t < kWarp ? kWarp : t);
    };
    if (n4 <= 1024 * 1) {
        quantize_int4_rows_kernel<1><<<(unsigned)rows, threads_for(1), 0, stream>>>(w, cols, q, s);
    } else if (n4 <= 1024 * 2) {
        quantize_int4_rows_kernel<2><<<(unsigned)rows, threads_for(2), 0, stream>>>(w, cols, q, s);
    } else if (n4 <= 1024 * 4) {
        quantize_int4_rows_kernel<4><<<(unsigned)rows, threads_for(4), 0, stream>>>(w, cols, q, s);
    } else if (n4 <= 1024 * 8) {
        quantize_int4_rows_kernel<8><<<(unsigned)rows, threads_for(8), 0, stream>>>(w, cols, q, s);
    } else {
        quantize_int4_long_rows_kernel<<<(unsigned)rows, 1024, 0, stream>>>(w, cols, q, s);
    }
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_colsum_int4(const uint8_t* q, int64_t N, int64_t K, int32_t* colsum, cudaStream_t stream) {
    if (N == 0) return cudaSuccess;
    const int warps_per_block = 8;
    const int64_t blocks = (N + warps_per_block - 1) / warps_per_block;
    colsum_int4_kernel<<<(unsigned)blocks, warps_per_block * kWarp, 0, stream>>>(q, N, K, colsum);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_quantize_weight_mx(const float* w, int64_t N, int64_t K, int G, int8_t* q, uint32_t* sf,
                                      cudaStream_t stream) {
    if (N == 0 || K == 0) return cudaSuccess;
    const int warps_per_block = 8;
    const int64_t items = N * (K / G);
    const int64_t blocks = (items + warps_per_block - 1) / warps_per_block;
    if (blocks >= (1LL << 31)) return cudaErrorNotSupported;
    quantize_weight_mx_kernel<<<(unsigned)blocks, warps_per_block * kWarp, 0, stream>>>(
        w, N, K, G, q, reinterpret_cast<uint8_t*>(sf));
    note_launch();
    return cudaGetLastError();
}

// int8 codes -> the fp16 numbers of equal value (exact: |code| <= 128). A word of codes
// (b0, b1, b2, b3) masked to its bytes 0 and 2, with 0x6400 | (byte ^ 0x80) = 1024 + 128 + code as
// fp16, minus 1152, gives the pair (b0, b2), and its bytes 1 and 3 the pair (b1, b3): the codes in
// pair order (0, 2, 1, 3). For K order the bytes are first permuted to (b0, b2, b1, b3). A stream:
// 16 codes in, 32 bytes out per thread step.
__device__ __forceinline__ uint32_t hsub_1152_q(uint32_t v) {
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;\n" : "=r"(r) : "r"(v), "r"(0x64806480u));
    return r;
}
template <bool kPairOrder>
__device__ __forceinline__ uint2 codes4_to_f16(uint32_t w) {
    const uint32_t x = kPairOrder ? w : __byte_perm(w, 0u, 0x3120u);
    return make_uint2(hsub_1152_q((x & 0x00FF00FFu) ^ 0x64806480u), hsub_1152_q(((x >> 8) & 0x00FF00FFu) ^ 0x64806480u));
}

template <bool kPairOrder>
__global__ void __launch_bounds__(256) codes_to_f16_kernel(const uint4* __restrict__ q, int64_t n16,
                                                           uint4* __restrict__ out) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n16; i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 v = __ldcs(q + i);
        const uint2 a = codes4_to_f16<kPairOrder>(v.x), b = codes4_to_f16<kPairOrder>(v.y);
        const uint2 c = codes4_to_f16<kPairOrder>(v.z), d = codes4_to_f16<kPairOrder>(v.w);
        out[2 * i] = make_uint4(a.x, a.y, b.x, b.y);
        out[2 * i + 1] = make_uint4(c.x, c.y, d.x, d.y);
    }
}

cudaError_t launch_codes_to_f16(const int8_t* q, int64_t n, uint16_t* out, cudaStream_t stream, bool pair_order) {
    const int64_t n16 = n / 16;
    if (n16 == 0) return cudaSuccess;
    int64_t blocks = (n16 + 255) / 256;
    const int64_t cap = (int64_t)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    auto kern = pair_order ? codes_to_f16_kernel<true> : codes_to_f16_kernel<false>;
    kern<<<(unsigned)blocks, 256, 0, stream>>>(reinterpret_cast<const uint4*>(q), n16, reinterpret_cast<uint4*>(out));
    note_launch();
    return cudaGetLastError();
}

cudaError_t read_and_clear_quant_error(uint32_t* code) {
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_quant_error, sizeof(v));
    if (e != cudaSuccess) return e;
    *code = v;
    if (v) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_quant_error, &zero, sizeof(zero));
    }
    return e;
}

cudaError_t launch_colsum(const int8_t* qw, int64_t N, int64_t K, int32_t* colsum, cudaStream_t stream) {
    if (N == 0) return cudaSuccess;
    const int warps_per_block = 8;
    const int64_t blocks = (N + warps_per_block - 1) / warps_per_block;
    colsum_kernel<<<(unsigned)blocks, warps_per_block * kWarp, 0, stream>>>(qw, N, K, colsum);
    note_launch();
    return cudaGetLastError();
}

}  // namespace q8
