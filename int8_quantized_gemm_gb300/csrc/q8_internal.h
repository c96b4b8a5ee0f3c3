// Internal declarations shared by the CUDA translation units of the library.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#ifdef __CUDACC__
#include <cuda_bf16.h>
#endif

#include "../../include/q8.h"

namespace q8 {

// Every kernel launch of the library goes through note_launch() so that
// q8_launch_count() can report how many of our kernels ran.
void note_launch(int n = 1);

// Symmetric rule: s = max(amax, 1e-8) / 127; codes clamp(rint(x / s), -127, 127).
// Asymmetric rule: lo = min(min, 0), hi = max(max, 0), s = max(hi - lo, 1e-8) / 255,
// z = clamp(-128 - rint(lo / s), -128, 127), q = clamp(rint(x / s) + z, -128, 127).
constexpr float kZeroGuard = 1e-8f;

// Quantize rows of x (rows x cols, row-major); per_row selects one scale per row
// or one for the whole tensor. z == nullptr selects the symmetric rule.
cudaError_t launch_quantize(const float* x, int64_t rows, int64_t cols, bool per_row,
                            int8_t* q, float* s, int32_t* z, cudaStream_t stream);
// Per-token quantization writing the int8 codes to q and the same codes as fp16 values to q16
// (K order) in one pass; cudaErrorNotSupported for rows longer than 32768 elements.
cudaError_t launch_quantize_dual(const float* x, int64_t rows, int64_t cols, int8_t* q, uint16_t* q16, float* s,
                                 int32_t* z, cudaStream_t stream);
// The same codes written as fp16 values (exact: |code| <= 128), two bytes each.
cudaError_t launch_quantize_f16(const float* x, int64_t rows, int64_t cols, bool per_row,
                                uint16_t* q, float* s, int32_t* z, cudaStream_t stream);

// int8 codes (n elements, n % 16 == 0, both bases 16-byte aligned) as the fp16 numbers of equal
// value, in order, or (pair_order) with each group of four codes stored as codes 0, 2, 1, 3.
cudaError_t launch_codes_to_f16(const int8_t* q, int64_t n, uint16_t* out, cudaStream_t stream,
                                bool pair_order = false);

// int4 weights (W4A8): per-row symmetric codes packed two per byte (K % 32 == 0), and their
// column sums.
cudaError_t launch_quantize_int4(const float* w, int64_t rows, int64_t cols, uint8_t* q, float* s,
                                 cudaStream_t stream);
cudaError_t launch_colsum_int4(const uint8_t* q, int64_t N, int64_t K, int32_t* colsum, cudaStream_t stream);

// Block-scaled int8 weights: one E8M0 scale per (row, group of G K elements), amax / 127
// rounded up to a power of two with the exponent clamped to [103, 136]; codes
// clamp(rint(w / s), -127, 127); scale bytes packed four per 32-bit word (byte g % 4 of word
// g / 4), words group-major (word w of row n at sf[w * N + n]). K % G == 0.
constexpr int kMxEmin = 103, kMxEmax = 136;
cudaError_t launch_quantize_weight_mx(const float* w, int64_t N, int64_t K, int G, int8_t* q, uint32_t* sf,
                                      cudaStream_t stream);

// Fused RMSNorm + per-token symmetric quantization of x[rows, cols] (cols % 4 == 0).
cudaError_t launch_rmsnorm_quantize(const float* x, const float* gamma, int64_t rows, int64_t cols, float eps,
                                   int8_t* q, float* s, cudaStream_t stream);
cudaError_t launch_colsum(const int8_t* qw, int64_t N, int64_t K, int32_t* colsum,
                          cudaStream_t stream);

// Epilogue operands shared by every GEMM kernel. When out_i32 != nullptr the
// kernel writes the raw accumulators there instead of y.
enum OutKind : int { kOutF32 = 0, kOutBF16 = 1, kOutI8 = 2 };

struct Epilogue {
    const float* s_a;
    const int32_t* z_a;      // nullptr: symmetric A
    const float* s_w;
    const int32_t* colsum;   // used iff z_a != nullptr
    bool a_per_row;
    bool w_per_row;
    float* y;                // kOutF32 output
    int32_t* out_i32;        // raw accumulators instead of the epilogue (diagnostic export)
    // Epilogue variants: y + bias[n], written as fp32 (y), bf16 (out_bf16, round to nearest
    // even) or int8 codes clamp(rint(y / out_scale), -127, 127) (out_i8).
    const float* bias = nullptr;
    int out_kind = kOutF32;
    uint16_t* out_bf16 = nullptr;
    int8_t* out_i8 = nullptr;
    float out_scale = 1.0f;
    // Block-scaled weights (CTA-pair kernel): E8M0 scale words and group size; the kernel then
    // accumulates sum_k qa * (q * s) in fp32 and the epilogue is y = fl(T * s_a) (+ bias).
    const uint32_t* mx_sf = nullptr;
    int mx_group = 0;
    // Decode kernels (programmatic dependent launch): load the first weight boxes before waiting
    // for the preceding kernel. Only for a launch that directly follows the library's activation
    // quantizer of the same layer on the same stream, whose outputs do not overlap the weights.
    bool pdl_early_weights = false;
    // Self-test of the bounded waits (q8_selftest_wait_timeout), 0 in every other launch. When
    // > 0, the TMA producer of the single-CTA tcgen05 kernel or of the int8 decode kernel issues
    // no load, and the consumers' wait on the first loaded stage (converter warps, compute
    // warps) gives up after this many clock cycles, with nothing asynchronous in flight; the
    // other roles leave on the abort flag.
    long long selftest_wait_cycles = 0;
};

#ifdef __CUDACC__
__device__ __forceinline__ float epi_bias(const Epilogue& ep, float v, int64_t n) {
    return ep.bias ? __fadd_rn(v, __ldg(ep.bias + n)) : v;
}

__device__ __forceinline__ void epi_store(const Epilogue& ep, int64_t idx, float v) {
    if (ep.out_kind == kOutBF16) {
        ep.out_bf16[idx] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
    } else if (ep.out_kind == kOutI8) {
        ep.out_i8[idx] = (int8_t)min(max(__float2int_rn(__fdiv_rn(v, ep.out_scale)), -127), 127);
    } else {
        ep.y[idx] = v;
    }
}
#endif

// Output of a layer with K == 0 in the epilogue's output type (bias only).
cudaError_t launch_epilogue_fill(const Epilogue& ep, int64_t M, int64_t N, cudaStream_t stream);

cudaError_t launch_gemm_mma(const int8_t* qa, const int8_t* qw, int64_t M, int64_t N, int64_t K,
                            const Epilogue& ep, bool skinny, cudaStream_t stream);

// tcgen05 kernel; returns cudaErrorNotSupported when the shape is outside its range.
cudaError_t launch_gemm_tc(const int8_t* qa, const int8_t* qw, int64_t M, int64_t N, int64_t K,
                           const Epilogue& ep, cudaStream_t stream);
bool gemm_tc_supports(int64_t M, int64_t N, int64_t K);

// Operand formats of the CTA-pair kernel: int8 codes, packed int4 codes, block-scaled int8
// weights (activations as int8 codes), or int8 / packed int4 / block-scaled weights with the
// activation codes as fp16 values (kWA16: in K order; kW4A16, kWMxA16: in pair order, each group
// of four K stored as K 0, 2, 1, 3, the order in which the kernel converts the weight codes).
enum WeightFormat : int { kWInt8 = 0, kWInt4 = 1, kWMx = 2, kWA16 = 3, kW4A16 = 4, kWMxA16 = 5 };

// tcgen05 kernel on CTA pairs (cta_group::2, 256 x 256 tiles). qa: int8 codes, or fp16 code
// values for kWA16, kW4A16 and kWMxA16.
cudaError_t launch_gemm_tc2(const void* qa, const void* qw, int64_t M, int64_t N, int64_t K, const Epilogue& ep,
                            cudaStream_t stream, int wfmt = kWInt8);
bool gemm_tc2_supports(int64_t M, int64_t N, int64_t K, int wfmt = kWInt8);

// tcgen05 kernel for M <= 16 (decode): weight rows on the MMA's M side.
cudaError_t launch_gemv_tc(const int8_t* qa, const int8_t* qw, int64_t M, int64_t N, int64_t K,
                           const Epilogue& ep, cudaStream_t stream);
bool gemv_tc_supports(int64_t M, int64_t N, int64_t K);

// Warp-level fp16 MMA kernel for M <= 16 (decode), int8 or packed int4 (w4) weights streamed by TMA.
cudaError_t launch_gemv_mma(const int8_t* qa, const void* qw, int64_t M, int64_t N, int64_t K, const Epilogue& ep,
                            cudaStream_t stream, bool w4 = false);
bool gemv_mma_supports(int64_t M, int64_t N, int64_t K, bool w4 = false);
// Block-scaled int8 weights (E8M0 words sf, group G) for M <= 16, on the same stream design.
cudaError_t launch_gemv_mx(const int8_t* qa, const int8_t* qw, const uint32_t* sf, int G, int64_t M, int64_t N,
                           int64_t K, const Epilogue& ep, cudaStream_t stream);
bool gemv_mx_supports(int64_t M, int64_t N, int64_t K, int G, const void* sf);

// Device error words (bounded waits that gave up), one per kernel file and device.
cudaError_t read_and_clear_gemm_tc_error(uint32_t* code);
cudaError_t read_and_clear_gemv_tc_error(uint32_t* code);
cudaError_t read_and_clear_gemv_mma_error(uint32_t* code);
cudaError_t read_and_clear_gemm_tc2_error(uint32_t* code);
cudaError_t read_and_clear_quant_error(uint32_t* code);

}  // namespace q8
