// C ABI of the library: host-side argument validation, kernel choice and the
// mapping of CUDA errors to q8_status. Validation runs before any CUDA call, so
// a rejected call enqueues nothing (and can be exercised without a GPU).
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <math.h>

#include "q8_internal.h"

namespace q8 {

static std::atomic<uint64_t> g_launches{0};
void note_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

}  // namespace q8

namespace {

// 128*128*K < 2^31 for any int8 codes; (255*128)*K < 2^31 once a zero point
// (|qa - z| <= 255) enters the correction.
constexpr int64_t kMaxKSym = 131056;
constexpr int64_t kMaxKAsym = 65792;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool valid_gran(q8_granularity g) { return g == Q8_PER_TENSOR || g == Q8_PER_ROW; }

q8_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return Q8_OK;
    if (e == cudaErrorNotSupported) return Q8_ERR_UNSUPPORTED;
    return Q8_ERR_CUDA;
}

q8_status check_k(int64_t K, bool asym) {
    if (K < 0) return Q8_ERR_INVALID_ARG;
    if (K % 16 != 0) return Q8_ERR_UNSUPPORTED;
    if (K > (asym ? kMaxKAsym : kMaxKSym)) return Q8_ERR_UNSUPPORTED;
    return Q8_OK;
}

q8_status check_quant_args(const float* x, int64_t rows, int64_t cols, q8_granularity g, const int8_t* q,
                           const float* s, bool need_matrix_ptrs) {
    if (rows < 0 || cols < 0 || !valid_gran(g)) return Q8_ERR_INVALID_ARG;
    if (!s || !aligned(s, 4)) return Q8_ERR_INVALID_ARG;
    if (need_matrix_ptrs) {
        if (!x || !q || !aligned(x, 16) || !aligned(q, 16)) return Q8_ERR_INVALID_ARG;
    }
    if (cols % 16 != 0) return Q8_ERR_UNSUPPORTED;
    return Q8_OK;
}

// Epilogue variants of q8_gemm_epilogue_ex (bias, output type); nullptr for the plain fp32 entries.
struct Variant {
    const float* bias;
    q8_out_type out_type;
    void* out;
    float out_scale;
};

// Block-scaled weights of q8_gemm_mx_ex: E8M0 scale words and the group size.
struct MxWeights {
    const uint32_t* sf;
    int group;
};

// Workspace the automatic kernel choice can use: an fp16 copy of the activation codes (2 M K bytes)
// for shapes on the CTA-pair kernel, else none.
size_t gemm_ws_bytes(int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0 || K <= 0 || K % 16 != 0) return 0;
    if (q8_gemm_pick(M, N, K) != Q8_GEMM_TCGEN05_PAIR || !q8::gemm_tc2_supports(M, N, K, q8::kWA16)) return 0;
    return (size_t)M * (size_t)K * 2;
}

// Workspace of the int4 and block-scaled weight formats on the CTA-pair kernel: an fp16 copy of the
// activation codes (2 M K bytes), used when the caller's buffer holds it.
bool use_lowbit_ws(int64_t M, int64_t K, const void* ws, size_t ws_bytes) {
    return ws && aligned(ws, 16) && ws_bytes >= (size_t)M * (size_t)K * 2;
}

// qa: int8 codes, or (a16) the same codes as fp16 values.
q8_status gemm_common(const void* qa, const float* s_a, const int32_t* z_a, q8_granularity ga,
                      const int8_t* qw, const float* s_w, q8_granularity gw, const int32_t* colsum,
                      int64_t M, int64_t N, int64_t K, float* y, int32_t* out_i32, q8_gemm_kernel kernel,
                      q8_stream_t stream, const Variant* var = nullptr, bool w4 = false,
                      const MxWeights* mx = nullptr, bool a16 = false, bool validate_only = false,
                      bool early_weights = false, long long selftest_wait = 0, void* ws = nullptr,
                      size_t ws_bytes = 0) {
    if (M < 0 || N < 0 || K < 0) return Q8_ERR_INVALID_ARG;
    if (kernel != Q8_GEMM_AUTO && kernel != Q8_GEMM_TCGEN05 && kernel != Q8_GEMM_MMA_S8 &&
        kernel != Q8_GEMM_SKINNY && kernel != Q8_GEMM_DECODE && kernel != Q8_GEMM_DECODE_TC &&
        kernel != Q8_GEMM_TCGEN05_PAIR)
        return Q8_ERR_INVALID_ARG;
    const bool epilogue = (out_i32 == nullptr);
    if (epilogue && (!valid_gran(ga) || !valid_gran(gw))) return Q8_ERR_INVALID_ARG;
    {
        q8_status kst = check_k(K, epilogue && z_a != nullptr);
        if (kst != Q8_OK) return kst;
        if (w4 && K % 32 != 0) return Q8_ERR_UNSUPPORTED;   // packed int4 rows: whole 16-byte multiples
    }
    if (a16 && kernel != Q8_GEMM_AUTO && kernel != Q8_GEMM_TCGEN05_PAIR) return Q8_ERR_UNSUPPORTED;
    if (mx) {
        if (mx->group != 32 && mx->group != 128) return Q8_ERR_INVALID_ARG;
        if (z_a || !epilogue) return Q8_ERR_UNSUPPORTED;     // symmetric activations, dequantized output
        if (kernel != Q8_GEMM_AUTO && kernel != Q8_GEMM_TCGEN05_PAIR && kernel != Q8_GEMM_DECODE)
            return Q8_ERR_UNSUPPORTED;
        if (K % mx->group != 0) return Q8_ERR_UNSUPPORTED;
    }
    if (M == 0 || N == 0) return Q8_OK;   // empty output: nothing is read or written
    if (var) {
        if (var->out_type != Q8_OUT_F32 && var->out_type != Q8_OUT_BF16 && var->out_type != Q8_OUT_I8)
            return Q8_ERR_INVALID_ARG;
        if (var->out_type == Q8_OUT_I8 && !(var->out_scale > 0.0f && var->out_scale < INFINITY))
            return Q8_ERR_INVALID_ARG;
        if (var->bias && !aligned(var->bias, 4)) return Q8_ERR_INVALID_ARG;
        if (!var->out || !aligned(var->out, 16)) return Q8_ERR_INVALID_ARG;
        y = var->out_type == Q8_OUT_F32 ? static_cast<float*>(var->out) : nullptr;
    }
    if (epilogue) {
        if (!s_a || (!s_w && !mx) || (!y && !var)) return Q8_ERR_INVALID_ARG;
        if (!aligned(s_a, 4) || (s_w && !aligned(s_w, 4)) || (y && !aligned(y, 16))) return Q8_ERR_INVALID_ARG;
        if (z_a && (!colsum || !aligned(z_a, 4) || !aligned(colsum, 4))) return Q8_ERR_INVALID_ARG;
    } else if (!aligned(out_i32, 16)) {
        return Q8_ERR_INVALID_ARG;
    }
    if (M > 0 && N > 0 && K > 0) {
        if (!qa || !qw || !aligned(qa, 16) || !aligned(qw, 16)) return Q8_ERR_INVALID_ARG;
        if (mx && (!mx->sf || !aligned(mx->sf, 4))) return Q8_ERR_INVALID_ARG;
    }
    if (M > INT32_MAX || N > INT32_MAX) return Q8_ERR_UNSUPPORTED;
    if (validate_only) return Q8_OK;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    q8::Epilogue ep{s_a, z_a, s_w, colsum, ga == Q8_PER_ROW, gw == Q8_PER_ROW, y, out_i32};
    ep.pdl_early_weights = early_weights;
    ep.selftest_wait_cycles = selftest_wait;
    if (var) {
        ep.bias = var->bias;
        ep.out_kind = var->out_type == Q8_OUT_BF16 ? q8::kOutBF16 : var->out_type == Q8_OUT_I8 ? q8::kOutI8 : q8::kOutF32;
        ep.out_bf16 = var->out_type == Q8_OUT_BF16 ? static_cast<uint16_t*>(var->out) : nullptr;
        ep.out_i8 = var->out_type == Q8_OUT_I8 ? static_cast<int8_t*>(var->out) : nullptr;
        ep.out_scale = var->out_scale;
    }
    if (K == 0) {
        // Empty dot products: acc = 0, colsum = 0, so y = 0 * scale = +0.0f (+ bias).
        if (var && (var->bias || var->out_type != Q8_OUT_F32)) return from_cuda(q8::launch_epilogue_fill(ep, M, N, s));
        const size_t bytes = (size_t)M * (size_t)N * 4;
        return from_cuda(cudaMemsetAsync(epilogue ? (void*)y : (void*)out_i32, 0, bytes, s));
    }
    const int8_t* qa8 = static_cast<const int8_t*>(qa);
    if (a16) {
        // fp16 activation codes: the CTA-pair kernel with TMA loads of A into its operand ring
        if (!q8::gemm_tc2_supports(M, N, K, q8::kWA16)) return Q8_ERR_UNSUPPORTED;
        return from_cuda(q8::launch_gemm_tc2(qa, qw, M, N, K, ep, s, q8::kWA16));
    }
    if (mx) {
        // block-scaled weights: the decode kernel for M <= 16 (N % 4 == 0, 16-byte aligned scale
        // words), the CTA-pair kernel otherwise
        ep.s_w = nullptr;
        ep.mx_sf = mx->sf;
        ep.mx_group = mx->group;
        if (kernel == Q8_GEMM_AUTO)
            kernel = q8::gemv_mx_supports(M, N, K, mx->group, mx->sf) ? Q8_GEMM_DECODE : Q8_GEMM_TCGEN05_PAIR;
        if (kernel == Q8_GEMM_DECODE) {
            if (!q8::gemv_mx_supports(M, N, K, mx->group, mx->sf)) return Q8_ERR_UNSUPPORTED;
            return from_cuda(q8::launch_gemv_mx(qa8, qw, mx->sf, mx->group, M, N, K, ep, s));
        }
        if (!q8::gemm_tc2_supports(M, N, K, q8::kWMx)) return Q8_ERR_UNSUPPORTED;
        if (use_lowbit_ws(M, K, ws, ws_bytes)) {   // the codes as fp16 values (pair order) by TMA
            uint16_t* qa16 = static_cast<uint16_t*>(ws);
            cudaError_t e = q8::launch_codes_to_f16(qa8, M * K, qa16, s, true);
            if (e != cudaSuccess) return from_cuda(e);
            return from_cuda(q8::launch_gemm_tc2(qa16, qw, M, N, K, ep, s, q8::kWMxA16));
        }
        return from_cuda(q8::launch_gemm_tc2(qa8, qw, M, N, K, ep, s, q8::kWMx));
    }
    if (w4) {
        // int4 weights run on the decode kernel (M <= 16) and the CTA-pair kernel
        if (kernel == Q8_GEMM_AUTO) kernel = q8::gemv_mma_supports(M, N, K, true) ? Q8_GEMM_DECODE : Q8_GEMM_TCGEN05_PAIR;
        if (kernel == Q8_GEMM_DECODE) {
            if (!q8::gemv_mma_supports(M, N, K, true)) return Q8_ERR_UNSUPPORTED;
            return from_cuda(q8::launch_gemv_mma(qa8, qw, M, N, K, ep, s, true));
        }
        if (kernel == Q8_GEMM_TCGEN05_PAIR) {
            if (!q8::gemm_tc2_supports(M, N, K, q8::kWInt4)) return Q8_ERR_UNSUPPORTED;
            if (use_lowbit_ws(M, K, ws, ws_bytes)) {   // the codes as fp16 values (pair order) by TMA
                uint16_t* qa16 = static_cast<uint16_t*>(ws);
                cudaError_t e = q8::launch_codes_to_f16(qa8, M * K, qa16, s, true);
                if (e != cudaSuccess) return from_cuda(e);
                return from_cuda(q8::launch_gemm_tc2(qa16, qw, M, N, K, ep, s, q8::kW4A16));
            }
            return from_cuda(q8::launch_gemm_tc2(qa8, qw, M, N, K, ep, s, q8::kWInt4));
        }
        return Q8_ERR_UNSUPPORTED;
    }
    if (kernel == Q8_GEMM_AUTO) {
        kernel = q8_gemm_pick(M, N, K);
        // With a workspace for an fp16 copy of the activation codes, the CTA-pair layer converts
        // the codes once (a stream through HBM) and loads them by TMA straight into its operand
        // stages, instead of converting every code once per output tile in shared memory.
        if (kernel == Q8_GEMM_TCGEN05_PAIR && ws && ws_bytes >= gemm_ws_bytes(M, N, K) && aligned(ws, 16) &&
            q8::gemm_tc2_supports(M, N, K, q8::kWA16)) {
            uint16_t* qa16 = static_cast<uint16_t*>(ws);
            cudaError_t e = q8::launch_codes_to_f16(qa8, M * K, qa16, s);
            if (e != cudaSuccess) return from_cuda(e);
            return from_cuda(q8::launch_gemm_tc2(qa16, qw, M, N, K, ep, s, q8::kWA16));
        }
    }
    switch (kernel) {
        case Q8_GEMM_TCGEN05:
            if (!q8::gemm_tc_supports(M, N, K)) return Q8_ERR_UNSUPPORTED;
            return from_cuda(q8::launch_gemm_tc(qa8, qw, M, N, K, ep, s));
        case Q8_GEMM_TCGEN05_PAIR:
            if (!q8::gemm_tc2_supports(M, N, K)) return Q8_ERR_UNSUPPORTED;
            return from_cuda(q8::launch_gemm_tc2(qa8, qw, M, N, K, ep, s));
        case Q8_GEMM_DECODE:
            if (!q8::gemv_mma_supports(M, N, K)) return Q8_ERR_UNSUPPORTED;
            return from_cuda(q8::launch_gemv_mma(qa8, qw, M, N, K, ep, s));
        case Q8_GEMM_DECODE_TC:
            if (!q8::gemv_tc_supports(M, N, K)) return Q8_ERR_UNSUPPORTED;
            return from_cuda(q8::launch_gemv_tc(qa8, qw, M, N, K, ep, s));
        case Q8_GEMM_SKINNY:
            return from_cuda(q8::launch_gemm_mma(qa8, qw, M, N, K, ep, true, s));
        case Q8_GEMM_MMA_S8:
        default:
            return from_cuda(q8::launch_gemm_mma(qa8, qw, M, N, K, ep, false, s));
    }
}

q8_status check_act_args(const float* a, int64_t M, int64_t K, q8_granularity g, q8_symmetry sym, const int8_t* qa,
                         const float* s_a, const int32_t* z_a) {
    if (sym != Q8_SYMMETRIC && sym != Q8_ASYMMETRIC) return Q8_ERR_INVALID_ARG;
    if ((sym == Q8_ASYMMETRIC) != (z_a != nullptr)) return Q8_ERR_INVALID_ARG;
    if (z_a && !aligned(z_a, 4)) return Q8_ERR_INVALID_ARG;
    return check_quant_args(a, M, K, g, qa, s_a, M > 0 && K > 0);
}

// [p, p + bytes) and [q, q + bytes2) share a byte.
bool overlap(const void* p, size_t bytes, const void* q, size_t bytes2) {
    if (!p || !q || bytes == 0 || bytes2 == 0) return false;
    const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
    return a < b + bytes2 && b < a + bytes;
}

}  // namespace

extern "C" {

q8_status q8_quantize_act(const float* a, int64_t M, int64_t K, q8_granularity g, q8_symmetry sym,
                          int8_t* qa, float* s_a, int32_t* z_a, q8_stream_t stream) {
    q8_status st = check_act_args(a, M, K, g, sym, qa, s_a, z_a);
    if (st != Q8_OK) return st;
    if (g == Q8_PER_ROW && M == 0) return Q8_OK;
    return from_cuda(q8::launch_quantize(a, M, K, g == Q8_PER_ROW, qa, s_a, z_a,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

q8_status q8_linear(const float* a, int64_t M, int64_t K, q8_granularity ga, q8_symmetry sym, int8_t* qa, float* s_a,
                    int32_t* z_a, const int8_t* qw, const float* s_w, q8_granularity gw, const int32_t* colsum,
                    int64_t N, float* y, q8_stream_t stream) {
    // Both halves are validated before either is enqueued.
    q8_status st = check_act_args(a, M, K, ga, sym, qa, s_a, z_a);
    if (st != Q8_OK) return st;
    st = gemm_common(qa, s_a, z_a, ga, qw, s_w, gw, colsum, M, N, K, y, nullptr, Q8_GEMM_AUTO, stream, nullptr, false,
                     nullptr, false, true);
    if (st != Q8_OK) return st;
    if (M == 0) return Q8_OK;
    st = q8_quantize_act(a, M, K, ga, sym, qa, s_a, z_a, stream);
    if (st != Q8_OK) return st;
    // The decode kernels may start their weight stream while the quantizer runs, unless the
    // quantizer's outputs share memory with a weight operand.
    const size_t ns = ga == Q8_PER_ROW ? (size_t)M * 4 : 4, nw = gw == Q8_PER_ROW ? (size_t)N * 4 : 4;
    const void* outs[3] = {qa, s_a, z_a};
    const size_t out_bytes[3] = {(size_t)M * (size_t)K, ns, z_a ? ns : 0};
    const void* ins[3] = {qw, s_w, z_a ? colsum : nullptr};
    const size_t in_bytes[3] = {(size_t)N * (size_t)K, nw, (size_t)N * 4};
    bool early = true;
    for (int i = 0; i < 3; ++i)
        for (int j = 0; j < 3; ++j) early = early && !overlap(outs[i], out_bytes[i], ins[j], in_bytes[j]);
    return gemm_common(qa, s_a, z_a, ga, qw, s_w, gw, colsum, M, N, K, y, nullptr, Q8_GEMM_AUTO, stream, nullptr,
                       false, nullptr, false, false, early);
}

q8_status q8_quantize_act_dual(const float* a, int64_t M, int64_t K, q8_granularity g, q8_symmetry sym, int8_t* qa,
                               uint16_t* qa16, float* s_a, int32_t* z_a, q8_stream_t stream) {
    q8_status st = check_act_args(a, M, K, g, sym, qa, s_a, z_a);
    if (st != Q8_OK) return st;
    if (M > 0 && K > 0 && (!qa16 || !aligned(qa16, 16))) return Q8_ERR_INVALID_ARG;
    if (g == Q8_PER_ROW && M == 0) return Q8_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (g == Q8_PER_ROW && K > 0) {
        // one pass: both code formats from the row in registers
        cudaError_t e = q8::launch_quantize_dual(a, M, K, qa, qa16, s_a, z_a, s);
        if (e != cudaErrorNotSupported) return from_cuda(e);
    }
    cudaError_t e = q8::launch_quantize(a, M, K, g == Q8_PER_ROW, qa, s_a, z_a, s);
    if (e != cudaSuccess) return from_cuda(e);
    return from_cuda(q8::launch_codes_to_f16(qa, M * K, qa16, s));
}

q8_status q8_linear_ws(const float* a, int64_t M, int64_t K, q8_granularity ga, q8_symmetry sym, int8_t* qa,
                       float* s_a, int32_t* z_a, const int8_t* qw, const float* s_w, q8_granularity gw,
                       const int32_t* colsum, int64_t N, float* y, void* workspace, size_t workspace_bytes,
                       q8_stream_t stream) {
    if (workspace && !aligned(workspace, 16)) return Q8_ERR_INVALID_ARG;
    const size_t need = gemm_ws_bytes(M, N, K);
    if (!workspace || need == 0 || workspace_bytes < need)
        return q8_linear(a, M, K, ga, sym, qa, s_a, z_a, qw, s_w, gw, colsum, N, y, stream);
    // Both halves are validated before either is enqueued: the quantizer writes the int8 codes to qa
    // and the same codes as fp16 values into the workspace, which the CTA-pair kernel loads by TMA.
    q8_status st = check_act_args(a, M, K, ga, sym, qa, s_a, z_a);
    if (st != Q8_OK) return st;
    st = gemm_common(workspace, s_a, z_a, ga, qw, s_w, gw, colsum, M, N, K, y, nullptr, Q8_GEMM_AUTO, stream, nullptr,
                     false, nullptr, true, true);
    if (st != Q8_OK) return st;
    st = q8_quantize_act_dual(a, M, K, ga, sym, qa, static_cast<uint16_t*>(workspace), s_a, z_a, stream);
    if (st != Q8_OK) return st;
    return gemm_common(workspace, s_a, z_a, ga, qw, s_w, gw, colsum, M, N, K, y, nullptr, Q8_GEMM_AUTO, stream,
                       nullptr, false, nullptr, true);
}

q8_status q8_quantize_act_f16(const float* a, int64_t M, int64_t K, q8_granularity g, q8_symmetry sym,
                              uint16_t* qa16, float* s_a, int32_t* z_a, q8_stream_t stream) {
    q8_status st = check_act_args(a, M, K, g, sym, reinterpret_cast<const int8_t*>(qa16), s_a, z_a);
    if (st != Q8_OK) return st;
    if (g == Q8_PER_ROW && M == 0) return Q8_OK;
    return from_cuda(q8::launch_quantize_f16(a, M, K, g == Q8_PER_ROW, qa16, s_a, z_a,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

q8_status q8_rmsnorm_quantize_act(const float* a, const float* gamma, int64_t M, int64_t K, float eps, int8_t* qa,
                                  float* s_a, q8_stream_t stream) {
    if (M < 0 || !(eps > 0.0f) || !(eps < INFINITY)) return Q8_ERR_INVALID_ARG;
    if (M == 0) return Q8_OK;
    if (K <= 0) return Q8_ERR_INVALID_ARG;
    if (!a || !gamma || !qa || !s_a || !aligned(a, 16) || !aligned(gamma, 16) || !aligned(qa, 16) ||
        !aligned(s_a, 4))
        return Q8_ERR_INVALID_ARG;
    if (K % 16 != 0 || K > (int64_t(1) << 24)) return Q8_ERR_UNSUPPORTED;
    return from_cuda(q8::launch_rmsnorm_quantize(a, gamma, M, K, eps, qa, s_a,
                                                 reinterpret_cast<cudaStream_t>(stream)));
}

q8_status q8_quantize_weight_int4(const float* w, int64_t N, int64_t K, uint8_t* qw4, float* s_w,
                                  q8_stream_t stream) {
    if (N < 0 || K < 0) return Q8_ERR_INVALID_ARG;
    if (K % 32 != 0) return Q8_ERR_UNSUPPORTED;
    if (N == 0) return Q8_OK;
    if (!s_w || !aligned(s_w, 4)) return Q8_ERR_INVALID_ARG;
    if (K > 0 && (!w || !qw4 || !aligned(w, 16) || !aligned(qw4, 16))) return Q8_ERR_INVALID_ARG;
    return from_cuda(q8::launch_quantize_int4(w, N, K, qw4, s_w, reinterpret_cast<cudaStream_t>(stream)));
}

q8_status q8_colsum_int4(const uint8_t* qw4, int64_t N, int64_t K, int32_t* colsum, q8_stream_t stream) {
    if (N < 0 || K < 0) return Q8_ERR_INVALID_ARG;
    if (K % 32 != 0) return Q8_ERR_UNSUPPORTED;
    if (N == 0) return Q8_OK;
    if (!colsum || !aligned(colsum, 4)) return Q8_ERR_INVALID_ARG;
    if (K > 0 && (!qw4 || !aligned(qw4, 16))) return Q8_ERR_INVALID_ARG;
    return from_cuda(q8::launch_colsum_int4(qw4, N, K, colsum, reinterpret_cast<cudaStream_t>(stream)));
}

q8_status q8_quantize_weight(const float* w, int64_t N, int64_t K, q8_granularity g, int8_t* qw, float* s_w,
                             q8_stream_t stream) {
    q8_status st = check_quant_args(w, N, K, g, qw, s_w, N > 0 && K > 0);
    if (st != Q8_OK) return st;
    if (g == Q8_PER_ROW && N == 0) return Q8_OK;
    return from_cuda(q8::launch_quantize(w, N, K, g == Q8_PER_ROW, qw, s_w, nullptr,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

q8_status q8_colsum(const int8_t* qw, int64_t N, int64_t K, int32_t* colsum, q8_stream_t stream) {
    if (N < 0 || K < 0) return Q8_ERR_INVALID_ARG;
    if (K % 16 != 0 || K > kMaxKSym) return Q8_ERR_UNSUPPORTED;
    if (N == 0) return Q8_OK;
    if (!colsum || !aligned(colsum, 4)) return Q8_ERR_INVALID_ARG;
    if (K > 0 && (!qw || !aligned(qw, 16))) return Q8_ERR_INVALID_ARG;
    return from_cuda(q8::launch_colsum(qw, N, K, colsum, reinterpret_cast<cudaStream_t>(stream)));
}

q8_status q8_gemm_dequant(const int8_t* qa, const float* s_a, const int32_t* z_a, q8_granularity ga,
                          const int8_t* qw, const float* s_w, q8_granularity gw, const int32_t* colsum,
                          int64_t M, int64_t N, int64_t K, float* y, q8_stream_t stream) {
    return gemm_common(qa, s_a, z_a, ga, qw, s_w, gw, colsum, M, N, K, y, nullptr, Q8_GEMM_AUTO, stream);
}

size_t q8_gemm_workspace(int64_t M, int64_t N, int64_t K) { return gemm_ws_bytes(M, N, K); }

q8_status q8_gemm_dequant_ws(const int8_t* qa, const float* s_a, const int32_t* z_a, q8_granularity ga,
                             const int8_t* qw, const float* s_w, q8_granularity gw, const int32_t* colsum,
                             int64_t M, int64_t N, int64_t K, float* y, void* workspace, size_t workspace_bytes,
                             q8_stream_t stream) {
    if (workspace && !aligned(workspace, 16)) return Q8_ERR_INVALID_ARG;
    return gemm_common(qa, s_a, z_a, ga, qw, s_w, gw, colsum, M, N, K, y, nullptr, Q8_GEMM_AUTO, stream, nullptr,
                       false, nullptr, false, false, false, 0, workspace, workspace_bytes);
}

q8_status q8_gemm_dequant_ex(const int8_t* qa, const float* s_a, const int32_t* z_a, q8_granularity ga,
                             const int8_t* qw, const float* s_w, q8_granularity gw, const int32_t* colsum,
                             int64_t M, int64_t N, int64_t K, float* y, q8_gemm_kernel kernel,
                             q8_stream_t stream) {
    return gemm_common(qa, s_a, z_a, ga, qw, s_w, gw, colsum, M, N, K, y, nullptr, kernel, stream);
}

q8_status q8_gemm_epilogue_ex(const int8_t* qa, const float* s_a, const int32_t* z_a, q8_granularity ga,
                              const int8_t* qw, const float* s_w, q8_granularity gw, const int32_t* colsum,
                              const float* bias, int64_t M, int64_t N, int64_t K, q8_out_type out_type, void* out,
                              float out_scale, q8_gemm_kernel kernel, q8_stream_t stream) {
    const Variant var{bias, out_type, out, out_scale};
    return gemm_common(qa, s_a, z_a, ga, qw, s_w, gw, colsum, M, N, K, nullptr, nullptr, kernel, stream, &var);
}

q8_status q8_gemm_w4a8_ex(const int8_t* qa, const float* s_a, const int32_t* z_a, q8_granularity ga, const uint8_t* qw4,
                          const float* s_w, const int32_t* colsum, const float* bias, int64_t M, int64_t N, int64_t K,
                          q8_out_type out_type, void* out, float out_scale, q8_gemm_kernel kernel,
                          q8_stream_t stream) {
    const Variant var{bias, out_type, out, out_scale};
    return gemm_common(qa, s_a, z_a, ga, reinterpret_cast<const int8_t*>(qw4), s_w, Q8_PER_ROW, colsum, M, N, K,
                       nullptr, nullptr, kernel, stream, &var, true);
}

q8_status q8_gemm_w4a8_ws(const int8_t* qa, const float* s_a, const int32_t* z_a, q8_granularity ga, const uint8_t* qw4,
                          const float* s_w, const int32_t* colsum, const float* bias, int64_t M, int64_t N, int64_t K,
                          q8_out_type out_type, void* out, float out_scale, void* workspace, size_t workspace_bytes,
                          q8_stream_t stream) {
    if (workspace && !aligned(workspace, 16)) return Q8_ERR_INVALID_ARG;
    const Variant var{bias, out_type, out, out_scale};
    return gemm_common(qa, s_a, z_a, ga, reinterpret_cast<const int8_t*>(qw4), s_w, Q8_PER_ROW, colsum, M, N, K,
                       nullptr, nullptr, Q8_GEMM_AUTO, stream, &var, true, nullptr, false, false, false, 0, workspace,
                       workspace_bytes);
}

q8_status q8_gemm_w4a8_s32_ex(const int8_t* qa, const uint8_t* qw4, int64_t M, int64_t N, int64_t K, int32_t* acc,
                              q8_gemm_kernel kernel, q8_stream_t stream) {
    return gemm_common(qa, nullptr, nullptr, Q8_PER_ROW, reinterpret_cast<const int8_t*>(qw4), nullptr, Q8_PER_ROW,
                       nullptr, M, N, K, nullptr, acc, kernel, stream, nullptr, true);
}

q8_status q8_quantize_weight_mx(const float* w, int64_t N, int64_t K, int group, int8_t* qw, uint32_t* sf,
                                q8_stream_t stream) {
    if (N < 0 || K < 0 || (group != 32 && group != 128)) return Q8_ERR_INVALID_ARG;
    if (K % group != 0) return Q8_ERR_UNSUPPORTED;
    if (N == 0 || K == 0) return Q8_OK;
    if (!w || !qw || !sf || !aligned(w, 16) || !aligned(qw, 16) || !aligned(sf, 4)) return Q8_ERR_INVALID_ARG;
    return from_cuda(q8::launch_quantize_weight_mx(w, N, K, group, qw, sf, reinterpret_cast<cudaStream_t>(stream)));
}

q8_status q8_gemm_mx_ex(const int8_t* qa, const float* s_a, q8_granularity ga, const int8_t* qw, const uint32_t* sf,
                        int group, const float* bias, int64_t M, int64_t N, int64_t K, q8_out_type out_type,
                        void* out, float out_scale, q8_gemm_kernel kernel, q8_stream_t stream) {
    const Variant var{bias, out_type, out, out_scale};
    const MxWeights mx{sf, group};
    return gemm_common(qa, s_a, nullptr, ga, qw, nullptr, Q8_PER_ROW, nullptr, M, N, K, nullptr, nullptr, kernel,
                       stream, &var, false, &mx);
}

q8_status q8_gemm_mx_ws(const int8_t* qa, const float* s_a, q8_granularity ga, const int8_t* qw, const uint32_t* sf,
                        int group, const float* bias, int64_t M, int64_t N, int64_t K, q8_out_type out_type,
                        void* out, float out_scale, void* workspace, size_t workspace_bytes, q8_stream_t stream) {
    if (workspace && !aligned(workspace, 16)) return Q8_ERR_INVALID_ARG;
    const Variant var{bias, out_type, out, out_scale};
    const MxWeights mx{sf, group};
    return gemm_common(qa, s_a, nullptr, ga, qw, nullptr, Q8_PER_ROW, nullptr, M, N, K, nullptr, nullptr,
                       Q8_GEMM_AUTO, stream, &var, false, &mx, false, false, false, 0, workspace, workspace_bytes);
}

q8_status q8_gemm_f16a_ex(const uint16_t* qa16, const float* s_a, const int32_t* z_a, q8_granularity ga,
                          const int8_t* qw, const float* s_w, q8_granularity gw, const int32_t* colsum,
                          const float* bias, int64_t M, int64_t N, int64_t K, q8_out_type out_type, void* out,
                          float out_scale, q8_stream_t stream) {
    const Variant var{bias, out_type, out, out_scale};
    return gemm_common(qa16, s_a, z_a, ga, qw, s_w, gw, colsum, M, N, K, nullptr, nullptr, Q8_GEMM_AUTO, stream, &var,
                       false, nullptr, true);
}

q8_status q8_gemm_f16a_s32(const uint16_t* qa16, const int8_t* qw, int64_t M, int64_t N, int64_t K, int32_t* acc,
                           q8_stream_t stream) {
    if (!acc && M > 0 && N > 0) return Q8_ERR_INVALID_ARG;
    if (!acc) {  // empty output
        if (M < 0 || N < 0 || K < 0) return Q8_ERR_INVALID_ARG;
        return check_k(K, false);
    }
    return gemm_common(qa16, nullptr, nullptr, Q8_PER_TENSOR, qw, nullptr, Q8_PER_TENSOR, nullptr, M, N, K, nullptr,
                       acc, Q8_GEMM_AUTO, stream, nullptr, false, nullptr, true);
}

q8_status q8_gemm_s32_ex(const int8_t* qa, const int8_t* qw, int64_t M, int64_t N, int64_t K, int32_t* acc,
                         q8_gemm_kernel kernel, q8_stream_t stream) {
    if (!acc && M > 0 && N > 0) return Q8_ERR_INVALID_ARG;
    if (!acc) {  // empty output
        if (M < 0 || N < 0 || K < 0) return Q8_ERR_INVALID_ARG;
        return check_k(K, false);
    }
    return gemm_common(qa, nullptr, nullptr, Q8_PER_TENSOR, qw, nullptr, Q8_PER_TENSOR, nullptr, M, N, K,
                       nullptr, acc, kernel, stream);
}

q8_status q8_selftest_wait_timeout(q8_gemm_kernel kernel, const int8_t* qa, const int8_t* qw, int64_t M, int64_t N,
                                   int64_t K, int32_t* acc, int64_t wait_cycles, q8_stream_t stream) {
    if (kernel != Q8_GEMM_DECODE && kernel != Q8_GEMM_TCGEN05) return Q8_ERR_INVALID_ARG;
    if (wait_cycles < 1 || wait_cycles > (int64_t(1) << 31)) return Q8_ERR_INVALID_ARG;
    if (!acc || M <= 0 || N <= 0 || K <= 0) return Q8_ERR_INVALID_ARG;
    return gemm_common(qa, nullptr, nullptr, Q8_PER_TENSOR, qw, nullptr, Q8_PER_TENSOR, nullptr, M, N, K, nullptr,
                       acc, kernel, stream, nullptr, false, nullptr, false, false, false, (long long)wait_cycles);
}

// Measured on GB300: the CTA-pair kernel is the fastest tcgen05 kernel at every
// shape tried (M 64..8192); the 16 x 64-tile mma.sync kernel wins only where the
// pair grid would be tiny (at most 8 tiles of 256 x 256) or M is small and the
// weight matrix is small.
q8_gemm_kernel q8_gemm_pick(int64_t M, int64_t N, int64_t K) {
    if (q8::gemv_mma_supports(M, N, K)) return Q8_GEMM_DECODE;
    if (M >= 1 && N >= 1) {
        // measured with the pair kernel's K split: the mma.sync kernel wins only on small layers
        if (M <= 128 && N * K <= (int64_t(1) << 22)) return Q8_GEMM_SKINNY;
    }
    if (q8::gemm_tc2_supports(M, N, K)) return Q8_GEMM_TCGEN05_PAIR;
    if (q8::gemm_tc_supports(M, N, K)) return Q8_GEMM_TCGEN05;
    if (M <= 16) return Q8_GEMM_SKINNY;
    return Q8_GEMM_MMA_S8;
}

const char* q8_status_string(q8_status status) {
    switch (status) {
        case Q8_OK: return "ok";
        case Q8_ERR_INVALID_ARG: return "invalid argument";
        case Q8_ERR_UNSUPPORTED: return "unsupported shape or size";
        case Q8_ERR_CUDA: return "CUDA error";
        case Q8_ERR_TIMEOUT: return "device-side wait timed out";
        default: return "unknown status";
    }
}

q8_status q8_device_error(uint32_t* code_out) {
    if (!code_out) return Q8_ERR_INVALID_ARG;
    uint32_t a = 0, b = 0, c = 0, d = 0, qz = 0;
    cudaError_t e = q8::read_and_clear_gemm_tc_error(&a);
    if (e == cudaSuccess) e = q8::read_and_clear_gemv_tc_error(&b);
    if (e == cudaSuccess) e = q8::read_and_clear_gemv_mma_error(&c);
    if (e == cudaSuccess) e = q8::read_and_clear_gemm_tc2_error(&d);
    if (e == cudaSuccess) e = q8::read_and_clear_quant_error(&qz);
    if (e != cudaSuccess) return Q8_ERR_CUDA;
    *code_out = (a | qz) | (b << 8) | (c << 16) | (d << 24);
    return *code_out ? Q8_ERR_TIMEOUT : Q8_OK;
}

uint64_t q8_launch_count(void) { return q8::g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
