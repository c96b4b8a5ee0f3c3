// Integer GEMM on the warp-level int8 tensor-core instruction
// mma.sync.m16n8k32.s32.s8.s8.s32 (exact INT32 accumulation by definition of
// the instruction), with the dequantization epilogue fused on the registers.
//
// This is the simple, general kernel: any M and N (ragged tiles are zero
// filled on load and masked on store), K a multiple of 16. Operands stream
// through a multi-stage cp.async ring in shared memory; each 128-byte smem row
// is XOR-swizzled by 16-byte chunk so that ldmatrix reads are conflict free.
//
//   acc[m][n] = sum_k qa[m][k] * qw[n][k]
//   y[m][n]   = (float)(acc - z_a[m] * colsum[n]) * (s_a[m] * s_w[n])
#include <cuda_runtime.h>
#include <stdint.h>

#include "q8_internal.h"

namespace q8 {
namespace {

constexpr int BK = 128;  // bytes (= int8 elements) of K per stage, one 128 B smem row

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte async copy global -> shared; src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                            uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_s8(int (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of 16-byte chunk `c` (0..7) of smem row `r` in a swizzled tile.
__device__ __forceinline__ uint32_t swz(int r, int c) { return (uint32_t)(r * BK + ((c ^ (r & 7)) << 4)); }

template <int BM, int BN, int WM, int WN, int STAGES>
struct Cfg {
    static constexpr int kWarpsM = BM / WM, kWarpsN = BN / WN;
    static constexpr int kThreads = kWarpsM * kWarpsN * 32;
    static constexpr int kMT = WM / 16, kNT = WN / 8;  // mma tiles per warp
    static constexpr int kStageBytes = (BM + BN) * BK;
    static constexpr int kSmem = STAGES * kStageBytes;
    static_assert(kNT % 2 == 0, "B fragments are loaded two n8 tiles at a time");
};

template <int BM, int BN, int WM, int WN, int STAGES>
__global__ void __launch_bounds__(Cfg<BM, BN, WM, WN, STAGES>::kThreads)
    gemm_mma_kernel(const int8_t* __restrict__ qa, const int8_t* __restrict__ qw, int M, int N, int K,
                    Epilogue ep) {
    using C = Cfg<BM, BN, WM, WN, STAGES>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int wm = (warp / C::kWarpsN) * WM, wn = (warp % C::kWarpsN) * WN;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const int ktiles = (K + BK - 1) / BK;

    auto load_stage = [&](int stage, int kt) {
        uint8_t* sa = smem + stage * C::kStageBytes;
        uint8_t* sb = sa + BM * BK;
        const int k0 = kt * BK;
        for (int i = tid; i < (BM + BN) * (BK / 16); i += C::kThreads) {
            const int r = i / (BK / 16), c = i % (BK / 16);
            const int k = k0 + c * 16;
            if (r < BM) {
                const int m = m0 + r;
                const bool ok = (m < M) && (k < K);
                const int8_t* src = qa + (ok ? ((int64_t)m * K + k) : 0);
                cp_async16(smem_u32(sa + swz(r, c)), src, ok ? 16 : 0);
            } else {
                const int rr = r - BM;
                const int n = n0 + rr;
                const bool ok = (n < N) && (k < K);
                const int8_t* src = qw + (ok ? ((int64_t)n * K + k) : 0);
                cp_async16(smem_u32(sb + swz(rr, c)), src, ok ? 16 : 0);
            }
        }
    };

    int acc[C::kMT][C::kNT][4];
#pragma unroll
    for (int i = 0; i < C::kMT; ++i)
#pragma unroll
        for (int j = 0; j < C::kNT; ++j)
#pragma unroll
            for (int t = 0; t < 4; ++t) acc[i][j][t] = 0;

#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
        if (s < ktiles) load_stage(s, s);
        cp_async_commit();
    }

    for (int kt = 0; kt < ktiles; ++kt) {
        cp_async_wait<STAGES - 2>();
        __syncthreads();
        // Refill the slot consumed in the previous iteration.
        const int nk = kt + STAGES - 1;
        if (nk < ktiles) load_stage(nk % STAGES, nk);
        cp_async_commit();

        const uint8_t* sa = smem + (kt % STAGES) * C::kStageBytes;
        const uint8_t* sb = sa + BM * BK;
#pragma unroll
        for (int kk = 0; kk < BK / 32; ++kk) {
            uint32_t af[C::kMT][4];
            uint32_t bf[C::kNT][2];
#pragma unroll
            for (int i = 0; i < C::kMT; ++i) {
                const int r = wm + i * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int c = kk * 2 + (lane >> 4);
                ldmatrix_x4(smem_u32(sa + swz(r, c)), af[i][0], af[i][1], af[i][2], af[i][3]);
            }
#pragma unroll
            for (int j = 0; j < C::kNT; j += 2) {
                const int r = wn + j * 8 + (lane & 7) + (lane >> 4) * 8;
                const int c = kk * 2 + ((lane >> 3) & 1);
                ldmatrix_x4(smem_u32(sb + swz(r, c)), bf[j][0], bf[j][1], bf[j + 1][0], bf[j + 1][1]);
            }
#pragma unroll
            for (int i = 0; i < C::kMT; ++i)
#pragma unroll
                for (int j = 0; j < C::kNT; ++j) mma_s8(acc[i][j], af[i], bf[j][0], bf[j][1]);
        }
    }
    cp_async_wait<0>();

    // Epilogue straight from the accumulator fragments: c0,c1 are row g,
    // columns 2t, 2t+1 of the m16n8 tile; c2,c3 are row g + 8.
    const int g = lane / 4, t4 = lane % 4;
#pragma unroll
    for (int i = 0; i < C::kMT; ++i) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int m = m0 + wm + i * 16 + g + h * 8;
            if (m >= M) continue;
            const float sa_m = ep.s_a ? ep.s_a[ep.a_per_row ? m : 0] : 1.0f;
            const int za_m = ep.z_a ? ep.z_a[ep.a_per_row ? m : 0] : 0;
#pragma unroll
            for (int j = 0; j < C::kNT; ++j) {
                const int n = n0 + wn + j * 8 + t4 * 2;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int nn = n + e;
                    if (nn >= N) continue;
                    const int a = acc[i][j][h * 2 + e];
                    if (ep.out_i32) {
                        ep.out_i32[(int64_t)m * N + nn] = a;
                    } else {
                        const int corr = ep.z_a ? a - za_m * ep.colsum[nn] : a;
                        const float scale = __fmul_rn(sa_m, ep.s_w[ep.w_per_row ? nn : 0]);
                        epi_store(ep, (int64_t)m * N + nn, epi_bias(ep, __fmul_rn(__int2float_rn(corr), scale), nn));
                    }
                }
            }
        }
    }
}

template <int BM, int BN, int WM, int WN, int STAGES>
cudaError_t launch_cfg(const int8_t* qa, const int8_t* qw, int64_t M, int64_t N, int64_t K,
                       const Epilogue& ep, cudaStream_t st) {
    using C = Cfg<BM, BN, WM, WN, STAGES>;
    auto kern = gemm_mma_kernel<BM, BN, WM, WN, STAGES>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((N + BN - 1) / BN), (unsigned)((M + BM - 1) / BM));
    kern<<<grid, C::kThreads, C::kSmem, st>>>(qa, qw, (int)M, (int)N, (int)K, ep);
    note_launch();
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_mma(const int8_t* qa, const int8_t* qw, int64_t M, int64_t N, int64_t K,
                            const Epilogue& ep, bool skinny, cudaStream_t stream) {
    if (skinny) return launch_cfg<16, 64, 16, 16, 6>(qa, qw, M, N, K, ep, stream);
    return launch_cfg<128, 128, 64, 32, 4>(qa, qw, M, N, K, ep, stream);
}

}  // namespace q8
