// Decode-shaped integer GEMM (M <= 16 tokens) + dequantization epilogue on the
// warp-level fp16 tensor-core instruction mma.sync.m16n8k16 (fp32 accumulate).
//
// With a handful of tokens the layer is a stream of the int8 weights from HBM
// with little arithmetic per byte. The weights go HBM -> shared memory by TMA
// (an 8-stage ring per SM; a stage is 64 rows x 256 bytes of K, fetched as two
// 128-byte boxes, which streams DRAM better than 128-byte row pieces) and shared
// memory -> registers by ordinary loads;
// each warp converts its int8 fragments to fp16 in registers and feeds them
// straight to the MMA, so converted data never goes back through shared memory.
// (The int8 MMA of this GPU runs at a fraction of the fp16 rate, too low for
// this stream.)
//
// Exactness: int8 codes and their products are exact in fp16 / fp32; each
// fp32 accumulator holds the sum of at most 1024 products (|sum| <= 2^24, an
// exactly representable integer) before it is converted to int32 and added to
// an INT32 total, so the result is the exact integer dot product.
//
// K order inside a stage: compute warp s (of 16) owns the 16 K values
// [16s, 16s+16) of every stage, one MMA K-step; lane quad t holds the 4 bytes
// [16s + 4t, +4) of its rows, bytes (0, 2) as the k pair (2t, 2t+1) and (1, 3)
// as (8+2t, 9+2t).
// Weights and activations use the same mapping, so the dot products are
// unchanged. With the 128-byte TMA swizzle these 4-byte loads hit 32 distinct
// banks.
//
// Work: 64 weight rows (output channels) per tile, tiles dealt round-robin to
// one CTA per SM. Each compute warp covers all 64 rows (eight n8 groups, eight
// independent accumulators) for its K-step, so a token fragment is converted
// once per eight MMAs; at the end of a tile the sixteen K-step partials are
// added in shared memory (integer adds, exact) and written out.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "q8_internal.h"
#include "q8_tc_ptx.cuh"

namespace q8 {

static __device__ unsigned int g_gemv_mma_error;

namespace {

using namespace tc;

constexpr int RW = 64;             // weight rows per tile
constexpr int NT = 16;             // token rows (MMA M)
constexpr int BK = 256;            // K of one step of all compute warps (one 16-wide K-step each)
constexpr int BKH = 128;           // bytes of one swizzled TMA box row
constexpr int kComputeWarps = BK / 16;
constexpr int kThreads = 32 * (1 + kComputeWarps);
// int32 tile sums [2 (tile parity)][16 tokens][64 rows], token rows padded to 72 words so
// that the eight tokens of one atomic instruction fall in different banks (2-way, not 8-way)
constexpr int RWP = RW + 8;
constexpr int kRedBytes = 2 * NT * RWP * 4;

// Weight format: int8 codes or int4 codes packed two per byte; a stage holds two W boxes of
// 64 rows x 128 bytes (16 KB). An fp32 partial sum may hold 2^24 / max|product| products
// exactly: 1024 for int8 x int8 (|p| <= 2^14), 16384 for int8 x int4 (|p| <= 2^10); each warp
// adds 16 per step. int4 stages hold two steps (512 K: two W boxes of 256 K each, four A boxes), so that the
// per-stage costs (waits, arrives, bookkeeping) are spread over twice the MMAs.
template <bool W4>
struct GemvCfg {
    static constexpr int SPW = W4 ? 2 : 1;           // K-steps per warp per stage
    static constexpr int kBK = BK * SPW;             // K per stage
    static constexpr int kW8 = RW * (W4 ? kBK / 2 : kBK);
    static constexpr int kA8 = NT * kBK;
    static constexpr int kStage = kW8 + kA8;
    static constexpr int S8 = W4 ? 8 : 10;   // stages in the ring
    static constexpr int kStagesPerChunk = (W4 ? 16384 : 1024) / (16 * SPW);
    static constexpr int kOffRed = S8 * kStage;
    static constexpr int kOffBar = kOffRed + kRedBytes;
    static constexpr int kSmem = kOffBar + 16 * S8 + 16 + 1024;
};

__device__ __forceinline__ void mma_m16n8k16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];\n" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];\n" : "=h"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void named_barrier(int id, int threads) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(threads) : "memory");
}

template <bool W4>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_mma_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_a,
                    int M, int N, int K, Epilogue ep) {
    using C = GemvCfg<W4>;
    constexpr int S8 = C::S8, kW8 = C::kW8, kStage = C::kStage, kStagesPerChunk = C::kStagesPerChunk;
    constexpr int SPW = C::SPW, kBK = C::kBK;
    constexpr int kOffRed = C::kOffRed, kOffBar = C::kOffBar;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t sraw = smem_u32(smem_raw);
    const uint32_t sbase = (sraw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (sbase - sraw);
    const uint32_t bar_full = sbase + kOffBar;
    const uint32_t bar_empty = bar_full + 8 * S8;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + 16 * S8);
    int32_t* red = reinterpret_cast<int32_t*>(smem + kOffRed);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S8; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kComputeWarps);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmap_w)) : "memory");
        asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmap_a)) : "memory");
    }
    __syncthreads();

    const int tiles = (N + RW - 1) / RW;
    const int KB = (K + kBK - 1) / kBK;
    const int my_tiles = (int)blockIdx.x < tiles ? (tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int total_g = my_tiles * KB;
    // each CTA starts its K sweep at its own block, spreading activation reads over L2
    const int k_rot = (int)(((long long)blockIdx.x * KB) / gridDim.x);

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            int i = 0, kb = 0;
            for (int g = 0; g < total_g; ++g) {
                const int n0 = ((int)blockIdx.x + i * (int)gridDim.x) * RW;
                const int s = g % S8;
                if (!mbar_wait(bar_empty + 8 * s, (uint32_t)(((g / S8) & 1) ^ 1), abort_flag, kErrProducer,
                               &g_gemv_mma_error))
                    break;
                const int kx = (kb + k_rot >= KB ? kb + k_rot - KB : kb + k_rot) * kBK;
                const uint32_t dst = sbase + s * kStage;
                mbar_expect_tx(bar_full + 8 * s, kStage);
                // W: two boxes of 64 rows x 128 bytes (int8: 256 K; int4: 512 K packed)
                const int wx = W4 ? kx / 2 : kx;
                tma_load_2d(dst, &tmap_w, wx, n0, bar_full + 8 * s);
                tma_load_2d(dst + RW * BKH, &tmap_w, wx + BKH, n0, bar_full + 8 * s);
#pragma unroll
                for (int b = 0; b < kBK / BKH; ++b)   // A: 16 tokens x 128 K per box
                    tma_load_2d(dst + kW8 + b * (NT * BKH), &tmap_a, kx + b * BKH, 0, bar_full + 8 * s);
                if (++kb == KB) { kb = 0; ++i; }
            }
        }
    } else {
        // ---------------------------------------------------------------- compute warps
        const int ks = warp - 1;          // K-step of each stage: bytes [16 ks, 16 ks + 16)
        const int ct = threadIdx.x - 32;  // 0 .. 511
        const int g8 = lane >> 2, t = lane & 3;
        const int half = ks >> 3, kc = ks & 7;   // which 128-byte box, 16-byte chunk in its rows
        // weight row 8j + g and token rows g, g+8 at chunk kc of box `half` (swizzled), word t.
        // int4: the step's 16 K are 8 packed bytes, half of chunk ks / 2 of the first W box; lane
        // quad t takes bytes 2t, 2t + 1 of them (K 4t .. 4t + 3). The warp's second step (K-step
        // ks + 16 of the 512-K stage) sits one W box (64 x 128 bytes) and two A boxes further.
        // Row 8j + g lies 1024 j bytes past row g: the swizzle depends on (row & 7) = g only.
        const uint32_t w_base = W4 ? sw128(g8, ks >> 1) + 8 * (ks & 1) + 2 * t : half * (RW * BKH) + sw128(g8, kc) + 4 * t;
        const uint32_t a_off0 = kW8 + half * (NT * BKH) + sw128(g8, kc) + 4 * t;
        const uint32_t a_off1 = kW8 + half * (NT * BKH) + sw128(g8 + 8, kc) + 4 * t;
        for (int i = ct; i < 2 * NT * RWP; i += 32 * kComputeWarps) red[i] = 0;
        named_barrier(1, 32 * kComputeWarps);
        // Epilogue outputs of this thread: tokens em and em + 8, row er of each tile. The token
        // scales are loaded once here; the channel scales at the tile's end (loading them at the
        // tile's first stage measured slower).
        const int em = ct / RW, er = ct % RW;
        float esa0 = 0.0f, esa1 = 0.0f, esw = 0.0f;
        int eza0 = 0, eza1 = 0, ecs = 0;
        if (!ep.out_i32) {
            if (em < M) {
                esa0 = __ldg(ep.s_a + (ep.a_per_row ? em : 0));
                if (ep.z_a) eza0 = __ldg(ep.z_a + (ep.a_per_row ? em : 0));
            }
            if (em + 8 < M) {
                esa1 = __ldg(ep.s_a + (ep.a_per_row ? em + 8 : 0));
                if (ep.z_a) eza1 = __ldg(ep.z_a + (ep.a_per_row ? em + 8 : 0));
            }
        }
        int tot[8][4];
        float part[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) tot[j][e] = 0, part[j][e] = 0.0f;
        int kb = 0, ti = 0, in_chunk = 0, g = 0;
        for (; g < total_g; ++g) {
            const int s = g % S8;
            // warp-uniform: the whole warp leaves together when a wait gives up (abort)
            if (!__all_sync(0xffffffffu, mbar_wait(bar_full + 8 * s, (uint32_t)((g / S8) & 1), abort_flag,
                                                   kErrConvFull, &g_gemv_mma_error)))
                break;
            const uint32_t st = sbase + s * kStage;
#pragma unroll
            for (int u = 0; u < SPW; ++u) {   // steps in turn: 17 warps leave at most 96 registers a thread
                uint32_t wq[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    wq[j] = W4 ? lds16(st + w_base + 1024 * j + u * (RW * BKH)) : lds32(st + w_base + 1024 * j);
                const uint32_t aq0 = lds32(st + a_off0 + u * (2 * NT * BKH));
                const uint32_t aq1 = lds32(st + a_off1 + u * (2 * NT * BKH));
                uint32_t a[4], b[8][2];
                cvt_word(aq0, a[0], a[2]);     // token row g:   k pair (2t,2t+1) and (8+2t,9+2t)
                cvt_word(aq1, a[1], a[3]);     // token row g+8
#pragma unroll
                for (int j = 0; j < 8; ++j) {   // weight row 8j + g
                    if constexpr (W4)
                        cvt_int4x4<0x4140u>(wq[j], b[j][0], b[j][1]);
                    else
                        cvt_word(wq[j], b[j][0], b[j][1]);
                }
                if (u == SPW - 1) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_empty + 8 * s);   // every loaded word has been consumed
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) mma_m16n8k16(part[j], a, b[j][0], b[j][1]);
            }
            const bool tile_end = (kb == KB - 1);
            // int4: one exact fp32 chunk covers any tile (K <= kStagesPerChunk * kBK, checked by
            // gemv_mma_supports), so the partials go to the tile sums directly at the tile's end
            if (!W4 && (++in_chunk == kStagesPerChunk || tile_end)) {
                in_chunk = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        tot[j][e] += __float2int_rn(part[j][e]);
                        part[j][e] = 0.0f;
                    }
            }
            if (tile_end) {
                // add the sixteen K-step partials of the tile in shared memory (integer adds),
                // in the tile-sum buffer of this tile's parity
                int32_t* rb = red + (ti & 1) * (NT * RWP);
#pragma unroll
                for (int j = 0; j < 8; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int m = g8 + (e >> 1) * 8;            // c0,c1: token g; c2,c3: token g+8
                        const int r = 8 * j + 2 * t + (e & 1);
                        if constexpr (W4) {
                            atomicAdd(rb + m * RWP + r, __float2int_rn(part[j][e]));
                            part[j][e] = 0.0f;
                        } else {
                            atomicAdd(rb + m * RWP + r, tot[j][e]);
                            tot[j][e] = 0;
                        }
                    }
                named_barrier(1, 32 * kComputeWarps);
                // Read and re-zero this thread's two sums. The buffer is next written at tile
                // ti + 2, after every thread has passed the tile barrier of tile ti + 1.
                const int i0 = em * RWP + er, i1 = i0 + 8 * RWP;
                const int v0 = rb[i0], v1 = rb[i1];
                rb[i0] = 0;
                rb[i1] = 0;
                const int n = ((int)blockIdx.x + ti * (int)gridDim.x) * RW + er;
                if (n < N && !ep.out_i32) {
                    esw = __ldg(ep.s_w + (ep.w_per_row ? n : 0));
                    if (ep.z_a) ecs = __ldg(ep.colsum + n);
                }
                if (n < N) {
                    if (ep.out_i32) {
                        if (em < M) ep.out_i32[(int64_t)em * N + n] = v0;
                        if (em + 8 < M) ep.out_i32[(int64_t)(em + 8) * N + n] = v1;
                    } else {
                        if (em < M)
                            epi_store(ep, (int64_t)em * N + n,
                                      epi_bias(ep, __fmul_rn(__int2float_rn(v0 - eza0 * ecs), __fmul_rn(esa0, esw)), n));
                        if (em + 8 < M)
                            epi_store(ep, (int64_t)(em + 8) * N + n,
                                      epi_bias(ep, __fmul_rn(__int2float_rn(v1 - eza1 * ecs), __fmul_rn(esa1, esw)), n));
                    }
                }
            }
            if (++kb == KB) { kb = 0; ++ti; }
        }
        // After an abort: pass the tile-end barriers still ahead, so that no compute warp
        // waits at one forever.
        for (; g < total_g; ++g) {
            if (kb == KB - 1) named_barrier(1, 32 * kComputeWarps);
            if (++kb == KB) kb = 0;
        }
    }
    __syncthreads();
    if (*abort_flag) {
        const long long t0 = clock64();
        while (clock64() - t0 < (1LL << 22)) __nanosleep(1000);
    }
}

}  // namespace

bool gemv_mma_supports(int64_t M, int64_t N, int64_t K, bool w4) {
    if (!(M >= 1 && M <= NT && N >= 1 && N < (1LL << 31) && K >= 16 && (K % (w4 ? 32 : 16)) == 0)) return false;
    if (w4 && K > (int64_t)GemvCfg<true>::kStagesPerChunk * GemvCfg<true>::kBK) return false;   // one chunk per tile
    const int64_t tiles = (N + RW - 1) / RW;
    const int64_t kb = (K + BK - 1) / BK;
    return tiles * kb < (1LL << 31);
}

template <bool W4>
static cudaError_t launch_gemv_mma_t(const int8_t* qa, const void* qw, int64_t M, int64_t N, int64_t K,
                                     const Epilogue& ep, cudaStream_t stream) {
    using C = GemvCfg<W4>;
    CUtensorMap mw, ma;
    // int4: the packed weights are an int8 byte matrix [N, K / 2]; one box covers 256 K
    if (!make_tma_map_i8(&mw, static_cast<const int8_t*>(qw), N, W4 ? K / 2 : K, RW, BKH, true) ||
        !make_tma_map_i8(&ma, qa, M, K, NT, BKH, true))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(gemv_mma_kernel<W4>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    const int64_t tiles = (N + RW - 1) / RW;
    const int sms = device_sm_count();
    const int grid = (int)(tiles < sms ? tiles : sms);
    gemv_mma_kernel<W4><<<grid, kThreads, C::kSmem, stream>>>(mw, ma, (int)M, (int)N, (int)K, ep);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_gemv_mma(const int8_t* qa, const void* qw, int64_t M, int64_t N, int64_t K, const Epilogue& ep,
                            cudaStream_t stream, bool w4) {
    if (!gemv_mma_supports(M, N, K, w4)) return cudaErrorNotSupported;
    return w4 ? launch_gemv_mma_t<true>(qa, qw, M, N, K, ep, stream)
              : launch_gemv_mma_t<false>(qa, qw, M, N, K, ep, stream);
}

cudaError_t read_and_clear_gemv_mma_error(uint32_t* code) {
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_gemv_mma_error, sizeof(v));
    if (e != cudaSuccess) return e;
    *code = v;
    if (v) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_gemv_mma_error, &zero, sizeof(zero));
    }
    return e;
}

}  // namespace q8
