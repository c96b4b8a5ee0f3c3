// Integer GEMM + dequantization epilogue on the Blackwell tcgen05 tensor cores.
//
// sm_103a has no integer tcgen05 MMA in this toolkit (kind::i8 is rejected by
// ptxas for the target), so the exact INT8 x INT8 -> INT32 product is carried
// by the fp16 MMA (kind::f16, fp32 accumulator in tensor memory):
//  - every int8 code is exactly representable in fp16 and every product of two
//    codes (|p| <= 2^14) is exact;
//  - the fp32 accumulator only ever holds a sum of at most 1024 products, so
//    every partial sum is an integer of magnitude <= 1024 * 2^14 = 2^24, which
//    fp32 represents exactly;
//  - after each 1024-deep chunk of K, the chunk sum is read out of tensor
//    memory, converted to int32 and added into INT32 registers, and the next
//    chunk starts from zero in the other accumulator buffer.
// The int32 sum of exact chunk sums is the exact dot product. Whether the
// hardware adds the integer-valued products without loss inside a chunk is
// checked bit for bit against the CPU oracle (including worst-case codes).
//
// Data flow per CTA (persistent, one CTA per SM, 128 x 256 output tiles,
// 16 warps):
//   warp 0       TMA: int8 tiles of A [128 x 64] and W [256 x 64] -> smem staging ring
//   warp 1       allocates tensor memory and issues tcgen05.mma (one thread)
//   warps 2..7   convert int8 staging -> fp16 operand ring (128-byte swizzled,
//                K-major, the layout the MMA descriptors read)
//   warps 8..15  drain each fp32 chunk accumulator into INT32 registers (128
//                per thread) and, at the end of a tile, apply the epilogue
//                and store y, while the MMA fills the other buffer
// The drain warpgroups hold the 128 x 256 INT32 accumulator (half the
// register file), so registers are moved to them with setmaxnreg: the two
// other warpgroups drop to 72 per thread and the drain warpgroups rise to
// 184 (2*128*72 + 2*128*184 = 65536 = 512 threads x 128 at launch).
// Every wait on an mbarrier is bounded: a wait that runs out sets the device
// error word and an abort flag, and the kernel winds down and frees its tensor
// memory instead of hanging.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "q8_internal.h"
#include "q8_tc_ptx.cuh"

namespace q8 {

// Device error word of this kernel (one per device): bits name the bounded wait that gave up.
static __device__ unsigned int g_tc_error;

namespace {

using namespace tc;

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;              // K elements per pipeline stage
constexpr int S8 = 4;               // int8 staging stages
constexpr int S16 = 2;              // fp16 operand stages
constexpr int KB_PER_CHUNK = 16;    // 16 * 64 = 1024 K per exact fp32 chunk
constexpr int kConv = 192;          // converter threads, warps 2..7
constexpr int kDrainWarps = 8;      // warps 8..15
constexpr int kThreads = 512;
constexpr int kRegsLow = 72, kRegsHigh = 184;   // setmaxnreg split, see above
constexpr int kTmemCols = 512;      // two 128 x 256 fp32 accumulator buffers

constexpr int kA8 = BM * BK, kB8 = BN * BK, kStage8 = kA8 + kB8;                  // 24 KB
constexpr int kA16 = BM * BK * 2, kB16 = BN * BK * 2, kStage16 = kA16 + kB16;     // 48 KB
constexpr int kOffStage8 = S16 * kStage16;
constexpr int kOffBar = kOffStage8 + S8 * kStage8;
constexpr int kBarBytes = 8 * (2 * S8 + 2 * S16 + 4) + 16;
constexpr int kSmem = kOffBar + kBarBytes + 1024;  // + alignment slack

// Instruction descriptor of kind::f16: fp16 A and B, both K-major, fp32 D, M = 128, N = 256.
constexpr uint32_t kIdesc = idesc_f16(BM, BN);

struct TileGeom {
    int num_m, num_n, tiles;
};

// Tile order: bands of 8 M-tiles, N-tiles swept inside a band, so that the
// CTAs running at the same time share A rows and W columns in L2.
__device__ __forceinline__ void tile_coords(const TileGeom& tg, int t, int& m0, int& n0) {
    constexpr int GM = 8;
    const int band = t / (GM * tg.num_n);
    const int within = t - band * GM * tg.num_n;
    const int rows = min(GM, tg.num_m - band * GM);
    const int mt = band * GM + within % rows;
    const int nt = within / rows;
    m0 = mt * BM;
    n0 = nt * BN;
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_w,
                   int M, int N, int K, Epilogue ep) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full8 = sbase + kOffBar;
    const uint32_t bar_empty8 = bar_full8 + 8 * S8;
    const uint32_t bar_full16 = bar_empty8 + 8 * S8;
    const uint32_t bar_empty16 = bar_full16 + 8 * S16;
    const uint32_t bar_accfull = bar_empty16 + 8 * S16;
    const uint32_t bar_accempty = bar_accfull + 16;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * (2 * S8 + 2 * S16 + 4));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S8; ++s) {
            mbar_init(bar_full8 + 8 * s, 1);
            mbar_init(bar_empty8 + 8 * s, kConv / 32);
        }
        for (int s = 0; s < S16; ++s) {
            mbar_init(bar_full16 + 8 * s, kConv);
            mbar_init(bar_empty16 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_accfull + 8 * b, 1);
            mbar_init(bar_accempty + 8 * b, kDrainWarps);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmap_a)) : "memory");
        asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmap_w)) : "memory");
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    TileGeom tg;
    tg.num_m = (M + BM - 1) / BM;
    tg.num_n = (N + BN - 1) / BN;
    tg.tiles = tg.num_m * tg.num_n;
    const int KB = (K + BK - 1) / BK;
    const int CPT = (KB + KB_PER_CHUNK - 1) / KB_PER_CHUNK;  // chunks per tile
    const int my_tiles = (int)blockIdx.x < tg.tiles ? (tg.tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int total_g = my_tiles * KB;   // host guarantees this fits in int

    if (warp < 8) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kRegsLow));
      if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0 && ep.selftest_wait_cycles == 0) {
            int i = 0, kb = 0, m0 = 0, n0 = 0;
            for (int g = 0; g < total_g; ++g) {
                if (kb == 0) tile_coords(tg, blockIdx.x + i * gridDim.x, m0, n0);
                const int s = g % S8;
                const uint32_t par = (uint32_t)((g / S8) & 1);
                if (!mbar_wait(bar_empty8 + 8 * s, par ^ 1u, abort_flag, kErrProducer, &g_tc_error)) break;
                const uint32_t dst = sbase + kOffStage8 + s * kStage8;
                mbar_expect_tx(bar_full8 + 8 * s, kStage8);
                tma_load_2d(dst, &tmap_a, kb * BK, m0, bar_full8 + 8 * s);
                tma_load_2d(dst + kA8, &tmap_w, kb * BK, n0, bar_full8 + 8 * s);
                if (++kb == KB) { kb = 0; ++i; }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int kb = 0, c = 0;   // k-block within the tile, running chunk index
            for (int g = 0; g < total_g; ++g) {
                const bool first = (kb % KB_PER_CHUNK) == 0;
                const bool last = (kb % KB_PER_CHUNK) == KB_PER_CHUNK - 1 || kb == KB - 1;
                const int buf = c & 1;
                if (first) {
                    if (!mbar_wait(bar_accempty + 8 * buf, (uint32_t)(((c >> 1) & 1) ^ 1), abort_flag, kErrMmaAcc, &g_tc_error))
                        break;
                    tc_fence_after();
                }
                const int s = g % S16;
                if (!mbar_wait(bar_full16 + 8 * s, (uint32_t)((g / S16) & 1), abort_flag, kErrMmaFull, &g_tc_error)) break;
                tc_fence_after();
                const uint32_t a_addr = sbase + s * kStage16;
                const uint64_t adesc = smem_desc_sw128(a_addr);
                const uint64_t bdesc = smem_desc_sw128(a_addr + kA16);
                const uint32_t d = tmem_base + (uint32_t)(buf * BN);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
                    // advance 16 fp16 = 32 bytes along K inside the swizzled rows
                    mma_f16(d, adesc + (uint64_t)(kk * 2), bdesc + (uint64_t)(kk * 2), kIdesc, (first && kk == 0) ? 0u : 1u);
                }
                mma_commit(bar_empty16 + 8 * s);
                if (last) {
                    mma_commit(bar_accfull + 8 * buf);
                    ++c;
                }
                if (++kb == KB) kb = 0;
            }
        }
      } else {
        // ---------------------------------------------------------------- converters
        // 1536 16-byte int8 chunks per stage ([A 128 rows | W 256 rows] x 4
        // chunks of each 64-byte staging row), 8 per thread. The fp16 stage is
        // [A | W] in one run of 128-byte swizzled rows, so row r of the
        // combined staging tile lands at sw128(r, .) for both operands.
        const int ct = threadIdx.x - 64;
        // Chunk j of this thread is idx = ct + 192 j: staging byte idx * 16, fp16 row
        // r = ct / 4 + 48 j with (r & 7) independent of j, so both addresses are a
        // per-thread base plus a constant stride (3072 and 6144 bytes).
        const int r0 = ct >> 2, c0 = ct & 3;
        const uint32_t src0 = (uint32_t)(ct * 16);
        const uint32_t dst0 = sw128(r0, 2 * c0);
        const uint32_t dst1 = sw128(r0, 2 * c0 + 1);
        const long long full_limit = ep.selftest_wait_cycles > 0 ? ep.selftest_wait_cycles : kTimeoutCycles;
        for (int g = 0; g < total_g; ++g) {
            const int s8 = g % S8, s16 = g % S16;
            if (!mbar_wait(bar_full8 + 8 * s8, (uint32_t)((g / S8) & 1), abort_flag, kErrConvFull, &g_tc_error, 0,
                           full_limit))
                break;
            const uint32_t st8 = sbase + kOffStage8 + s8 * kStage8 + src0;
            uint4 in[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) in[j] = lds128(st8 + kConv * 16 * j);
            if (!mbar_wait(bar_empty16 + 8 * s16, (uint32_t)(((g / S16) & 1) ^ 1), abort_flag, kErrConvEmpty, &g_tc_error)) break;
            const uint32_t st16 = sbase + s16 * kStage16;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint4 o0, o1;
                cvt_word(in[j].x, o0.x, o0.y);
                cvt_word(in[j].y, o0.z, o0.w);
                cvt_word(in[j].z, o1.x, o1.y);
                cvt_word(in[j].w, o1.z, o1.w);
                sts128(st16 + dst0 + 6144 * j, o0);
                sts128(st16 + dst1 + 6144 * j, o1);
            }
            fence_proxy_async_smem();
            mbar_arrive(bar_full16 + 8 * s16);
            // Release the staging slot only now: the converted values were built from
            // every loaded register, so the shared-memory reads have completed. (An
            // arrive right after issuing the loads let the next TMA write, which is
            // not ordered after pending generic-proxy reads, land first.)
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty8 + 8 * s8);
        }
      }
    } else {
        // ---------------------------------------------------------------- drain + epilogue
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kRegsHigh));
        const int quarter = warp & 3;            // TMEM lane quarter this warp may access
        const int col_half = (warp - 8) >> 2;    // 0: columns 0..127, 1: 128..255
        int acc[128];
#pragma unroll
        for (int c = 0; c < 128; ++c) acc[c] = 0;
        const int chunks_total = my_tiles * CPT;
        int ti = 0, cc = 0;    // tile (in this CTA's sequence) and chunk within it
        for (int c = 0; c < chunks_total; ++c, (++cc == CPT ? (cc = 0, ++ti) : 0)) {
            const int buf = c & 1;
            if (!mbar_wait(bar_accfull + 8 * buf, (uint32_t)((c >> 1) & 1), abort_flag, kErrDrain, &g_tc_error)) break;
            tc_fence_after();
            const uint32_t taddr =
                tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(buf * BN + col_half * 128);
            // The first chunk of a tile starts the sums afresh (keep = 0); written
            // without a branch, which keeps the 128 sums in registers.
            const int keep = cc != 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t v[32];
                tmem_ld32(taddr + j * 32, v);
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    acc[j * 32 + e] = acc[j * 32 + e] * keep + __float2int_rn(__uint_as_float(v[e]));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_accempty + 8 * buf);
            if (cc != CPT - 1) continue;   // (the loop header advances cc / ti)
            // Last chunk of the tile: epilogue.
            int m0, n0;
            tile_coords(tg, blockIdx.x + ti * gridDim.x, m0, n0);
            const int m = m0 + quarter * 32 + lane;
            const int nb = n0 + col_half * 128;
            if (m < M) {
                if (ep.out_i32) {
                    int32_t* row = ep.out_i32 + (int64_t)m * N;
#pragma unroll
                    for (int e = 0; e < 128; ++e)
                        if (nb + e < N) row[nb + e] = acc[e];
                } else {
                    const float sa = ep.s_a[ep.a_per_row ? m : 0];
                    const int za = ep.z_a ? ep.z_a[ep.a_per_row ? m : 0] : 0;
                    float* row = ep.y + (int64_t)m * N;
                    const bool vec = ((N & 3) == 0);
                    // per-channel scales and column sums four at a time when they are 16-byte aligned
                    const bool vsw = ep.w_per_row && vec && ((reinterpret_cast<uintptr_t>(ep.s_w) & 15) == 0);
                    const bool vcs = ep.z_a && vec && ((reinterpret_cast<uintptr_t>(ep.colsum) & 15) == 0);
#pragma unroll
                    for (int e4 = 0; e4 < 32; ++e4) {
                        const int n = nb + e4 * 4;
                        const bool full = n + 3 < N;
                        float sw4[4];
                        int cs4[4] = {0, 0, 0, 0};
                        if (vsw && full) {
                            const float4 t = __ldg(reinterpret_cast<const float4*>(ep.s_w + n));
                            sw4[0] = t.x; sw4[1] = t.y; sw4[2] = t.z; sw4[3] = t.w;
                        } else {
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                sw4[q] = __ldg(ep.s_w + (ep.w_per_row ? (n + q < N ? n + q : 0) : 0));
                        }
                        if (ep.z_a) {
                            if (vcs && full) {
                                const int4 t = __ldg(reinterpret_cast<const int4*>(ep.colsum + n));
                                cs4[0] = t.x; cs4[1] = t.y; cs4[2] = t.z; cs4[3] = t.w;
                            } else {
#pragma unroll
                                for (int q = 0; q < 4; ++q) cs4[q] = __ldg(ep.colsum + (n + q < N ? n + q : 0));
                            }
                        }
                        float o[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int corr = acc[e4 * 4 + q] - za * cs4[q];
                            o[q] = __fmul_rn(__int2float_rn(corr), __fmul_rn(sa, sw4[q]));
                            if (ep.bias) o[q] = __fadd_rn(o[q], __ldg(ep.bias + (n + q < N ? n + q : 0)));
                        }
                        if (ep.out_kind != kOutF32) {
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                if (n + q < N) epi_store(ep, (int64_t)m * N + n + q, o[q]);
                        } else if (vec && n + 3 < N) {
                            *reinterpret_cast<float4*>(row + n) = make_float4(o[0], o[1], o[2], o[3]);
                        } else {
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                if (n + q < N) row[n + q] = o[q];
                        }
                    }
                }
            }
        }
    }

    // Wind down. On an abort, give copies and MMAs already in flight time to land
    // (bounded) before tensor memory is released.
    __syncthreads();
    if (*abort_flag) {
        const long long t0 = clock64();
        while (clock64() - t0 < (1LL << 22)) __nanosleep(1000);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace

namespace {
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D int8 tensor map over a row-major [rows, K] matrix, box [box_rows, box_k],
// with the given shared-memory swizzle, zero fill outside.
bool make_map_impl(CUtensorMap* map, const int8_t* base, int64_t rows, int64_t K, int box_rows, int box_k,
                   CUtensorMapSwizzle swizzle) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K};
    cuuint32_t box[2] = {(cuuint32_t)box_k, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int sm_count_impl() {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 0 ? sms : 1;
}

}  // namespace

bool make_tma_map_i8(CUtensorMap* map, const int8_t* base, int64_t rows, int64_t K, int box_rows, int box_k,
                     bool swizzle128) {
    return make_map_impl(map, base, rows, K, box_rows, box_k,
                         swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
}

bool make_tma_map_f16(CUtensorMap* map, const uint16_t* base, int64_t rows, int64_t K, int box_rows, int box_k) {
    auto enc = get_encode();
    if (!enc || ((K * 2) % 16) != 0 || (reinterpret_cast<uintptr_t>(base) & 15) != 0) return false;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(K * 2)};
    cuuint32_t box[2] = {(cuuint32_t)box_k, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_tma_map_i8_sw64(CUtensorMap* map, const int8_t* base, int64_t rows, int64_t K, int box_rows) {
    return make_map_impl(map, base, rows, K, box_rows, 64, CU_TENSOR_MAP_SWIZZLE_64B);
}

bool make_tma_map_out(CUtensorMap* map, void* base, int kind, int64_t rows, int64_t cols) {
    auto enc = get_encode();
    CUtensorMapDataType dt;
    int esz;
    switch (kind) {
        case kMapF32: dt = CU_TENSOR_MAP_DATA_TYPE_FLOAT32; esz = 4; break;
        case kMapI32: dt = CU_TENSOR_MAP_DATA_TYPE_INT32; esz = 4; break;
        case kMapBF16: dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16; esz = 2; break;
        case kMapI8: dt = CU_TENSOR_MAP_DATA_TYPE_UINT8; esz = 1; break;
        default: return false;
    }
    if (!enc || ((cols * esz) % 16) != 0 || (reinterpret_cast<uintptr_t>(base) & 15) != 0) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(cols * esz)};
    cuuint32_t box[2] = {(cuuint32_t)(128 / esz), 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, dt, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int device_sm_count() { return sm_count_impl(); }

bool gemm_tc_supports(int64_t M, int64_t N, int64_t K) {
    if (!(M >= 1 && N >= 1 && K >= 16 && (K % 16) == 0 && M < (1LL << 31) && N < (1LL << 31))) return false;
    // per-CTA k-block counters are 32-bit: bound the tiles x k-blocks of one CTA
    const int64_t tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    const int64_t kb = (K + BK - 1) / BK;
    return tiles < (1LL << 30) && tiles * kb < (1LL << 31);
}

cudaError_t launch_gemm_tc(const int8_t* qa, const int8_t* qw, int64_t M, int64_t N, int64_t K,
                           const Epilogue& ep, cudaStream_t stream) {
    if (!gemm_tc_supports(M, N, K)) return cudaErrorNotSupported;
    CUtensorMap ma, mw;
    if (!make_tma_map_i8(&ma, qa, M, K, BM, BK) || !make_tma_map_i8(&mw, qw, N, K, BN, BK)) return cudaErrorInvalidValue;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int64_t tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    const int sms = device_sm_count();
    const int grid = (int)(tiles < sms ? tiles : sms);
    gemm_tc_kernel<<<grid, kThreads, kSmem, stream>>>(ma, mw, (int)M, (int)N, (int)K, ep);
    note_launch();
    return cudaGetLastError();
}

cudaError_t read_and_clear_gemm_tc_error(uint32_t* code) {
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_tc_error, sizeof(v));
    if (e != cudaSuccess) return e;
    *code = v;
    if (v) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(zero));
    }
    return e;
}

}  // namespace q8
