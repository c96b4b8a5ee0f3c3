// Decode-shaped integer GEMM (M <= 16 tokens) + dequantization epilogue on the
// warp-level fp16 tensor-core instruction mma.sync.m16n8k16 (fp32 accumulate).
//
// With a handful of tokens the layer is a stream of the weight codes from HBM
// with little arithmetic per byte. The weights go HBM -> shared memory by TMA
// (a ring of stages per SM; an int8 stage is 64 rows x 256 bytes of K, fetched as
// two 128-byte boxes, which streams DRAM better than 128-byte row pieces) and
// shared memory -> registers by ordinary loads;
// each warp converts its code fragments to fp16 in registers and feeds them
// straight to the MMA, so converted data never goes back through shared memory.
// (The int8 MMA of this GPU runs at a fraction of the fp16 rate, too low for
// this stream.)
//
// Exactness: the codes, offset weight codes and their products are exact in fp16 /
// fp32, and each fp32 accumulator is drained to int32 before its integer sum can
// pass 2^24 (the weight format note below), so the result is the exact integer
// dot product.
//
// int8 K order inside a stage: compute warp s (of 16) owns the 16 K values
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

// Weight format: int8 codes or int4 codes packed two per byte. A weight code enters the MMA
// offset to a non-negative integer and scaled to an fp16 subnormal, made by one lop3 (mask the
// code, flip its sign bit), with no fp16 arithmetic:
//   int8: (w + 128) 2^-24, exact in the 10-bit subnormal significand;
//   int4: (n + 8) 2^-24; a high nibble, four bits up, is (n + 8) 2^-20 and meets the token code
//         a / 16 (exact in fp16) instead of a.
// Every product is then an integer times 2^-24 (|a (w + 128)| <= 32640, |a (n + 8)| <= 1920),
// so an fp32 partial is exact while it holds at most 2^24 / that many products: 512 (int8; the
// warp drains its partials to int32 every 32 K-steps) or, for int4, a whole tile (K / 16
// products for K <= 139810). A drained partial is scaled by 2^24 (exact), and at the end
// c sum_k a_k (c = 128 or 8), the token's code sum taken with dp4a while a CTA runs its first
// tile, is subtracted. The int32 sums may wrap; the result, |sum_k a_k w_k| < 2^31, is exact.
// int8: a stage is 256 K (two W boxes of 64 rows x 128 bytes, two A boxes), one K-step per warp.
// int4: a stage is kW4Segs segments of 512 K; a segment is two W boxes (64 rows x 128 packed
// bytes = 256 K each) and four A boxes, and warp ks owns the 32 K [32 ks, 32 ks + 32) of each
// segment: one 4-byte load per weight row (8 codes) feeds two K-steps. Longer stages spread the
// per-stage costs (waits, arrives, bookkeeping) over more MMAs.
constexpr int kW4Segs = 2;
template <bool W4>
struct GemvCfg {
    static constexpr int SPW = W4 ? 2 * kW4Segs : 1;   // K-steps per warp per stage
    static constexpr int kBK = BK * SPW;             // K per stage
    static constexpr int kW8 = RW * (W4 ? kBK / 2 : kBK);
    static constexpr int kA8 = NT * kBK;
    static constexpr int kStage = kW8 + kA8;
    static constexpr int S8 = W4 ? 8 / kW4Segs : 10;   // stages in the ring
    static constexpr int kStagesPerChunk = 512 / 16;   // int8
    static constexpr int kOffRed = S8 * kStage;
    static constexpr int kOffBar = kOffRed + kRedBytes;
    static constexpr int kOffSum = kOffBar + 16 * S8 + 16;    // token code sums [16]
    static constexpr int kSmem = kOffSum + 4 * NT + 1024;
};

__device__ __forceinline__ void mma_m16n8k16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Programmatic dependent launch: the decode kernels are launched so that they may start while
// the kernel before them on the stream is still running. Nothing they read is touched before
// griddep_wait(), which returns once the preceding kernel has completed and its writes are
// visible (at once when there is none), with one exception: when the launch follows the
// library's own activation quantizer of the same layer (Epilogue::pdl_early_weights, set only by
// q8_linear and the host-buffer layer, which launch the two back to back and check that the
// quantizer's outputs do not overlap the weight operands), the first ring of weight (and scale)
// boxes is loaded before the wait. That quantizer writes only codes, scales and zero points, and
// it was itself launched without the attribute, so every earlier kernel has completed before it
// started and before this kernel could start.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];\n" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "r"(addr) : "memory");
    return v;
}

// int8 weights: lo = {byte 0, byte 2} and hi = {byte 1, byte 3} of w as the fp16 subnormals
// (w + 128) 2^-24: (x & 0x00FF00FF) ^ 0x00800080.
__device__ __forceinline__ void cvt_int8_subnormal(uint32_t w, uint32_t& lo, uint32_t& hi) {
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;\n" : "=r"(lo) : "r"(w), "r"(0x00FF00FFu), "r"(0x00800080u));
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;\n" : "=r"(hi) : "r"(w >> 8), "r"(0x00FF00FFu), "r"(0x00800080u));
}

// int4 weights (step of one 32-bit word w: bytes 0 and 2, i.e. the caller shifts w right by 8
// for bytes 1 and 3): lo = {low nibble of byte 0, of byte 2} and hi = {high nibbles}, as fp16
// subnormals: (x & 0x000F000F) ^ 0x00080008 is (n + 8) 2^-24, and the high nibbles four bits up
// are (n + 8) 2^-20. One lop3 each.
__device__ __forceinline__ void cvt_int4_subnormal(uint32_t w, uint32_t& lo, uint32_t& hi) {
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;\n" : "=r"(lo) : "r"(w), "r"(0x000F000Fu), "r"(0x00080008u));
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;\n" : "=r"(hi) : "r"(w), "r"(0x00F000F0u), "r"(0x00800080u));
}

// The token codes that meet step U of cvt_int4_subnormal: q.x holds K 8t .. 8t + 3, q.y K 8t + 4
// .. 8t + 7. lo = {x.byte 2U, y.byte 2U} as fp16 a (meeting the low nibbles), hi = {x.byte 2U+1,
// y.byte 2U+1} as fp16 a / 16 (meeting the high nibbles, which carry a factor 16). With
// 0x6480 | (byte ^ 0x80) = 1024 + 128 + a: minus 1152 gives a; / 16 - 72 gives a / 16, exactly.
__device__ __forceinline__ void cvt_tokens_w4(int U, uint2 q, uint32_t& lo, uint32_t& hi) {
    uint32_t p, l, h;
    asm("prmt.b32 %0, %1, %2, %3;\n" : "=r"(p) : "r"(q.x), "r"(q.y), "r"(U ? 0x7632u : 0x5410u));
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;\n" : "=r"(l) : "r"(p), "r"(0x00FF00FFu), "r"(0x64806480u));
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;\n" : "=r"(h) : "r"(p >> 8), "r"(0x00FF00FFu), "r"(0x64806480u));
    asm("sub.rn.f16x2 %0, %1, %2;\n" : "=r"(lo) : "r"(l), "r"(0x64806480u));
    asm("fma.rn.f16x2 %0, %1, %2, %3;\n" : "=r"(hi) : "r"(h), "r"(0x2C002C00u), "r"(0xD480D480u));
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
    constexpr int kBK = C::kBK;
    constexpr int kOffRed = C::kOffRed, kOffBar = C::kOffBar;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t sraw = smem_u32(smem_raw);
    const uint32_t sbase = (sraw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (sbase - sraw);
    const uint32_t bar_full = sbase + kOffBar;
    const uint32_t bar_empty = bar_full + 8 * S8;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + 16 * S8);
    int32_t* red = reinterpret_cast<int32_t*>(smem + kOffRed);
    int32_t* tok_sum = reinterpret_cast<int32_t*>(smem + C::kOffSum);

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
        if (lane == 0 && ep.selftest_wait_cycles == 0) {
            // The first ring's worth of stages gets its weight boxes (before the wait on the
            // quantizer where the launch allows it), its token boxes after the wait (the ring is
            // empty, so no empty-slot waits).
            const int pre = total_g < S8 ? total_g : S8;
            auto kx_of = [&](int kb) { return (kb + k_rot >= KB ? kb + k_rot - KB : kb + k_rot) * kBK; };
            auto load_w = [&](int g, int kb, int i) {
                const int n0 = ((int)blockIdx.x + i * (int)gridDim.x) * RW;
                const int s = g % S8;
                const int wx = W4 ? kx_of(kb) / 2 : kx_of(kb);
                // W: boxes of 64 rows x 128 bytes (int8: 128 K; int4: 256 K packed)
#pragma unroll
                for (int b = 0; b < kW8 / (RW * BKH); ++b)
                    tma_load_2d(sbase + s * kStage + b * (RW * BKH), &tmap_w, wx + b * BKH, n0, bar_full + 8 * s);
            };
            auto load_a = [&](int g, int kb) {
                const int s = g % S8;
#pragma unroll
                for (int b = 0; b < kBK / BKH; ++b)   // A: 16 tokens x 128 K per box
                    tma_load_2d(sbase + s * kStage + kW8 + b * (NT * BKH), &tmap_a, kx_of(kb) + b * BKH, 0,
                                bar_full + 8 * s);
            };
            int i = 0, kb = 0;
            if (!ep.pdl_early_weights) griddep_wait();
            for (int g = 0; g < pre; ++g) {
                mbar_expect_tx(bar_full + 8 * (g % S8), kStage);
                load_w(g, kb, i);
                if (++kb == KB) { kb = 0; ++i; }
            }
            griddep_wait();
            for (int g = 0; g < pre; ++g) load_a(g, g % KB);
            for (int g = pre; g < total_g; ++g) {
                const int s = g % S8;
                if (!mbar_wait(bar_empty + 8 * s, (uint32_t)(((g / S8) & 1) ^ 1), abort_flag, kErrProducer,
                               &g_gemv_mma_error))
                    break;
                mbar_expect_tx(bar_full + 8 * s, kStage);
                load_w(g, kb, i);
                load_a(g, kb);
                if (++kb == KB) { kb = 0; ++i; }
            }
        }
    } else {
        // ---------------------------------------------------------------- compute warps
        const int ks = warp - 1;          // K-step of each stage: bytes [16 ks, 16 ks + 16)
        const int ct = threadIdx.x - 32;  // 0 .. 511
        const int g8 = lane >> 2, t = lane & 3;
        const int half = ks >> 3, kc = ks & 7;   // which 128-byte box, 16-byte chunk in its rows
        // int8: weight row 8j + g and token rows g, g+8 at chunk kc of box `half` (swizzled), word t.
        // int4 (per 512-K segment): the warp's 32 K are chunk ks & 7 of W box ks >> 3 (16 packed
        // bytes a row); lane quad t takes word t, K 8t .. 8t + 7: bytes 0, 1 (K 8t .. 8t + 3) for
        // the first K-step, bytes 2, 3 for the second. The same K of the tokens are 8 bytes at 8t
        // of the warp's 32 bytes in A box ks >> 2: chunk 2 (ks & 3) + t / 2, offset 8 (t & 1).
        // Row 8j + g lies 1024 j bytes past row g: the swizzle depends on (row & 7) = g only.
        const uint32_t w_base = W4 ? (ks >> 3) * (RW * BKH) + sw128(g8, ks & 7) + 4 * t
                                   : half * (RW * BKH) + sw128(g8, kc) + 4 * t;
        const uint32_t a_off0 = W4 ? kW8 + (ks >> 2) * (NT * BKH) + sw128(g8, 2 * (ks & 3) + (t >> 1)) + 8 * (t & 1)
                                   : kW8 + half * (NT * BKH) + sw128(g8, kc) + 4 * t;
        const uint32_t a_off1 = W4 ? kW8 + (ks >> 2) * (NT * BKH) + sw128(g8 + 8, 2 * (ks & 3) + (t >> 1)) + 8 * (t & 1)
                                   : kW8 + half * (NT * BKH) + sw128(g8 + 8, kc) + 4 * t;
        for (int i = ct; i < 2 * NT * RWP; i += 32 * kComputeWarps) red[i] = 0;
        if (ct < NT) tok_sum[ct] = 0;
        named_barrier(1, 32 * kComputeWarps);
        griddep_wait();   // the token scales and zero points below come from the quantizer
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
        int sum0 = 0, sum1 = 0;        // first tile: code sums of tokens g, g + 8 over this lane's K
        int esum0 = 0, esum1 = 0;      // code sums of the epilogue tokens em, em + 8
        const long long full_limit = ep.selftest_wait_cycles > 0 ? ep.selftest_wait_cycles : kTimeoutCycles;
        for (; g < total_g; ++g) {
            const int s = g % S8;
            // warp-uniform: the whole warp leaves together when a wait gives up (abort)
            if (!__all_sync(0xffffffffu, mbar_wait(bar_full + 8 * s, (uint32_t)((g / S8) & 1), abort_flag,
                                                   kErrConvFull, &g_gemv_mma_error, 0, full_limit)))
                break;
            const uint32_t st = sbase + s * kStage;
            if constexpr (W4) {
#pragma unroll
                for (int sg = 0; sg < kW4Segs; ++sg) {   // segments in turn: 17 warps leave at most 96 registers a thread
                    uint32_t wq[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) wq[j] = lds32(st + w_base + 1024 * j + sg * (2 * RW * BKH));
                    const uint2 aq0 = lds64(st + a_off0 + sg * (4 * NT * BKH));
                    const uint2 aq1 = lds64(st + a_off1 + sg * (4 * NT * BKH));
                    if (ti == 0) {
                        sum0 = __dp4a((int)aq0.x, 0x01010101, __dp4a((int)aq0.y, 0x01010101, sum0));
                        sum1 = __dp4a((int)aq1.x, 0x01010101, __dp4a((int)aq1.y, 0x01010101, sum1));
                    }
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        // step u: weight bytes u, u + 2 of each word (K 8t + 2u, + 1 | 8t + 4 + 2u, + 1)
                        uint32_t a[4], b[8][2];
                        cvt_tokens_w4(u, aq0, a[0], a[2]);   // token row g
                        cvt_tokens_w4(u, aq1, a[1], a[3]);   // token row g+8
#pragma unroll
                        for (int j = 0; j < 8; ++j)    // weight row 8j + g
                            cvt_int4_subnormal(u ? wq[j] >> 8 : wq[j], b[j][0], b[j][1]);
                        if (sg == kW4Segs - 1 && u == 0) {
                            __syncwarp();
                            if (lane == 0) mbar_arrive(bar_empty + 8 * s);   // every loaded word has been consumed
                        }
#pragma unroll
                        for (int j = 0; j < 8; ++j) mma_m16n8k16(part[j], a, b[j][0], b[j][1]);
                    }
                }
            } else {
                uint32_t wq[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) wq[j] = lds32(st + w_base + 1024 * j);
                const uint32_t aq0 = lds32(st + a_off0);
                const uint32_t aq1 = lds32(st + a_off1);
                if (ti == 0) {
                    sum0 = __dp4a((int)aq0, 0x01010101, sum0);
                    sum1 = __dp4a((int)aq1, 0x01010101, sum1);
                }
                uint32_t a[4], b[8][2];
                cvt_word(aq0, a[0], a[2]);     // token row g:   k pair (2t,2t+1) and (8+2t,9+2t)
                cvt_word(aq1, a[1], a[3]);     // token row g+8
#pragma unroll
                for (int j = 0; j < 8; ++j) cvt_int8_subnormal(wq[j], b[j][0], b[j][1]);   // weight row 8j + g
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_empty + 8 * s);   // every loaded word has been consumed
#pragma unroll
                for (int j = 0; j < 8; ++j) mma_m16n8k16(part[j], a, b[j][0], b[j][1]);
            }
            const bool tile_end = (kb == KB - 1);
            // int4: the fp32 partials are exact over the whole tile (K bounded in
            // gemv_mma_supports), so they go to the tile sums directly at the tile's end
            if (!W4 && (++in_chunk == kStagesPerChunk || tile_end)) {
                in_chunk = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        tot[j][e] += __float2int_rn(part[j][e] * 16777216.0f);
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
                            atomicAdd(rb + m * RWP + r, __float2int_rn(part[j][e] * 16777216.0f));
                            part[j][e] = 0.0f;
                        } else {
                            atomicAdd(rb + m * RWP + r, tot[j][e]);
                            tot[j][e] = 0;
                        }
                    }
                if (ti == 0) {   // token code sums: over the lane quad, then over the warps
                    sum0 += __shfl_xor_sync(0xffffffffu, sum0, 1);
                    sum0 += __shfl_xor_sync(0xffffffffu, sum0, 2);
                    sum1 += __shfl_xor_sync(0xffffffffu, sum1, 1);
                    sum1 += __shfl_xor_sync(0xffffffffu, sum1, 2);
                    if (t == 0) {
                        atomicAdd(tok_sum + g8, sum0);
                        atomicAdd(tok_sum + g8 + 8, sum1);
                    }
                }
                named_barrier(1, 32 * kComputeWarps);
                if (ti == 0) {
                    esum0 = tok_sum[em];
                    esum1 = tok_sum[em + 8];
                }
                // Read and re-zero this thread's two sums. The buffer is next written at tile
                // ti + 2, after every thread has passed the tile barrier of tile ti + 1.
                const int i0 = em * RWP + er, i1 = i0 + 8 * RWP;
                constexpr uint32_t kOffset = W4 ? 8u : 128u;
                const int v0 = (int)((uint32_t)rb[i0] - kOffset * (uint32_t)esum0);
                const int v1 = (int)((uint32_t)rb[i1] - kOffset * (uint32_t)esum1);
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


// ------------------------------------------------------------------------------------------
// Block-scaled int8 weights (one E8M0 scale per row and group of G = 32 or 128 K), M <= 16.
// The int8 stream design (64-row tiles, sixteen compute warps) with 512-K stages: warp ks owns
// the 32 K [32 ks, 32 ks + 32) of every stage, one group for G = 32 (inside one for G = 128),
// so each row's scale is read and converted once per stage; a lane's 8-byte load of a row
// (K 32 ks + 8 t .. + 8) feeds two MMA K-steps (bytes 0-3, then 4-7), and the tokens take the
// same K order. Per stage the TMA also brings the tile's four scale words of the stage's K
// (64 rows x 16 bytes, the 4-byte words viewed as a byte matrix [words, 4 N]).
// A weight fragment enters the MMA as the fp16 values q * s (exact: the codes are exact in
// fp16 and s = 2^(e - 127) scales them without rounding for e = 103 .. 136). The MMA sums the
// exact products in fp32 over the tile, so the result is not bit-reproducible against an
// exactly rounded sum. At the tile's end the sixteen per-warp partials are added in a fixed
// order (warp w + 8 onto warp w in shared memory, then the eight sums in warp order), so every
// run gives the same bits.
constexpr int kMxBK = 512;                        // K per stage
constexpr int kMxS8 = 4;                          // stages in the ring
constexpr int kMxSf = RW * 4 * 4;                 // scale bytes per stage: 64 rows x 4 words
constexpr int kMxStage = RW * kMxBK + NT * kMxBK; // 32 KB of weights + 8 KB of tokens
constexpr int kMxOffSf = kMxS8 * kMxStage;
constexpr int kMxOffRed = kMxOffSf + kMxS8 * kMxSf;
constexpr int kMxRedBytes = 8 * NT * RWP * 4;     // fp32 [8 warps][16 tokens][72 (64 rows)]
constexpr int kMxOffBar = kMxOffRed + kMxRedBytes;
constexpr int kMxSmem = kMxOffBar + 16 * kMxS8 + 16 + 1024;

__device__ __forceinline__ uint32_t lds8(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u8 %0, [%1];\n" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__global__ void __launch_bounds__(kThreads, 1)
    gemv_mx_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_a,
                   const __grid_constant__ CUtensorMap tmap_sf, int M, int N, int K, int G, Epilogue ep) {
    constexpr int S8 = kMxS8;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t sraw = smem_u32(smem_raw);
    const uint32_t sbase = (sraw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (sbase - sraw);
    const uint32_t bar_full = sbase + kMxOffBar;
    const uint32_t bar_empty = bar_full + 8 * S8;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMxOffBar + 16 * S8);
    float* red = reinterpret_cast<float*>(smem + kMxOffRed);

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
        asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmap_sf)) : "memory");
    }
    __syncthreads();

    const int tiles = (N + RW - 1) / RW;
    const int KB = (K + kMxBK - 1) / kMxBK;
    const int my_tiles = (int)blockIdx.x < tiles ? (tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int total_g = my_tiles * KB;
    const int k_rot = (int)(((long long)blockIdx.x * KB) / gridDim.x);
    const int wshift = G == 32 ? 7 : 9;   // K per scale word: 4 G

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            // As in the int8 kernel: the first ring's weight and scale boxes (before the wait on
            // the quantizer where the launch allows it), its token boxes after the wait.
            const int pre = total_g < S8 ? total_g : S8;
            auto kx_of = [&](int kb) { return (kb + k_rot >= KB ? kb + k_rot - KB : kb + k_rot) * kMxBK; };
            auto load_w = [&](int g, int kb, int i) {
                const int n0 = ((int)blockIdx.x + i * (int)gridDim.x) * RW;
                const int s = g % S8, kx = kx_of(kb);
#pragma unroll
                for (int b = 0; b < kMxBK / BKH; ++b)   // W: 64 rows x 128 K per box
                    tma_load_2d(sbase + s * kMxStage + b * (RW * BKH), &tmap_w, kx + b * BKH, n0, bar_full + 8 * s);
                // scales: words kx / 4G .. + 3, bytes [4 n0, 4 n0 + 256) of each
                tma_load_2d(sbase + kMxOffSf + s * kMxSf, &tmap_sf, 4 * n0, kx >> wshift, bar_full + 8 * s);
            };
            auto load_a = [&](int g, int kb) {
                const int s = g % S8, kx = kx_of(kb);
#pragma unroll
                for (int b = 0; b < kMxBK / BKH; ++b)   // A: 16 tokens x 128 K per box
                    tma_load_2d(sbase + s * kMxStage + RW * kMxBK + b * (NT * BKH), &tmap_a, kx + b * BKH, 0,
                                bar_full + 8 * s);
            };
            int i = 0, kb = 0;
            if (!ep.pdl_early_weights) griddep_wait();
            for (int g = 0; g < pre; ++g) {
                mbar_expect_tx(bar_full + 8 * (g % S8), kMxStage + kMxSf);
                load_w(g, kb, i);
                if (++kb == KB) { kb = 0; ++i; }
            }
            griddep_wait();
            for (int g = 0; g < pre; ++g) load_a(g, g % KB);
            for (int g = pre; g < total_g; ++g) {
                const int s = g % S8;
                if (!mbar_wait(bar_empty + 8 * s, (uint32_t)(((g / S8) & 1) ^ 1), abort_flag, kErrProducer,
                               &g_gemv_mma_error))
                    break;
                mbar_expect_tx(bar_full + 8 * s, kMxStage + kMxSf);
                load_w(g, kb, i);
                load_a(g, kb);
                if (++kb == KB) { kb = 0; ++i; }
            }
        }
    } else {
        // ---------------------------------------------------------------- compute warps
        const int ks = warp - 1;          // K of each stage: [32 ks, 32 ks + 32)
        const int ct = threadIdx.x - 32;  // 0 .. 511
        const int g8 = lane >> 2, t = lane & 3;
        // weight row 8j + g8 and token rows g8, g8 + 8: 8 bytes at byte 8 (t & 1) of chunk
        // 2 (ks & 3) + t / 2 of box ks / 4 (swizzled); row 8j + g8 lies 1024 j bytes past row g8
        const int box = ks >> 2, chunk = 2 * (ks & 3) + (t >> 1);
        const uint32_t w_base = box * (RW * BKH) + sw128(g8, chunk) + 8 * (t & 1);
        const uint32_t a_off0 = RW * kMxBK + box * (NT * BKH) + sw128(g8, chunk) + 8 * (t & 1);
        const uint32_t a_off1 = RW * kMxBK + box * (NT * BKH) + sw128(g8 + 8, chunk) + 8 * (t & 1);
        // scale byte of weight row r for this warp's 32 K: G = 32: group ks of the stage's 16, word
        // ks / 4 of the four, byte ks % 4; G = 128: group ks / 4 of the stage's 4 (kx is a multiple
        // of 512), word 0, byte ks / 4
        const uint32_t sf_off = (uint32_t)((G == 32 ? (ks >> 2) * (RW * 4) + (ks & 3) : (ks >> 2)) + g8 * 4);
        const int em = ct / RW, er = ct % RW;   // epilogue outputs: tokens em, em + 8 of row er
        float esa0 = 0.0f, esa1 = 0.0f;
        griddep_wait();   // the token scales come from the quantizer
        if (em < M) esa0 = __ldg(ep.s_a + (ep.a_per_row ? em : 0));
        if (em + 8 < M) esa1 = __ldg(ep.s_a + (ep.a_per_row ? em + 8 : 0));
        float part[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) part[j][e] = 0.0f;
        int kb = 0, ti = 0, g = 0;
        for (; g < total_g; ++g) {
            const int s = g % S8;
            if (!__all_sync(0xffffffffu, mbar_wait(bar_full + 8 * s, (uint32_t)((g / S8) & 1), abort_flag,
                                                   kErrConvFull, &g_gemv_mma_error)))
                break;
            const uint32_t st = sbase + s * kMxStage;
            const uint32_t sfa = sbase + kMxOffSf + s * kMxSf + sf_off;
            uint2 wq[8];
            uint32_t h[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) wq[j] = lds64(st + w_base + 1024 * j);
#pragma unroll
            for (int j = 0; j < 8; ++j) h[j] = lds8(sfa + 32 * j);   // row 8j + g8
            const uint2 aq0 = lds64(st + a_off0);
            const uint2 aq1 = lds64(st + a_off1);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * s);   // every loaded word has been consumed
#pragma unroll
            for (int j = 0; j < 8; ++j) h[j] = scale_f16x2(min(h[j], 136u));
#pragma unroll
            for (int u = 0; u < 2; ++u) {  // K-step u: bytes 4u .. 4u + 3 of every 8-byte load
                uint32_t a[4], b[8][2];
                cvt_word(u ? aq0.y : aq0.x, a[0], a[2]);     // token row g8
                cvt_word(u ? aq1.y : aq1.x, a[1], a[3]);     // token row g8 + 8
#pragma unroll
                for (int j = 0; j < 8; ++j) {  // weight row 8j + g8: q exactly, then q * s (exact)
                    cvt_word(u ? wq[j].y : wq[j].x, b[j][0], b[j][1]);
                    b[j][0] = hmul2(b[j][0], h[j]);
                    b[j][1] = hmul2(b[j][1], h[j]);
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) mma_m16n8k16(part[j], a, b[j][0], b[j][1]);
            }
            if (kb == KB - 1) {
                // Tile end: warps 0-7 write their partials, warps 8-15 add theirs onto warp
                // ks - 8's, then every thread sums the eight slots of its two outputs in order.
                float* slot = red + (ks & 7) * (NT * RWP);
#pragma unroll
                for (int j = 0; j < 8; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int m = g8 + (e >> 1) * 8, r = 8 * j + 2 * t + (e & 1);
                        if (ks < 8) slot[m * RWP + r] = part[j][e];
                    }
                named_barrier(1, 32 * kComputeWarps);
                if (ks >= 8) {
#pragma unroll
                    for (int j = 0; j < 8; ++j)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int m = g8 + (e >> 1) * 8, r = 8 * j + 2 * t + (e & 1);
                            slot[m * RWP + r] = __fadd_rn(slot[m * RWP + r], part[j][e]);
                        }
                }
#pragma unroll
                for (int j = 0; j < 8; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) part[j][e] = 0.0f;
                named_barrier(1, 32 * kComputeWarps);
                float T0 = 0.0f, T1 = 0.0f;
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    T0 = __fadd_rn(T0, red[w * (NT * RWP) + em * RWP + er]);
                    T1 = __fadd_rn(T1, red[w * (NT * RWP) + (em + 8) * RWP + er]);
                }
                const int n = ((int)blockIdx.x + ti * (int)gridDim.x) * RW + er;
                if (n < N) {
                    if (em < M) epi_store(ep, (int64_t)em * N + n, epi_bias(ep, __fmul_rn(T0, esa0), n));
                    if (em + 8 < M) epi_store(ep, (int64_t)(em + 8) * N + n, epi_bias(ep, __fmul_rn(T1, esa1), n));
                }
                named_barrier(1, 32 * kComputeWarps);   // the slots are free for the next tile
            }
            if (++kb == KB) { kb = 0; ++ti; }
        }
        // After an abort: pass the tile-end barriers still ahead, so that no compute warp
        // waits at one forever.
        for (; g < total_g; ++g) {
            if (kb == KB - 1) {
                named_barrier(1, 32 * kComputeWarps);
                named_barrier(1, 32 * kComputeWarps);
                named_barrier(1, 32 * kComputeWarps);
            }
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

// Launch with programmatic stream serialization: the kernel may start before the preceding
// kernel on the stream has finished (it waits for it with griddepcontrol.wait where needed).
template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*kernel)(KArgs...), int grid, int threads, int smem, cudaStream_t stream,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

bool gemv_mma_supports(int64_t M, int64_t N, int64_t K, bool w4) {
    if (!(M >= 1 && M <= NT && N >= 1 && N < (1LL << 31) && K >= 16 && (K % (w4 ? 32 : 16)) == 0)) return false;
    if (w4) {   // int4: each warp's fp32 partial must stay exact over a tile: products 1920 at most
        const int64_t stages = (K + GemvCfg<true>::kBK - 1) / GemvCfg<true>::kBK;
        if (stages * 16 * GemvCfg<true>::SPW * 1920 >= (1LL << 24)) return false;
    }
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
    e = launch_pdl(gemv_mma_kernel<W4>, grid, kThreads, C::kSmem, stream, mw, ma, (int)M, (int)N, (int)K, ep);
    if (e != cudaSuccess) return e;
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_gemv_mma(const int8_t* qa, const void* qw, int64_t M, int64_t N, int64_t K, const Epilogue& ep,
                            cudaStream_t stream, bool w4) {
    if (!gemv_mma_supports(M, N, K, w4)) return cudaErrorNotSupported;
    return w4 ? launch_gemv_mma_t<true>(qa, qw, M, N, K, ep, stream)
              : launch_gemv_mma_t<false>(qa, qw, M, N, K, ep, stream);
}

bool gemv_mx_supports(int64_t M, int64_t N, int64_t K, int G, const void* sf) {
    // the scale words are fetched by TMA as a byte matrix [words, 4 N]: 16-byte row pitch and base
    if (!(M >= 1 && M <= NT && N >= 1 && N < (1LL << 29) && K >= 16 && K % 16 == 0 && (G == 32 || G == 128) &&
          K % G == 0 && N % 4 == 0 && (reinterpret_cast<uintptr_t>(sf) & 15) == 0))
        return false;
    const int64_t tiles = (N + RW - 1) / RW;
    const int64_t kb = (K + kMxBK - 1) / kMxBK;
    return tiles * kb < (1LL << 31);
}

cudaError_t launch_gemv_mx(const int8_t* qa, const int8_t* qw, const uint32_t* sf, int G, int64_t M, int64_t N,
                           int64_t K, const Epilogue& ep, cudaStream_t stream) {
    if (!gemv_mx_supports(M, N, K, G, sf)) return cudaErrorNotSupported;
    const int64_t words = (K / G + 3) / 4;
    CUtensorMap mw, ma, ms;
    if (!make_tma_map_i8(&mw, qw, N, K, RW, BKH, true) || !make_tma_map_i8(&ma, qa, M, K, NT, BKH, true) ||
        !make_tma_map_i8(&ms, reinterpret_cast<const int8_t*>(sf), words, 4 * N, 4, RW * 4))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(gemv_mx_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMxSmem);
    if (e != cudaSuccess) return e;
    const int64_t tiles = (N + RW - 1) / RW;
    const int sms = device_sm_count();
    const int grid = (int)(tiles < sms ? tiles : sms);
    e = launch_pdl(gemv_mx_kernel, grid, kThreads, kMxSmem, stream, mw, ma, ms, (int)M, (int)N, (int)K, G, ep);
    if (e != cudaSuccess) return e;
    note_launch();
    return cudaGetLastError();
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
