// Integer GEMM + dequantization epilogue on CTA pairs (tcgen05 cta_group::2).
//
// The exactness argument is the one of the single-CTA kernel (q8_gemm_tc.cu):
// int8 codes are exact in fp16, each fp32 TMEM accumulator holds at most 1024
// products (|partial| <= 2^24), and chunk sums are added in INT32 registers.
//
// Why pairs: the single-CTA kernel streams every operand byte through shared
// memory four times (TMA write, conversion read, fp16 write, MMA read) and is
// bound by shared-memory bandwidth, not by the tensor core. Two CTAs of a
// cluster share one 256 x 256 MMA tile: each CTA holds and converts 128 rows
// of A and 128 rows (one half) of W, and the pair's tensor cores exchange the
// W halves, so per SM the shared-memory traffic per FLOP drops by a third.
//
//   both CTAs   warp 0       TMA: int8 A [128 x 64] (own rows) and W [128 x 64]
//                            (own half of the 256 columns) -> staging ring
//               warps 2..7   int8 -> fp16 into the swizzled operand ring; each
//                            warp then arrives on the even CTA's stage barrier
//               warps 8..15  drain their own TMEM rows (128 x 256) per 1024-K chunk
//                            into INT32 registers, epilogue, store y
//   even CTA    warp 1       issues tcgen05.mma.cta_group::2 (M = 256, N = 256) and
//                            commits to the barriers of both CTAs
//   both CTAs   warp 1       allocates / frees TMEM collectively with the peer
// setmaxnreg: 72 registers for warpgroups 0-1, 184 for the drain warpgroups.
// Waits on mbarriers are bounded (device error word + abort flag).
//
// Weight formats: int8 codes (above), packed int4 codes (same roles; 16384-K exact chunks)
// and block-scaled int8 codes (each weight enters the MMA as the exact fp16 value q * s, the
// accumulator runs in fp32 over the whole K and is drained once per tile: warps 2..11
// convert, warps 12..15 drain, each taking its 256 columns in two halves).
// K split: for grids that fill at most half of the resident clusters the host splits K into
// slices; each (tile, slice) unit adds its INT32 partial sums into the output's storage by
// TMA reduce-add, and the host runs the dequantization epilogue in place afterwards.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <type_traits>

#include "q8_internal.h"
#include "q8_tc_ptx.cuh"

namespace q8 {

static __device__ unsigned int g_tc2_error;

// Two fp32 values (bit patterns) as a bf16x2 word, low half first, round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo, uint32_t hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
    return *reinterpret_cast<const uint32_t*>(&v);
}

// Four fp32 values (bit patterns) as int8 codes clamp(rint(v / s), -127, 127), packed.
__device__ __forceinline__ uint32_t pack_codes4(uint4 v, float s) {
    auto code = [&](uint32_t b) {
        return (uint32_t)(min(max(__float2int_rn(__fdiv_rn(__uint_as_float(b), s)), -127), 127) & 0xFF);
    };
    return code(v.x) | (code(v.y) << 8) | (code(v.z) << 16) | (code(v.w) << 24);
}

namespace {

using namespace tc;

constexpr int BM = 256;             // rows of the pair tile (128 per CTA)
constexpr int BMH = 128;
constexpr int BN = 256;             // columns of the pair tile (W rows; 128 per CTA)
constexpr int BNH = 128;
constexpr int BK = 64;
constexpr int kThreads = 512;
constexpr int kTmemCols = 512;      // two 128 x 256 fp32 accumulator buffers per CTA

constexpr int kA8 = BMH * BK;                                                     // 8 KB int8 A staging
constexpr int kA16 = BMH * BK * 2, kB16 = BNH * BK * 2, kStage16 = kA16 + kB16;   // 32 KB
constexpr int kEpiBytes = 32 * 128;    // per drain warp: a 32 x 128-byte output block (TMA store source)
constexpr uint32_t kIdesc = idesc_f16(BM, BN);
constexpr uint16_t kPairMask = 0x3;
// Block-scaled weights whose scale words cannot be staged by TMA (N % 4 != 0 or a scale array
// that is not 16-byte aligned): the converters load them from global memory this many stages ahead.
constexpr int kSfAhead = 2;
constexpr int kSfStage = BNH * 4;   // scale words of one stage's 128 weight rows, staged by TMA

// Weight formats (WF): int8 codes (staged as 128 rows x 64 bytes per CTA), int4 codes packed
// two per byte (128 rows x 32 bytes), or block-scaled int8 codes (kWMx: as int8, plus one E8M0
// scale per row and group of G K elements). An exact fp32 TMEM chunk holds 2^24 / max|product|
// products: 1024 K for int8 x int8 (|p| <= 2^14), 16384 K for int8 x int4 (|p| <= 2^10).
// Block-scaled weights enter the MMA as the fp16 values q * s (exact: s = 2^-24 .. 2^9), so the
// products are no longer integers and TMEM accumulates the whole K in fp32 (one chunk).
// Warp roles: warp 0 TMA, warp 1 MMA (even CTA) or relay (odd CTA), then kConvWarps converter
// warps, then (block-scaled weights with fp16 activations) a warp that issues the activation
// loads and an idle warp, then kDrainWarps drain warps (a multiple of 4: warp w reads TMEM lanes
// 32 (w % 4) ..). The int8 and int4 formats
// drain every exact chunk and take 6 converters and 8 drains; the block-scaled formats drain once
// per tile and take 4 drains (each drain warp then reads its 256 accumulator columns in two
// halves) and 10 converters, or 8 with fp16 activations (two weight chunks per thread and stage).
// Registers: warps [0, kDrain0) shrink to kRegsLow and the drain warps grow to kRegsHigh;
// setmaxnreg acts on whole warpgroups, so kDrain0 is a multiple of 4, and kDrain0 * 32 *
// kRegsLow + kDrainWarps * 32 * kRegsHigh <= 512 * 128, the registers the block is launched with.
// Activation codes as fp16 values (kWA16, kW4A16, kWMxA16): TMA writes the A half of each fp16
// operand stage directly (the 128-byte swizzle of a [128 x 64] fp16 box is the K-major layout of
// the UMMA descriptors), the staging ring holds the weights only, and the converters convert W.
// The freed staging bytes give the operand ring a fifth stage. The converters write int8 and
// int4 weight codes alike in pair order (each group of four K as K 0, 2, 1, 3: cvt_word's
// pairs); with kWA16 (codes in K order, also a public input format) the int8 weight bytes are
// permuted into K order first, with kW4A16 and kWMxA16 the fp16 codes arrive in pair order.
template <int WF>
struct PairCfg {
    static constexpr bool W4 = WF == kWInt4 || WF == kW4A16;
    static constexpr bool MX = WF == kWMx || WF == kWMxA16;
    static constexpr bool A16 = WF == kWA16 || WF == kW4A16 || WF == kWMxA16;
    static constexpr int S16 = A16 ? 5 : 4;                   // fp16 operand stages (32 KB each)
    static constexpr int kOffStage8 = S16 * kStage16;
    // block-scaled weights with fp16 activations: eight converter warps (two weight chunks per
    // thread and stage), then the warp that issues the activation loads, an idle warp, then the drains
    static constexpr int kConvWarps = MX ? (A16 ? 8 : 10) : 6;
    static constexpr int kDrainWarps = MX ? 4 : 8;
    static constexpr int kDrain0 = 16 - kDrainWarps;                // first drain warp
    static constexpr int kConvT = 32 * kConvWarps;                  // converter threads
    static constexpr int kRegsLow = MX ? 104 : 72, kRegsHigh = 184;
    // tile order: bands of 8 M-tiles with fp16 activation codes (an A block is twice the bytes of
    // a W block, which favours taller bands), 4 with int8 codes (measured at prefill16k)
    static constexpr int kBand = A16 ? 8 : 4;
    static_assert(2 + kConvWarps <= kDrain0, "warp roles above the block");
    // setmaxnreg acts on whole warpgroups: warps [0, kDrain0) shrink, warps [kDrain0, 16) grow
    static_assert(kDrain0 % 4 == 0, "the register split must fall on a warpgroup boundary");
    static_assert(kDrain0 * 32 * kRegsLow + kDrainWarps * 32 * kRegsHigh <= kThreads * 128,
                  "register split above the launch's registers");
    static_assert(kDrainWarps % 4 == 0 && (kConvT / 4) % 8 == 0, "drain warps cover whole TMEM lane quarters");
    static constexpr int kB8 = BNH * (W4 ? BK / 2 : BK);
    static constexpr int kStage8 = (A16 ? 0 : kA8) + kB8;     // 16 KB (int8), 12 KB (int4); fp16 A: 8 KB, 4 KB
    static constexpr int S8 = (W4 || (MX && A16)) ? 5 : 4;    // staging stages
    static constexpr int KB_PER_CHUNK = W4 ? 256 : MX ? (1 << 30) : 16;
    static constexpr int kOffSf = kOffStage8 + S8 * kStage8;   // block-scaled: S8 x 128 scale words
    static constexpr int kOffEpi = (kOffSf + (MX ? S8 * kSfStage : 0) + 1023) / 1024 * 1024;
    static constexpr int kOffBar = kOffEpi + kDrainWarps * kEpiBytes;
    static constexpr int kBarBytes = 8 * (2 * S8 + 3 * S16 + 4) + 16;
    static constexpr int kSmem = kOffBar + kBarBytes + 1024;
    static_assert(kStage16 % 1024 == 0 && kStage8 % 1024 == 0 && kOffEpi % 1024 == 0,
                  "stages and the swizzled output buffers must keep 1024-byte alignment");
    static_assert(kSmem <= 227 * 1024, "above the shared memory of one CTA");
};

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];\n" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

struct PairGeom {
    int num_m, num_n, tiles, band;   // band: M-tiles per band of the tile order (pair_coords)
};

// Pair tiles in bands of tg.band M-tiles, N swept inside a band. The clusters of one wave run
// consecutive tiles at about the same K, so each A and W block a wave touches is read from DRAM
// about once per wave: band A blocks and (clusters / band) W blocks.
__device__ __forceinline__ void pair_coords(const PairGeom& tg, int t, int& m0, int& n0) {
    const int GM = tg.band;
    const int band = t / (GM * tg.num_n);
    const int within = t - band * GM * tg.num_n;
    const int rows = min(GM, tg.num_m - band * GM);
    m0 = (band * GM + within % rows) * BM;
    n0 = (within / rows) * BN;
}

// Work units: tiles [0, n_full) whole, each later tile as ksplit K slices of kb_part k-blocks
// (the host makes the k-blocks divide evenly). A sliced unit's INT32 partial sums are added into
// an int32 view of the output by TMA reduce-add; the host zeroes those tiles first and applies
// the epilogue to them afterwards.
struct PairUnits {
    int n_full, ksplit, kb_all, kb_part;
    __device__ __forceinline__ void get(int u, int& tile, int& k0, int& kbn, bool& part) const {
        if (u < n_full) {
            tile = u; k0 = 0; kbn = kb_all; part = false;
        } else {
            const int v = u - n_full;
            tile = n_full + v / ksplit; kbn = kb_part; k0 = (v % ksplit) * kb_part; part = true;
        }
    }
};

template <int WF>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_tc2_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_w,
                    const __grid_constant__ CUtensorMap tmap_out, const __grid_constant__ CUtensorMap tmap_acc,
                    const __grid_constant__ CUtensorMap tmap_sf, int tma_out, int sf_tma, int M, int N, int K,
                    int n_full, int ksplit, Epilogue ep) {
    using C = PairCfg<WF>;
    constexpr bool W4 = C::W4, MX = C::MX, A16 = C::A16;
    constexpr int S8 = C::S8, S16 = C::S16, kStage8 = C::kStage8, KB_PER_CHUNK = C::KB_PER_CHUNK;
    constexpr int kOffStage8 = C::kOffStage8;
    constexpr int kOffEpi = C::kOffEpi, kOffBar = C::kOffBar;
    constexpr int kConvWarps = C::kConvWarps, kDrainWarps = C::kDrainWarps;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t sraw = smem_u32(smem_raw);
    const uint32_t sbase = (sraw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (sbase - sraw);
    const uint32_t bar_full8 = sbase + kOffBar;
    const uint32_t bar_empty8 = bar_full8 + 8 * S8;
    const uint32_t bar_full16 = bar_empty8 + 8 * S8;     // used in the even CTA: its converter warps + relay
                                                         // (+ the A TMA's bytes for A16)
    const uint32_t bar_empty16 = bar_full16 + 8 * S16;   // both CTAs: the pair MMA's commit
    const uint32_t bar_accfull = bar_empty16 + 8 * S16;  // both CTAs: the pair MMA's commit
    const uint32_t bar_accempty = bar_accfull + 16;      // used in the even CTA: 2 x 8 drain warps
    const uint32_t bar_conv16 = bar_accempty + 16;       // used in the odd CTA: its converter warps (+ A TMA)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * (2 * S8 + 3 * S16 + 4));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank();            // 0: issues the MMA; 1: peer
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S8; ++s) {
            mbar_init(bar_full8 + 8 * s, 1);
            mbar_init(bar_empty8 + 8 * s, kConvWarps);
        }
        for (int s = 0; s < S16; ++s) {
            mbar_init(bar_full16 + 8 * s, kConvWarps + 1 + (A16 ? 1 : 0));
            mbar_init(bar_empty16 + 8 * s, 1);
            mbar_init(bar_conv16 + 8 * s, kConvWarps + (A16 ? 1 : 0));
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_accfull + 8 * b, 1);
            mbar_init(bar_accempty + 8 * b, 2 * kDrainWarps);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmap_a)) : "memory");
        asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmap_w)) : "memory");
    }
    if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tc_fence_before();
    cluster_sync();   // barriers of both CTAs initialised, TMEM allocated in both
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    PairGeom tg;
    tg.num_m = (M + BM - 1) / BM;
    tg.num_n = (N + BN - 1) / BN;
    tg.tiles = tg.num_m * tg.num_n;
    tg.band = C::kBand;
    const int cluster = (int)(blockIdx.x >> 1), nclusters = (int)(gridDim.x >> 1);
    const int KB = (K + BK - 1) / BK;   // k-blocks of a whole tile
    const PairUnits un{n_full, ksplit, KB, KB / ksplit};
    const int units = n_full + (tg.tiles - n_full) * ksplit;
    const int my_units = cluster < units ? (units - 1 - cluster) / nclusters + 1 : 0;
    const int my_full = cluster < n_full ? (n_full - 1 - cluster) / nclusters + 1 : 0;
    const int total_g = my_full * KB + (my_units - my_full) * un.kb_part;   // stages of this cluster

    if (warp < C::kDrain0) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(C::kRegsLow));
      if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            int i = 0, kb = 0, m0 = 0, n0 = 0, k0 = 0, kbn = 0;
            for (int g = 0; g < total_g; ++g) {
                if (kb == 0) {
                    int tile;
                    bool part;
                    un.get(cluster + i * nclusters, tile, k0, kbn, part);
                    pair_coords(tg, tile, m0, n0);
                }
                const int s = g % S8;
                if (!mbar_wait(bar_empty8 + 8 * s, (uint32_t)(((g / S8) & 1) ^ 1), abort_flag, kErrProducer,
                               &g_tc2_error))
                    break;
                const uint32_t dst = sbase + kOffStage8 + s * kStage8;
                const bool sf_now = MX && sf_tma;
                mbar_expect_tx(bar_full8 + 8 * s, kStage8 + (sf_now ? kSfStage : 0));
                const int kx = k0 + kb;
                if (sf_now) {
                    // the stage's scale words of the CTA's 128 weight rows (word row kx BK / 4G of the
                    // [words, N] array, viewed as bytes [words, 4 N]), in two 256-byte boxes
                    const int wrow = (kx * BK) / (4 * ep.mx_group);
                    const uint32_t sdst = sbase + C::kOffSf + s * kSfStage;
                    const int x0 = 4 * (n0 + (int)rank * BNH);
                    tma_load_2d(sdst, &tmap_sf, x0, wrow, bar_full8 + 8 * s);
                    tma_load_2d(sdst + kSfStage / 2, &tmap_sf, x0 + kSfStage / 2, wrow, bar_full8 + 8 * s);
                }
                if constexpr (A16 && MX) {
                    // the fp16 A codes are loaded by their own warp (below), so that this loop does not
                    // wait for the MMA to release an operand stage before it stages the next weights
                    tma_load_2d(dst, &tmap_w, kx * BK, n0 + (int)rank * BNH, bar_full8 + 8 * s);
                } else if constexpr (A16) {
                    tma_load_2d(dst, &tmap_w, W4 ? kx * (BK / 2) : kx * BK, n0 + (int)rank * BNH, bar_full8 + 8 * s);
                    // the fp16 A codes go straight into the operand stage once the MMA has released it;
                    // their bytes complete on the barrier the converters arrive on
                    const int s16 = g % S16;
                    if (!mbar_wait(bar_empty16 + 8 * s16, (uint32_t)(((g / S16) & 1) ^ 1), abort_flag, kErrProducer,
                                   &g_tc2_error))
                        break;
                    const uint32_t fb = (leader ? bar_full16 : bar_conv16) + 8 * s16;
                    mbar_expect_tx(fb, kA16);
                    tma_load_2d(sbase + s16 * kStage16, &tmap_a, kx * BK, m0 + (int)rank * BMH, fb);
                } else {
                    tma_load_2d(dst, &tmap_a, kx * BK, m0 + (int)rank * BMH, bar_full8 + 8 * s);
                    tma_load_2d(dst + kA8, &tmap_w, W4 ? kx * (BK / 2) : kx * BK, n0 + (int)rank * BNH,
                                bar_full8 + 8 * s);
                }
                if (++kb == kbn) { kb = 0; ++i; }
            }
        }
      } else if (warp == 1) {
        // ---------------------------------------------------------------- pair MMA issuer
        if (leader && lane == 0) {
            int kb = 0, c = 0, i = 0, kbn = 0;
            for (int g = 0; g < total_g; ++g) {
                if (kb == 0) {
                    int tile, k0;
                    bool part;
                    un.get(cluster + i * nclusters, tile, k0, kbn, part);
                }
                const bool first = (kb % KB_PER_CHUNK) == 0;
                const bool last = (kb % KB_PER_CHUNK) == KB_PER_CHUNK - 1 || kb == kbn - 1;
                const int buf = c & 1;
                if (first) {
                    if (!mbar_wait_cluster(bar_accempty + 8 * buf, (uint32_t)(((c >> 1) & 1) ^ 1), abort_flag,
                                           kErrMmaAcc, &g_tc2_error))
                        break;
                    tc_fence_after();
                }
                const int s = g % S16;
                if (!mbar_wait_cluster(bar_full16 + 8 * s, (uint32_t)((g / S16) & 1), abort_flag, kErrMmaFull,
                                       &g_tc2_error))
                    break;
                tc_fence_after();
                const uint32_t a_addr = sbase + s * kStage16;
                const uint64_t adesc = smem_desc_sw128(a_addr);
                const uint64_t bdesc = smem_desc_sw128(a_addr + kA16);
                const uint32_t d = tmem_base + (uint32_t)(buf * BN);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    mma_f16_pair(d, adesc + (uint64_t)(kk * 2), bdesc + (uint64_t)(kk * 2), kIdesc,
                                 (first && kk == 0) ? 0u : 1u);
                mma_commit_pair(bar_empty16 + 8 * s, kPairMask);
                if (last) {
                    mma_commit_pair(bar_accfull + 8 * buf, kPairMask);
                    ++c;
                }
                if (++kb == kbn) { kb = 0; ++i; }
            }
        } else if (!leader && lane == 0) {
            // ---------------------------------------------------------------- relay (odd CTA)
            // Forwards "stage converted" to the even CTA with one remote arrive per stage.
            // The converted operands stay in this CTA's shared memory, fenced to the async
            // proxy by the converters, and the pair MMA reads them from here.
            for (int g = 0; g < total_g; ++g) {
                const int s = g % S16;
                if (!mbar_wait(bar_conv16 + 8 * s, (uint32_t)((g / S16) & 1), abort_flag, kErrRelay, &g_tc2_error))
                    break;
                mbar_arrive_remote(mapa_shared(bar_full16 + 8 * s, 0));
            }
        }
      } else if (MX && A16 && warp == 2 + kConvWarps) {
        // ---------------------------------------------------------------- activation loads
        // (block-scaled weights with fp16 activations): the fp16 A codes go straight into each
        // operand stage once the MMA has released it; their bytes complete on the barrier the
        // converters arrive on
        if (lane == 0) {
            int i = 0, kb = 0, m0 = 0, n0 = 0, k0 = 0, kbn = 0;
            for (int g = 0; g < total_g; ++g) {
                if (kb == 0) {
                    int tile;
                    bool part;
                    un.get(cluster + i * nclusters, tile, k0, kbn, part);
                    pair_coords(tg, tile, m0, n0);
                }
                const int s16 = g % S16;
                if (!mbar_wait(bar_empty16 + 8 * s16, (uint32_t)(((g / S16) & 1) ^ 1), abort_flag, kErrProducer,
                               &g_tc2_error))
                    break;
                const uint32_t fb = (leader ? bar_full16 : bar_conv16) + 8 * s16;
                mbar_expect_tx(fb, kA16);
                tma_load_2d(sbase + s16 * kStage16, &tmap_a, (k0 + kb) * BK, m0 + (int)rank * BMH, fb);
                if (++kb == kbn) { kb = 0; ++i; }
            }
        }
      } else if (warp < 2 + kConvWarps) {
        // ---------------------------------------------------------------- converters
        if constexpr (A16 && !W4 && !MX) {
            // W only: 512 16-byte int8 chunks per stage (128 rows x 4); thread ct takes idx = ct + T j
            // (idx < 512): row ct / 4 + (T / 4) j, chunk ct % 4, into the W half of the operand stage.
            constexpr int T = C::kConvT, NJ = (512 + T - 1) / T;
            const int ct = threadIdx.x - 64;
            const int r0 = ct >> 2, c0 = ct & 3;
            const uint32_t src0 = (uint32_t)(ct * 16);
            const uint32_t dst0 = (uint32_t)kA16 + sw128(r0, 2 * c0);
            const uint32_t dst1 = (uint32_t)kA16 + sw128(r0, 2 * c0 + 1);
            for (int g = 0; g < total_g; ++g) {
                const int s8 = g % S8, s16 = g % S16;
                if (!mbar_wait(bar_full8 + 8 * s8, (uint32_t)((g / S8) & 1), abort_flag, kErrConvFull, &g_tc2_error))
                    break;
                const uint32_t st8 = sbase + kOffStage8 + s8 * kStage8 + src0;
                uint4 in[NJ];
    #pragma unroll
                for (int j = 0; j < NJ; ++j)
                    in[j] = (ct + T * j < 512) ? lds128(st8 + T * 16 * j) : make_uint4(0, 0, 0, 0);
                if (!mbar_wait(bar_empty16 + 8 * s16, (uint32_t)(((g / S16) & 1) ^ 1), abort_flag, kErrConvEmpty,
                               &g_tc2_error))
                    break;
                const uint32_t st16 = sbase + s16 * kStage16;
    #pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    if (ct + T * j < 512) {
                        // cvt_word turns bytes (0, 1, 2, 3) into the fp16 pairs (0, 2) and (1, 3); TMA
                        // writes A in K order, so W's bytes are first permuted to (0, 2, 1, 3)
                        uint4 o0, o1;
                        cvt_word(__byte_perm(in[j].x, 0u, 0x3120u), o0.x, o0.y);
                        cvt_word(__byte_perm(in[j].y, 0u, 0x3120u), o0.z, o0.w);
                        cvt_word(__byte_perm(in[j].z, 0u, 0x3120u), o1.x, o1.y);
                        cvt_word(__byte_perm(in[j].w, 0u, 0x3120u), o1.z, o1.w);
                        sts128(st16 + dst0 + 32 * T * j, o0);
                        sts128(st16 + dst1 + 32 * T * j, o1);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive((leader ? bar_full16 : bar_conv16) + 8 * s16);
                    mbar_arrive(bar_empty8 + 8 * s8);
                }
            }
        } else
        // 1024 16-byte int8 chunks per stage ([A 128 rows | W 128 rows] x 4 chunks of each
        // 64-byte staging row); thread ct takes idx = ct + T j (T = kConvT converter threads,
        // j < kIters, idx < 1024): row ct / 4 + (T / 4) j, chunk ct % 4. (row & 7) does not
        // change with j, so the swizzled fp16 address is a per-thread base plus 32 T j bytes.
        // With fp16 activations (block-scaled weights only) the staging ring holds just the 512
        // weight chunks: the thread's chunks are idx = 512 + ct + T j (j < 2, idx < 1024), read from
        // staging offset 16 (idx - 512), and rows 128 .. 255 of the operand stage are its W half.
        if constexpr (!W4) {
            constexpr int T = C::kConvT;
            constexpr int kIdx0 = A16 ? 512 : 0;                      // chunk index of staging byte 0
            constexpr int NJ = (1024 - kIdx0 + T - 1) / T;            // chunks per thread and stage
            static_assert(!MX || T == 320 || (A16 && T == 256), "the block-scaled slot maps assume 10 converter "
                                                                 "warps, or 8 with fp16 activations");
            const int ct = threadIdx.x - 64;
            const int r0 = (kIdx0 >> 2) + (ct >> 2), c0 = ct & 3;
            const uint32_t src0 = (uint32_t)(ct * 16);
            const uint32_t dst0 = sw128(r0, 2 * c0);
            const uint32_t dst1 = sw128(r0, 2 * c0 + 1);
            // Block-scaled weights (T = 320): the thread's weight chunks (512 <= idx < 1024; weight
            // row (idx - 512) / 4 of the CTA's half, K chunk c0 of the stage) are, with int8
            // activations, j = 2 (slot 1) and one of j = 1 (ct >= 192) or j = 3 (ct < 64) (slot 0);
            // with fp16 activations j = 0 (slot 0) and j = 1 (slot 1: ct < 192 with ten converter warps,
            // every thread with eight). Their scale words arrive by TMA with the stage's weights or,
            // where the scale array's layout does not allow that, from L2 kSfAhead stages ahead.
            auto slot_j = [&](int jw) { return A16 ? jw : (jw == 1 ? 2 : (ct < 64 ? 3 : 1)); };
            auto slot_of = [](int j) { return A16 ? (j & 1) : (j == 2 ? 1 : 0); };
            // A ring of kSfAhead prefetched stages: slot 0 is the stage being converted.
            uint32_t sfw_cur[2] = {0u, 0u}, sfq[kSfAhead][2];
            int sh_cur = 0, shq[kSfAhead], pf_i = 0, pf_kb = 0;
            int sf_n[2] = {0, 0};                // weight rows of the slots in the prefetched stage's tile
            bool sf_ok[2] = {false, false};
            const int gshift = ep.mx_group == 32 ? 5 : 7;
            auto sf_fetch = [&](uint32_t (&dst)[2], int& sh) {
                if constexpr (MX) {
                    if (pf_kb == 0) {   // a new tile: its weight rows
                        int pm0, pn0;
                        pair_coords(tg, cluster + pf_i * nclusters, pm0, pn0);   // MX: whole tiles only
#pragma unroll
                        for (int jw = 0; jw < 2; ++jw) {
                            const int idx = kIdx0 + ct + T * slot_j(jw);
                            sf_n[jw] = pn0 + (int)rank * BNH + ((idx - 512) >> 2);
                            sf_ok[jw] = idx >= 512 && idx < 1024 && sf_n[jw] < N;
                        }
                    }
                    const int grp = (pf_kb * BK + 16 * c0) >> gshift;
                    const uint32_t* base = ep.mx_sf + (int64_t)(grp >> 2) * N;
                    sh = 8 * (grp & 3);
#pragma unroll
                    for (int jw = 0; jw < 2; ++jw) dst[jw] = sf_ok[jw] ? __ldg(base + sf_n[jw]) : 0u;
                    if (++pf_kb == KB) { pf_kb = 0; ++pf_i; }   // MX: whole tiles, KB stages each
                }
            };
            // Scale words staged by TMA: the slot's weight row within the CTA's half and the stage's
            // k-block within its tile (block-scaled launches take whole tiles, KB stages each).
            int sf_row[2] = {0, 0}, kbc = 0;
#pragma unroll
            for (int jw = 0; jw < 2; ++jw) {
                const int idx = kIdx0 + ct + T * slot_j(jw);
                sf_row[jw] = idx >= 512 && idx < 1024 ? (idx - 512) >> 2 : -1;
            }
#pragma unroll
            for (int d = 0; d < kSfAhead; ++d) {
                sfq[d][0] = sfq[d][1] = 0u;
                shq[d] = 0;
                if (MX && !sf_tma && d < total_g) sf_fetch(sfq[d], shq[d]);
            }
            for (int g = 0; g < total_g; ++g) {
                if constexpr (MX) {
                  if (!sf_tma) {
                    sfw_cur[0] = sfq[0][0];
                    sfw_cur[1] = sfq[0][1];
                    sh_cur = shq[0];
#pragma unroll
                    for (int d = 0; d + 1 < kSfAhead; ++d) {
                        sfq[d][0] = sfq[d + 1][0];
                        sfq[d][1] = sfq[d + 1][1];
                        shq[d] = shq[d + 1];
                    }
                    if (g + kSfAhead < total_g) sf_fetch(sfq[kSfAhead - 1], shq[kSfAhead - 1]);
                  }
                }
                const int s8 = g % S8, s16 = g % S16;
                if (!mbar_wait(bar_full8 + 8 * s8, (uint32_t)((g / S8) & 1), abort_flag, kErrConvFull, &g_tc2_error))
                    break;
                const uint32_t st8 = sbase + kOffStage8 + s8 * kStage8 + src0;
                uint4 in[NJ];
    #pragma unroll
                for (int j = 0; j < NJ; ++j)
                    in[j] = (kIdx0 + ct + T * j < 1024) ? lds128(st8 + T * 16 * j) : make_uint4(0, 0, 0, 0);
                if constexpr (MX) {
                    if (sf_tma) {   // this stage's scale words arrived with its weights
                        const uint32_t sfb = sbase + C::kOffSf + s8 * kSfStage;
#pragma unroll
                        for (int jw = 0; jw < 2; ++jw)
                            sfw_cur[jw] = sf_row[jw] >= 0 ? lds32(sfb + 4 * (uint32_t)sf_row[jw]) : 0u;
                        sh_cur = 8 * (((kbc * BK + 16 * c0) >> gshift) & 3);
                        if (++kbc == KB) kbc = 0;
                    }
                }
                if (!mbar_wait(bar_empty16 + 8 * s16, (uint32_t)(((g / S16) & 1) ^ 1), abort_flag, kErrConvEmpty,
                               &g_tc2_error))
                    break;
                const uint32_t st16 = sbase + s16 * kStage16;
                if constexpr (MX) {
                    // A weight chunk becomes q * s in two steps per code pair (a lop3, an fp16 add). The
                    // fp16 with exponent field E = e - 102 (s = 2^(e - 127) = 2^(E - 25)) and the
                    // code in the low mantissa bits, M | (byte ^ 0x80) with M = E << 10 | 0x80, is
                    // (1152 + q) s exactly; subtracting 1152 s (the same bits with the sign set) is
                    // exact. E must be a normal exponent, e <= 132: a warp in which some lane has a
                    // larger scale builds (1152 + q) s / 16 and multiplies the difference by 16
                    // (exact). Activation chunks are converted as in the int8 format.
                    uint32_t ev[2], mg[2];
                    bool big = false;
#pragma unroll
                    for (int jw = 0; jw < 2; ++jw) {
                        ev[jw] = min(max((sfw_cur[jw] >> sh_cur) & 0xFFu, 103u), 136u);
                        big |= ev[jw] > 132u;
                    }
                    const bool slow = __any_sync(0xffffffffu, big);
#pragma unroll
                    for (int jw = 0; jw < 2; ++jw) {
                        // ((e - 102) << 10 | 0x80) in both halves is e * 0x04000400 - 0x97819780 (mod 2^32,
                        // no carry between the halves); e > 132: (e - 106), 0x10001000 less
                        mg[jw] = ev[jw] * 0x04000400u - (ev[jw] > 132u ? 0xA781A780u : 0x97819780u);
                    }
#pragma unroll
                    for (int j = 0; j < NJ; ++j) {
                        if (kIdx0 + ct + T * j < 1024) {
                            uint4 o0, o1;
                            if (kIdx0 + ct + T * j >= 512) {   // a weight chunk (warp-uniform)
                                const uint32_t m = mg[slot_of(j)], c = m | 0x80008000u;
                                cvt_word_magic(in[j].x, m, c, o0.x, o0.y);
                                cvt_word_magic(in[j].y, m, c, o0.z, o0.w);
                                cvt_word_magic(in[j].z, m, c, o1.x, o1.y);
                                cvt_word_magic(in[j].w, m, c, o1.z, o1.w);
                                if (slow) {   // rows with e > 132 were built at s / 16
                                    const uint32_t pj = ev[slot_of(j)] > 132u ? 0x4C004C00u : 0x3C003C00u;   // 16 or 1
                                    o0 = make_uint4(hmul2(o0.x, pj), hmul2(o0.y, pj), hmul2(o0.z, pj), hmul2(o0.w, pj));
                                    o1 = make_uint4(hmul2(o1.x, pj), hmul2(o1.y, pj), hmul2(o1.z, pj), hmul2(o1.w, pj));
                                }
                            } else {
                                cvt_word(in[j].x, o0.x, o0.y);
                                cvt_word(in[j].y, o0.z, o0.w);
                                cvt_word(in[j].z, o1.x, o1.y);
                                cvt_word(in[j].w, o1.z, o1.w);
                            }
                            sts128(st16 + dst0 + 32 * T * j, o0);
                            sts128(st16 + dst1 + 32 * T * j, o1);
                        }
                    }
                } else {
    #pragma unroll
                    for (int j = 0; j < NJ; ++j) {
                        if (ct + T * j < 1024) {
                            uint4 o0, o1;
                            cvt_word(in[j].x, o0.x, o0.y);
                            cvt_word(in[j].y, o0.z, o0.w);
                            cvt_word(in[j].z, o1.x, o1.y);
                            cvt_word(in[j].w, o1.z, o1.w);
                            sts128(st16 + dst0 + 32 * T * j, o0);
                            sts128(st16 + dst1 + 32 * T * j, o1);
                        }
                    }
                }
                // Every lane makes its fp16 stores visible to the tensor core, then one lane per
                // warp arrives: on the MMA barrier in the even CTA, on the relay's barrier in
                // the odd one.
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive((leader ? bar_full16 : bar_conv16) + 8 * s16);
                    mbar_arrive(bar_empty8 + 8 * s8);   // after the loaded registers were consumed
                }
            }
        } else {
            // int4 weights: A as above over its 512 chunks (idx = ct + T j < 512; not with fp16
            // activations, which TMA has put in place); W's 256 packed chunks (128 rows x 2 chunks of
            // 32 K) take idx = ct + T j (idx < 256): row ct / 2 + (T / 2) j, chunk ct % 2; each becomes four
            // fp16 chunks 4 (ct % 2) + q of its row, word q of the packed chunk (8 K) giving fp16 chunk
            // q through two nibble pairs, in the pair order of cvt_word.
            constexpr int T = C::kConvT;   // converter threads (a multiple of 32)
            const int ct = threadIdx.x - 64;
            const int ra = ct >> 2, ca = ct & 3;
            const uint32_t srcA = (uint32_t)(ct * 16);
            const uint32_t dA0 = sw128(ra, 2 * ca), dA1 = sw128(ra, 2 * ca + 1);
            const int rw = ct >> 1, cw = ct & 1;
            const uint32_t srcW = (uint32_t)((A16 ? 0 : kA8) + ct * 16);
            uint32_t dW[4];
    #pragma unroll
            for (int q = 0; q < 4; ++q) dW[q] = (uint32_t)kA16 + sw128(rw, 4 * cw + q);
            for (int g = 0; g < total_g; ++g) {
                const int s8 = g % S8, s16 = g % S16;
                if (!mbar_wait(bar_full8 + 8 * s8, (uint32_t)((g / S8) & 1), abort_flag, kErrConvFull, &g_tc2_error))
                    break;
                const uint32_t st8 = sbase + kOffStage8 + s8 * kStage8;
                constexpr int NA = (512 + T - 1) / T, NW = (256 + T - 1) / T;
                uint4 ia[NA], iw[NW];
    #pragma unroll
                for (int j = 0; j < NA; ++j)
                    ia[j] = (!A16 && ct + T * j < 512) ? lds128(st8 + srcA + T * 16 * j) : make_uint4(0, 0, 0, 0);
    #pragma unroll
                for (int j = 0; j < NW; ++j)
                    iw[j] = (ct + T * j < 256) ? lds128(st8 + srcW + T * 16 * j) : make_uint4(0, 0, 0, 0);
                if (!mbar_wait(bar_empty16 + 8 * s16, (uint32_t)(((g / S16) & 1) ^ 1), abort_flag, kErrConvEmpty,
                               &g_tc2_error))
                    break;
                const uint32_t st16 = sbase + s16 * kStage16;
    #pragma unroll
                for (int j = 0; j < NA; ++j) {
                    if (!A16 && ct + T * j < 512) {
                        uint4 o0, o1;
                        cvt_word(ia[j].x, o0.x, o0.y);
                        cvt_word(ia[j].y, o0.z, o0.w);
                        cvt_word(ia[j].z, o1.x, o1.y);
                        cvt_word(ia[j].w, o1.z, o1.w);
                        sts128(st16 + dA0 + 32 * T * j, o0);   // rows ra + (T / 4) j
                        sts128(st16 + dA1 + 32 * T * j, o1);
                    }
                }
    #pragma unroll
                for (int j = 0; j < NW; ++j) {
                    if (ct + T * j < 256) {
                        const uint32_t wv[4] = {iw[j].x, iw[j].y, iw[j].z, iw[j].w};
    #pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint4 o;
                            cvt_int4x4<0x4140u>(wv[q], o.x, o.y);
                            cvt_int4x4<0x4342u>(wv[q], o.z, o.w);
                            sts128(st16 + dW[q] + 64 * T * j, o);   // rows rw + (T / 2) j
                        }
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive((leader ? bar_full16 : bar_conv16) + 8 * s16);
                    mbar_arrive(bar_empty8 + 8 * s8);   // after the loaded registers were consumed
                }
            }
        }
      }
    } else {
        // ---------------------------------------------------------------- drain + epilogue
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(C::kRegsHigh));
        const int quarter = warp & 3;
        // 8 drain warps: warp pair (w, w + 4) takes accumulator columns [0, 128) and [128, 256);
        // 4 drain warps: each takes both halves, one after the other
        constexpr int kHalves = 8 / kDrainWarps;
        const int col_half = kHalves == 1 ? (warp - C::kDrain0) >> 2 : 0;
        int acc[128];
#pragma unroll
        for (int c = 0; c < 128; ++c) acc[c] = 0;
        // chunks of this cluster's units in order; a unit's state is read at its first chunk
        const int cpt_full = (KB + KB_PER_CHUNK - 1) / KB_PER_CHUNK;
        const int cpt_part = (un.kb_part + KB_PER_CHUNK - 1) / KB_PER_CHUNK;
        const int chunks_total = my_full * cpt_full + (my_units - my_full) * cpt_part;
        int ti = 0, cc = 0, cpt = 1, dtile = 0;
        bool dpart = false;
        for (int c = 0; c < chunks_total; ++c, (++cc == cpt ? (cc = 0, ++ti) : 0)) {
            if (cc == 0) {
                if constexpr (MX) {   // whole tiles only
                    dtile = cluster + ti * nclusters;
                    cpt = cpt_full;
                } else {
                    int k0, kbn;
                    un.get(cluster + ti * nclusters, dtile, k0, kbn, dpart);
                    cpt = (kbn + KB_PER_CHUNK - 1) / KB_PER_CHUNK;
                }
            }
            const int buf = c & 1;
            if (!mbar_wait(bar_accfull + 8 * buf, (uint32_t)((c >> 1) & 1), abort_flag, kErrDrain, &g_tc2_error))
                break;
            tc_fence_after();
            for (int hh = 0; hh < kHalves; ++hh) {
                const int chalf = kHalves == 1 ? col_half : hh;
                const uint32_t taddr =
                    tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(buf * BN + chalf * 128);
                const int keep = cc != 0;
    #pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t v[32];
                    tmem_ld32(taddr + j * 32, v);
    #pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        if constexpr (MX)
                            acc[j * 32 + e] = (int)v[e];   // fp32 sums (bit patterns), one chunk per tile
                        else
                            acc[j * 32 + e] = acc[j * 32 + e] * keep + __float2int_rn(__uint_as_float(v[e]));
                    }
                }
                if (hh == kHalves - 1) {   // the whole buffer has been read
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(mapa_shared(bar_accempty + 8 * buf, 0));
                }
                if (cc != cpt - 1) continue;
                int m0, n0;
                pair_coords(tg, dtile, m0, n0);
                const int mrow0 = m0 + (int)rank * BMH + quarter * 32;
                const int m = mrow0 + lane;
                const int nb = n0 + chalf * 128;
                float sa = 0.0f;
                int za = 0;
                if (!ep.out_i32 && m < M) {
                    sa = ep.s_a[ep.a_per_row ? m : 0];
                    za = ep.z_a ? ep.z_a[ep.a_per_row ? m : 0] : 0;
                }
                const bool vec = ((N & 3) == 0);
                const bool vsw = ep.w_per_row && vec && ((reinterpret_cast<uintptr_t>(ep.s_w) & 15) == 0);
                const bool vcs = ep.z_a && vec && ((reinterpret_cast<uintptr_t>(ep.colsum) & 15) == 0);
                // outputs (m, n .. n + 3) of accumulator columns e .. e + 3, as 4-byte words
                auto out4 = [&](int e, int n) -> uint4 {
                    if (ep.out_i32 || dpart) return make_uint4(acc[e], acc[e + 1], acc[e + 2], acc[e + 3]);
                    if constexpr (MX) {   // y = fl(T * s_a) (+ bias)
                        uint32_t o[4];
    #pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            float v = __fmul_rn(__uint_as_float((uint32_t)acc[e + q]), sa);
                            if (ep.bias) v = __fadd_rn(v, __ldg(ep.bias + (n + q < N ? n + q : 0)));
                            o[q] = __float_as_uint(v);
                        }
                        return make_uint4(o[0], o[1], o[2], o[3]);
                    }
                    const bool full = n + 3 < N;
                    float sw4[4];
                    int cs4[4] = {0, 0, 0, 0};
                    if (vsw && full) {
                        const float4 t4 = __ldg(reinterpret_cast<const float4*>(ep.s_w + n));
                        sw4[0] = t4.x; sw4[1] = t4.y; sw4[2] = t4.z; sw4[3] = t4.w;
                    } else {
    #pragma unroll
                        for (int q = 0; q < 4; ++q) sw4[q] = __ldg(ep.s_w + (ep.w_per_row ? (n + q < N ? n + q : 0) : 0));
                    }
                    if (ep.z_a) {
                        if (vcs && full) {
                            const int4 t4 = __ldg(reinterpret_cast<const int4*>(ep.colsum + n));
                            cs4[0] = t4.x; cs4[1] = t4.y; cs4[2] = t4.z; cs4[3] = t4.w;
                        } else {
    #pragma unroll
                            for (int q = 0; q < 4; ++q) cs4[q] = __ldg(ep.colsum + (n + q < N ? n + q : 0));
                        }
                    }
                    uint32_t o[4];
    #pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float v = __fmul_rn(__int2float_rn(acc[e + q] - za * cs4[q]), __fmul_rn(sa, sw4[q]));
                        if (ep.bias) v = __fadd_rn(v, __ldg(ep.bias + (n + q < N ? n + q : 0)));
                        o[q] = __float_as_uint(v);
                    }
                    return make_uint4(o[0], o[1], o[2], o[3]);
                };
                if (tma_out) {
                    // Each block of 32 rows x 128 bytes (32 fp32, 64 bf16 or 128 int8 columns) goes
                    // through this warp's shared buffer (128-byte swizzle: row `lane`, 16-byte chunk c
                    // at chunk c ^ (lane & 7)) and one TMA store, which writes whole lines and clips
                    // rows >= M and columns >= N. ESZ (bytes per output) is a compile-time constant
                    // so that acc[] stays in registers.
                    const uint32_t ebuf = sbase + kOffEpi + (uint32_t)((warp - C::kDrain0) * kEpiBytes);
                    auto blocks = [&](auto esz_tag) {
                        constexpr int ESZ = decltype(esz_tag)::value;
                        constexpr int BCOLS = 128 / ESZ;
    #pragma unroll
                        for (int j = 0; j < ESZ; ++j) {
                            if (lane == 0) bulk_wait_read_all();   // the previous block has left the buffer
                            __syncwarp();
    #pragma unroll
                            for (int c = 0; c < 8; ++c) {
                                const int e0 = j * BCOLS + c * (16 / ESZ);
                                uint4 w;
                                if constexpr (ESZ == 4) {
                                    w = out4(e0, nb + e0);
                                } else if constexpr (ESZ == 2) {
                                    const uint4 a = out4(e0, nb + e0), b = out4(e0 + 4, nb + e0 + 4);
                                    w = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y),
                                                   pack_bf16x2(b.z, b.w));
                                } else {
                                    uint32_t q[4];
    #pragma unroll
                                    for (int t = 0; t < 4; ++t) {
                                        const uint4 a = out4(e0 + 4 * t, nb + e0 + 4 * t);
                                        q[t] = pack_codes4(a, ep.out_scale);
                                    }
                                    w = make_uint4(q[0], q[1], q[2], q[3]);
                                }
                                sts128(ebuf + (uint32_t)(lane * 128 + ((c ^ (lane & 7)) << 4)), w);
                            }
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                if (dpart)   // a K slice: its INT32 partial sums are added
                                tma_reduce_add_2d(&tmap_acc, ebuf, nb + j * BCOLS, mrow0);
                            else
                                tma_store_2d(&tmap_out, ebuf, nb + j * BCOLS, mrow0);
                                bulk_commit();
                            }
                        }
                    };
                    if (ep.out_i32 || dpart || ep.out_kind == kOutF32)
                        blocks(std::integral_constant<int, 4>{});
                    else if (ep.out_kind == kOutBF16)
                        blocks(std::integral_constant<int, 2>{});
                    else
                        blocks(std::integral_constant<int, 1>{});
                } else if (m < M && !ep.out_i32 && ep.out_kind != kOutF32) {
    #pragma unroll
                    for (int e4 = 0; e4 < 32; ++e4) {
                        const int n = nb + e4 * 4;
                        const uint4 o = out4(e4 * 4, n);
                        if (n < N) epi_store(ep, (int64_t)m * N + n, __uint_as_float(o.x));
                        if (n + 1 < N) epi_store(ep, (int64_t)m * N + n + 1, __uint_as_float(o.y));
                        if (n + 2 < N) epi_store(ep, (int64_t)m * N + n + 2, __uint_as_float(o.z));
                        if (n + 3 < N) epi_store(ep, (int64_t)m * N + n + 3, __uint_as_float(o.w));
                    }
                } else if (m < M) {
                    uint32_t* row = ep.out_i32 ? reinterpret_cast<uint32_t*>(ep.out_i32) + (int64_t)m * N
                                               : reinterpret_cast<uint32_t*>(ep.y) + (int64_t)m * N;
    #pragma unroll
                    for (int e4 = 0; e4 < 32; ++e4) {
                        const int n = nb + e4 * 4;
                        const uint4 o = out4(e4 * 4, n);
                        if (vec && n + 3 < N) {
                            *reinterpret_cast<uint4*>(row + n) = o;
                        } else {
                            if (n < N) row[n] = o.x;
                            if (n + 1 < N) row[n + 1] = o.y;
                            if (n + 2 < N) row[n + 2] = o.z;
                            if (n + 3 < N) row[n + 3] = o.w;
                        }
                    }
                }
            }
        }
        if (lane == 0) bulk_wait_all();   // stores done before the shared buffers go away
    }

    // Wind down: both CTAs finish (the even CTA's MMA reads the odd CTA's shared
    // memory and the odd CTA arrives on the even CTA's barriers until the end).
    if (*abort_flag) {
        const long long t0 = clock64();
        while (clock64() - t0 < (1LL << 22)) __nanosleep(1000);
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem_base, kTmemCols);
}

}  // namespace

bool gemm_tc2_supports(int64_t M, int64_t N, int64_t K, int wfmt) {
    const bool w4 = wfmt == kWInt4 || wfmt == kW4A16;
    if (!(M >= 1 && N >= 1 && K >= 16 && (K % (w4 ? 32 : 16)) == 0 && M < (1LL << 31) && N < (1LL << 31)))
        return false;
    const int64_t tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    const int64_t kb = (K + BK - 1) / BK;
    return tiles < (1LL << 30) && tiles * kb < (1LL << 31);
}

// Clusters of two that fit on the device at once (a GPC with an odd number of
// free SMs leaves one idle), so that the persistent grid runs in one wave.
// Cached per device and weight format; SMs / 2 if the occupancy query fails.
template <int WF>
static int resident_pairs() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return device_sm_count() / 2;
    if (cached[dev] > 0) return cached[dev];
    int pairs = device_sm_count() / 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = PairCfg<WF>::kSmem;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_tc2_kernel<WF>, &cfg) == cudaSuccess && n > 0 && n < pairs) pairs = n;
    (void)cudaGetLastError();
    cached[dev] = pairs;
    return pairs;
}

// Tiles [n_full, tiles) of the pair grid (order of pair_coords), 16 blocks of 256 threads per
// tile, four consecutive outputs per thread step; N % 4 == 0. The zeroing before a K-split
// launch, and the dequantization epilogue on the INT32 sums the slices left in y's storage,
// in place: y = fl(fl((float)(acc - z_a colsum) * fl(s_a s_w)) + bias), the fused epilogue's
// arithmetic.
__global__ void __launch_bounds__(256) part_tiles_zero_kernel(int32_t* acc, int M, int N, PairGeom tg, int n_full) {
    int m0, n0;
    pair_coords(tg, n_full + (int)blockIdx.y, m0, n0);
    for (int e = ((int)blockIdx.x * 256 + (int)threadIdx.x) * 4; e < BM * BN; e += 16 * 256 * 4) {
        const int m = m0 + e / BN, n = n0 + e % BN;
        if (m < M && n < N) *reinterpret_cast<int4*>(acc + (int64_t)m * N + n) = make_int4(0, 0, 0, 0);
    }
}

__global__ void __launch_bounds__(256) part_tiles_epilogue_kernel(Epilogue ep, int M, int N, PairGeom tg, int n_full) {
    int m0, n0;
    pair_coords(tg, n_full + (int)blockIdx.y, m0, n0);
    for (int e = ((int)blockIdx.x * 256 + (int)threadIdx.x) * 4; e < BM * BN; e += 16 * 256 * 4) {
        const int m = m0 + e / BN, n = n0 + e % BN;
        if (m >= M || n >= N) continue;
        const int64_t idx = (int64_t)m * N + n;
        const int4 acc = *reinterpret_cast<const int4*>(ep.y + idx);
        const float sa = ep.s_a[ep.a_per_row ? m : 0];
        const int za = ep.z_a ? ep.z_a[ep.a_per_row ? m : 0] : 0;
        const int a4[4] = {acc.x, acc.y, acc.z, acc.w};
        float o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float sw = ep.s_w[ep.w_per_row ? n + q : 0];
            const int cs = ep.z_a ? ep.colsum[n + q] : 0;
            o[q] = epi_bias(ep, __fmul_rn(__int2float_rn(a4[q] - za * cs), __fmul_rn(sa, sw)), n + q);
        }
        *reinterpret_cast<float4*>(ep.y + idx) = make_float4(o[0], o[1], o[2], o[3]);
    }
}

static PairGeom pair_geom(int64_t M, int64_t N, int band) {
    PairGeom tg;
    tg.num_m = (int)((M + BM - 1) / BM);
    tg.num_n = (int)((N + BN - 1) / BN);
    tg.tiles = tg.num_m * tg.num_n;
    tg.band = band;
    return tg;
}

template <int WF>
static cudaError_t launch_gemm_tc2_t(const void* qa, const void* qw, int64_t M, int64_t N, int64_t K,
                                     const Epilogue& ep, cudaStream_t stream, int n_full, int ksplit,
                                     int32_t* acc) {
    using C = PairCfg<WF>;
    constexpr bool W4 = C::W4;
    CUtensorMap ma, mw;
    // int4: the packed weights are a byte matrix [N, K / 2], staged 32 bytes (64 K) per k-block;
    // A16: fp16 codes in [128 rows x 64 K] boxes with the operand ring's 128-byte swizzle
    const bool map_a = C::A16 ? make_tma_map_f16(&ma, static_cast<const uint16_t*>(qa), M, K, BMH, BK)
                              : make_tma_map_i8(&ma, static_cast<const int8_t*>(qa), M, K, BMH, BK);
    if (!map_a ||
        !make_tma_map_i8(&mw, static_cast<const int8_t*>(qw), N, W4 ? K / 2 : K, BNH, W4 ? BK / 2 : BK))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(gemm_tc2_kernel<WF>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    const PairGeom tg = pair_geom(M, N, PairCfg<WF>::kBand);
    const int64_t units = n_full + (int64_t)(tg.tiles - n_full) * ksplit;
    const int64_t pairs = resident_pairs<WF>();
    const int clusters = (int)(units < pairs ? units : pairs);
    CUtensorMap mo, mc;
    const bool tma_out = ep.out_i32                  ? make_tma_map_out(&mo, ep.out_i32, kMapI32, M, N)
                         : ep.out_kind == kOutF32  ? make_tma_map_out(&mo, ep.y, kMapF32, M, N)
                         : ep.out_kind == kOutBF16 ? make_tma_map_out(&mo, ep.out_bf16, kMapBF16, M, N)
                                                   : make_tma_map_out(&mo, ep.out_i8, kMapI8, M, N);
    if (!tma_out) memset(&mo, 0, sizeof(mo));
    if (n_full < tg.tiles) {   // sliced tiles: partial sums are added by TMA only
        if (!tma_out || !acc || !make_tma_map_out(&mc, acc, kMapI32, M, N)) return cudaErrorInvalidValue;
    } else {
        memset(&mc, 0, sizeof(mc));
    }
    // block-scaled weights: the scale words [words, N] as a byte matrix [words, 4 N] for TMA, where
    // its rows are whole 16-byte multiples and its base is 16-byte aligned
    CUtensorMap ms;
    bool sf_tma = false;
    if (C::MX && N % 4 == 0 && (reinterpret_cast<uintptr_t>(ep.mx_sf) & 15) == 0) {
        const int64_t words = (K / ep.mx_group + 3) / 4;
        sf_tma = make_tma_map_i8(&ms, reinterpret_cast<const int8_t*>(ep.mx_sf), words, 4 * N, 1, kSfStage / 2);
    }
    if (!sf_tma) memset(&ms, 0, sizeof(ms));
    gemm_tc2_kernel<WF><<<2 * clusters, kThreads, C::kSmem, stream>>>(ma, mw, mo, mc, ms, tma_out ? 1 : 0,
                                                                      sf_tma ? 1 : 0, (int)M, (int)N, (int)K, n_full,
                                                                      ksplit, ep);
    note_launch();
    return cudaGetLastError();
}

// K slices where the pair grid would leave clusters idle: a grid that fills at most half of the
// resident clusters has every tile sliced; a grid with a partial last wave has the tiles of that
// wave sliced. The slice count is the largest of 2, 4, 8 that keeps the sliced units within one
// wave of clusters, divides the k-blocks evenly and leaves each slice at least 8 k-blocks
// (512 K). Only where the INT32 sums have 4-byte room to be added in: the INT32 export, or fp32
// output (the sums go into y, then the epilogue runs in place); rows of whole 16-byte multiples
// (N % 4 == 0) for the TMA reduce-add.
template <int WF>
static void plan_split(int64_t M, int64_t N, int64_t K, const Epilogue& ep, int& n_full, int& ksplit,
                       int32_t*& acc) {
    const PairGeom tg = pair_geom(M, N, PairCfg<WF>::kBand);
    n_full = tg.tiles;
    ksplit = 1;
    acc = nullptr;
    const bool i32 = ep.out_i32 != nullptr;
    if (!i32 && !(ep.out_kind == kOutF32 && ep.y)) return;
    int32_t* target = i32 ? ep.out_i32 : reinterpret_cast<int32_t*>(ep.y);
    if (N % 4 != 0 || (reinterpret_cast<uintptr_t>(target) & 15) != 0) return;
    const int64_t kb = (K + BK - 1) / BK;
    const int64_t pairs = resident_pairs<WF>();
    const int64_t sliced = 2 * tg.tiles <= pairs ? tg.tiles : tg.tiles % pairs;
    if (sliced == 0) return;
    int best = 1;
    for (int sl = 2; sl <= 8; sl *= 2)
        if (sliced * sl <= pairs && kb % sl == 0 && kb / sl >= 8) best = sl;
    if (best == 1) return;
    n_full = (int)(tg.tiles - sliced);
    ksplit = best;
    acc = target;
}

template <int WF>
static cudaError_t launch_gemm_tc2_split(const void* qa, const void* qw, int64_t M, int64_t N, int64_t K,
                                         const Epilogue& ep, cudaStream_t stream) {
    int n_full, ksplit;
    int32_t* acc;
    plan_split<WF>(M, N, K, ep, n_full, ksplit, acc);
    if (ksplit == 1) return launch_gemm_tc2_t<WF>(qa, qw, M, N, K, ep, stream, n_full, 1, nullptr);
    const PairGeom tg = pair_geom(M, N, PairCfg<WF>::kBand);
    const dim3 grid(16, (unsigned)(tg.tiles - n_full));
    part_tiles_zero_kernel<<<grid, 256, 0, stream>>>(acc, (int)M, (int)N, tg, n_full);
    note_launch();
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = launch_gemm_tc2_t<WF>(qa, qw, M, N, K, ep, stream, n_full, ksplit, acc);
    if (e != cudaSuccess || ep.out_i32) return e;
    part_tiles_epilogue_kernel<<<grid, 256, 0, stream>>>(ep, (int)M, (int)N, tg, n_full);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_gemm_tc2(const void* qa, const void* qw, int64_t M, int64_t N, int64_t K, const Epilogue& ep,
                            cudaStream_t stream, int wfmt) {
    if (!gemm_tc2_supports(M, N, K, wfmt)) return cudaErrorNotSupported;
    if (wfmt == kWMx || wfmt == kWMxA16) {
        if (!ep.mx_sf || (ep.mx_group != 32 && ep.mx_group != 128) || K % ep.mx_group != 0 || ep.out_i32 || ep.z_a)
            return cudaErrorInvalidValue;
        const int tiles = pair_geom(M, N, 1).tiles;   // the tile count (the band does not change it)
        return wfmt == kWMx ? launch_gemm_tc2_t<kWMx>(qa, qw, M, N, K, ep, stream, tiles, 1, nullptr)
                            : launch_gemm_tc2_t<kWMxA16>(qa, qw, M, N, K, ep, stream, tiles, 1, nullptr);
    }
    if (wfmt == kWA16) return launch_gemm_tc2_split<kWA16>(qa, qw, M, N, K, ep, stream);
    if (wfmt == kW4A16) return launch_gemm_tc2_split<kW4A16>(qa, qw, M, N, K, ep, stream);
    return wfmt == kWInt4 ? launch_gemm_tc2_split<kWInt4>(qa, qw, M, N, K, ep, stream)
                          : launch_gemm_tc2_split<kWInt8>(qa, qw, M, N, K, ep, stream);
}

cudaError_t read_and_clear_gemm_tc2_error(uint32_t* code) {
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_tc2_error, sizeof(v));
    if (e != cudaSuccess) return e;
    *code = v;
    if (v) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_tc2_error, &zero, sizeof(zero));
    }
    return e;
}

}  // namespace q8
