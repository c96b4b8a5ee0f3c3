// Decode-shaped integer GEMM (M <= 16 tokens) + dequantization epilogue on the
// tcgen05 tensor cores.
//
// With a handful of tokens the layer streams the int8 weights once from HBM and
// does almost no arithmetic per byte, so the kernel is built around the weight
// stream. The operands are swapped relative to the prefill kernel: 64 weight
// rows (output channels) are the MMA's M side (M = 128, rows 64..127 held at
// zero) and the <= 16 tokens are its N = 16 side, so the accumulator is a
// 128 x 16 fp32 tile in tensor memory and y is written transposed. 64-row
// tiles give 448 tiles for N = 28672, about three per SM on 152 SMs.
//
// An N = 16 MMA is short, so a chain of them into one accumulator is bound by
// the MMA latency, not the tensor pipe. The eight K-steps of a stage therefore
// accumulate into eight separate TMEM accumulators (independent chains); the
// drain adds them. Exactness is the prefill kernel's argument: int8 codes are
// exact in fp16, products are exact, every fp32 accumulator holds at most
// 1024 products (|partial| <= 2^24; here 128 per chain), and chunk sums are
// added in INT32 registers.
//
//   warp 0          TMA: W [64 x 128] and A [16 x 128] int8 boxes, 128-byte swizzled,
//                   -> staging ring (10 x 10 KB)
//   warp 1          TMEM allocation, tcgen05.mma issue (one thread)
//   warps 2..11,    int8 -> fp16 conversion into the swizzled operand ring (3 x 36 KB);
//   14, 15          twelve warps, so each thread converts at most two 16-byte chunks a stage
//   warps 12, 13    drain the chunk accumulators into INT32 and run the epilogue
// setmaxnreg gives the last warpgroup (drain + two converter warps) 232 registers and
// the other three 80: 3*128*80 + 128*232 = 60416 <= 512 threads x 128 at launch.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "q8_internal.h"
#include "q8_tc_ptx.cuh"

namespace q8 {

// Device error word of this kernel (one per device).
static __device__ unsigned int g_gemv_error;

namespace {

using namespace tc;

constexpr int RW = 64;             // real weight rows per tile
constexpr int MM = 128;            // MMA M (rows RW..MM-1 are zero)
constexpr int NT = 16;             // tokens: MMA N
constexpr int BK = 128;            // K per stage
constexpr int S8 = 10;             // int8 staging stages
constexpr int S16 = 3;             // fp16 operand stages
constexpr int KB_PER_CHUNK = 8;    // 8 * 128 = 1024 K per exact fp32 chunk
constexpr int kConv = 384;         // converter threads: warps 2..11, 14, 15
constexpr int kDrainWarps = 2;     // warps 12, 13: TMEM lane quarters 0 and 1 (weight rows 0..63)
constexpr int kThreads = 512;
constexpr int kRegsLow = 80, kRegsHigh = 232;
constexpr int kChains = BK / 16;   // independent accumulators, one per K-step of a stage
constexpr int kTmemCols = 2 * kChains * NT;   // two buffers of 8 chains x 16 columns = 256

constexpr int kW8 = RW * BK;                       // 8 KB
constexpr int kA8 = NT * BK;                       // 2 KB
constexpr int kStage8 = kW8 + kA8;                 // 10 KB
constexpr int kChunks8 = kStage8 / 16;             // 640 16-byte chunks per stage
constexpr int kAtomW = MM * 128;                   // one 64-wide fp16 K column of 128 swizzled rows
constexpr int kAtomA = NT * 128;
constexpr int kW16 = 2 * kAtomW;                   // K = 128 fp16 = two swizzle columns
constexpr int kA16 = 2 * kAtomA;
constexpr int kStage16 = kW16 + kA16;              // 36 KB
constexpr int kOffStage8 = S16 * kStage16;
constexpr int kOffBar = kOffStage8 + S8 * kStage8;
constexpr int kBarBytes = 8 * (2 * S8 + 2 * S16 + 4) + 16;
constexpr int kSmem = kOffBar + kBarBytes + 1024;
constexpr uint32_t kIdesc = idesc_f16(MM, NT);

static_assert(kStage16 % 1024 == 0 && kOffStage8 % 1024 == 0, "swizzled stages must be 1024-byte aligned");

__global__ void __launch_bounds__(kThreads, 1)
    gemv_tc_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_a,
                   int M, int N, int K, Epilogue ep) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t sraw = smem_u32(smem_raw);
    const uint32_t sbase = (sraw + 1023u) & ~1023u;
    const uint32_t bar_full8 = sbase + kOffBar;
    const uint32_t bar_empty8 = bar_full8 + 8 * S8;
    const uint32_t bar_full16 = bar_empty8 + 8 * S8;
    const uint32_t bar_empty16 = bar_full16 + 8 * S16;
    const uint32_t bar_accfull = bar_empty16 + 8 * S16;
    const uint32_t bar_accempty = bar_accfull + 16;
    uint8_t* smem = smem_raw + (sbase - sraw);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * (2 * S8 + 2 * S16 + 4));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    // Rows MM/2.. of every weight operand stage stay zero for the whole kernel.
    for (int i = threadIdx.x; i < S16 * 2 * (MM - RW) * 8; i += kThreads) {
        const int st = i / (2 * (MM - RW) * 8), rem = i % (2 * (MM - RW) * 8);
        const int atom = rem / ((MM - RW) * 8), r = RW + (rem / 8) % (MM - RW), j = rem % 8;
        sts128(sbase + st * kStage16 + atom * kAtomW + sw128(r, j), make_uint4(0, 0, 0, 0));
    }
    fence_proxy_async_smem();
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
        asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmap_w)) : "memory");
        asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmap_a)) : "memory");
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int tiles = (N + RW - 1) / RW;
    const int KB = (K + BK - 1) / BK;
    const int CPT = (KB + KB_PER_CHUNK - 1) / KB_PER_CHUNK;
    const int my_tiles = (int)blockIdx.x < tiles ? (tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int total_g = my_tiles * KB;
    const int k_rot = (int)(((long long)blockIdx.x * KB) / gridDim.x);

    const bool is_conv = (warp >= 2 && warp < 12) || warp >= 14;
    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kRegsLow));
        if (lane == 0) {
            int i = 0, kb = 0;
            for (int g = 0; g < total_g; ++g) {
                const int n0 = ((int)blockIdx.x + i * (int)gridDim.x) * RW;
                const int s = g % S8;
                if (!mbar_wait(bar_empty8 + 8 * s, (uint32_t)(((g / S8) & 1) ^ 1), abort_flag, kErrProducer,
                               &g_gemv_error))
                    break;
                const uint32_t dst = sbase + kOffStage8 + s * kStage8;
                // Each CTA walks K from its own starting block, so the SMs do not all read
                // the same activation slice (a handful of L2 lines) at the same moment.
                const int kx = (kb + k_rot >= KB ? kb + k_rot - KB : kb + k_rot) * BK;
                mbar_expect_tx(bar_full8 + 8 * s, kStage8);
                tma_load_2d(dst, &tmap_w, kx, n0, bar_full8 + 8 * s);
                tma_load_2d(dst + kW8, &tmap_a, kx, 0, bar_full8 + 8 * s);
                if (++kb == KB) { kb = 0; ++i; }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kRegsLow));
        if (lane == 0) {
            int kb = 0, c = 0;
            for (int g = 0; g < total_g; ++g) {
                const bool first = (kb % KB_PER_CHUNK) == 0;
                const bool last = (kb % KB_PER_CHUNK) == KB_PER_CHUNK - 1 || kb == KB - 1;
                const int buf = c & 1;
                if (first) {
                    if (!mbar_wait(bar_accempty + 8 * buf, (uint32_t)(((c >> 1) & 1) ^ 1), abort_flag, kErrMmaAcc,
                                   &g_gemv_error))
                        break;
                    tc_fence_after();
                }
                const int s = g % S16;
                if (!mbar_wait(bar_full16 + 8 * s, (uint32_t)((g / S16) & 1), abort_flag, kErrMmaFull, &g_gemv_error))
                    break;
                tc_fence_after();
                const uint32_t st = sbase + s * kStage16;
#pragma unroll
                for (int kk = 0; kk < kChains; ++kk) {
                    const uint32_t d = tmem_base + (uint32_t)((buf * kChains + kk) * NT);
                    const uint32_t off = (uint32_t)((kk & 3) * 32);   // 16 fp16 along K inside a swizzle column
                    const uint64_t adesc = smem_desc_sw128(st + (kk >> 2) * kAtomW + off);
                    const uint64_t bdesc = smem_desc_sw128(st + kW16 + (kk >> 2) * kAtomA + off);
                    mma_f16(d, adesc, bdesc, kIdesc, first ? 0u : 1u);
                }
                mma_commit(bar_empty16 + 8 * s);
                if (last) {
                    mma_commit(bar_accfull + 8 * buf);
                    ++c;
                }
                if (++kb == KB) kb = 0;
            }
        }
    } else if (is_conv) {
        // ---------------------------------------------------------------- converters
        // Staging rows (0..63 weights, 64..79 tokens) are 128 bytes = 8 chunks of 16 K
        // values, stored by TMA with the 128-byte swizzle (chunk c of row r at c ^ (r & 7)).
        // Thread chunk idx covers row = idx % rows, chunk c = idx / rows of its operand, so
        // eight neighbouring threads touch eight rows of one chunk column: conflict-free
        // for the loads and for the fp16 stores. Chunk c becomes fp16 chunks 2c, 2c+1 of
        // the 256-byte fp16 row, in swizzle column c / 4.
        if (warp < 12) {
            asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kRegsLow));
        } else {
            asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kRegsHigh));
        }
        const int ct = warp < 12 ? threadIdx.x - 64 : threadIdx.x - 128;   // 0 .. 383
        for (int g = 0; g < total_g; ++g) {
            const int s8 = g % S8, s16 = g % S16;
            if (!mbar_wait(bar_full8 + 8 * s8, (uint32_t)((g / S8) & 1), abort_flag, kErrConvFull, &g_gemv_error))
                break;
            const uint32_t st8 = sbase + kOffStage8 + s8 * kStage8;
            uint4 in[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int idx = ct + kConv * j;
                const bool is_w = idx < RW * 8;
                const int li = is_w ? idx : idx - RW * 8;
                const int r = is_w ? (li & (RW - 1)) : (li & (NT - 1));
                const int c = is_w ? (li / RW) : (li / NT);
                const uint32_t src = st8 + (is_w ? 0 : kW8) + sw128(r, c);
                in[j] = idx < kChunks8 ? lds128(src) : make_uint4(0, 0, 0, 0);
            }
            if (!mbar_wait(bar_empty16 + 8 * s16, (uint32_t)(((g / S16) & 1) ^ 1), abort_flag, kErrConvEmpty,
                           &g_gemv_error))
                break;
            const uint32_t st16 = sbase + s16 * kStage16;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int idx = ct + kConv * j;
                if (idx < kChunks8) {
                    const bool is_w = idx < RW * 8;
                    const int li = is_w ? idx : idx - RW * 8;
                    const int r = is_w ? (li & (RW - 1)) : (li & (NT - 1));
                const int c = is_w ? (li / RW) : (li / NT);
                    const int atom = c >> 2, w0 = (2 * c) & 7;
                    const uint32_t region = is_w ? st16 + atom * kAtomW : st16 + kW16 + atom * kAtomA;
                    uint4 o0, o1;
                    cvt_word(in[j].x, o0.x, o0.y);
                    cvt_word(in[j].y, o0.z, o0.w);
                    cvt_word(in[j].z, o1.x, o1.y);
                    cvt_word(in[j].w, o1.z, o1.w);
                    sts128(region + sw128(r, w0), o0);
                    sts128(region + sw128(r, w0 + 1), o1);
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(bar_full16 + 8 * s16);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty8 + 8 * s8);   // after the loaded registers were consumed
        }
    } else {
        // ---------------------------------------------------------------- drain + epilogue
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kRegsHigh));
        const int quarter = warp & 3;   // warps 12, 13: weight rows 0..31 / 32..63 of the tile
        int acc[NT];
#pragma unroll
        for (int j = 0; j < NT; ++j) acc[j] = 0;
        const int chunks_total = my_tiles * CPT;
        int ti = 0, cc = 0;
        for (int c = 0; c < chunks_total; ++c, (++cc == CPT ? (cc = 0, ++ti) : 0)) {
            const int buf = c & 1;
            if (!mbar_wait(bar_accfull + 8 * buf, (uint32_t)((c >> 1) & 1), abort_flag, kErrDrain, &g_gemv_error))
                break;
            tc_fence_after();
            const int keep = cc != 0;
#pragma unroll
            for (int j = 0; j < NT; ++j) acc[j] *= keep;
#pragma unroll 1
            for (int kk = 0; kk < kChains; ++kk) {
                uint32_t v[16];
                tmem_ld16(tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)((buf * kChains + kk) * NT), v);
#pragma unroll
                for (int j = 0; j < NT; ++j) acc[j] += __float2int_rn(__uint_as_float(v[j]));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_accempty + 8 * buf);
            if (cc != CPT - 1) continue;
            const int n = ((int)blockIdx.x + ti * (int)gridDim.x) * RW + quarter * 32 + lane;
            if (n < N) {
                if (ep.out_i32) {
#pragma unroll
                    for (int j = 0; j < NT; ++j)
                        if (j < M) ep.out_i32[(int64_t)j * N + n] = acc[j];
                } else {
                    const float sw = __ldg(ep.s_w + (ep.w_per_row ? n : 0));
                    const int cs = ep.z_a ? __ldg(ep.colsum + n) : 0;
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        if (j < M) {
                            const int r = ep.a_per_row ? j : 0;
                            const int corr = ep.z_a ? acc[j] - __ldg(ep.z_a + r) * cs : acc[j];
                            epi_store(ep, (int64_t)j * N + n,
                                      epi_bias(ep, __fmul_rn(__int2float_rn(corr), __fmul_rn(__ldg(ep.s_a + r), sw)), n));
                        }
                    }
                }
            }
        }
    }

    __syncthreads();
    if (*abort_flag) {
        const long long t0 = clock64();
        while (clock64() - t0 < (1LL << 22)) __nanosleep(1000);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

}  // namespace

bool gemv_tc_supports(int64_t M, int64_t N, int64_t K) {
    if (!(M >= 1 && M <= NT && N >= 1 && N < (1LL << 31) && K >= 16 && (K % 16) == 0)) return false;
    const int64_t tiles = (N + RW - 1) / RW;
    const int64_t kb = (K + BK - 1) / BK;
    return tiles * kb < (1LL << 31);
}

cudaError_t launch_gemv_tc(const int8_t* qa, const int8_t* qw, int64_t M, int64_t N, int64_t K,
                           const Epilogue& ep, cudaStream_t stream) {
    if (!gemv_tc_supports(M, N, K)) return cudaErrorNotSupported;
    CUtensorMap mw, ma;
    if (!make_tma_map_i8(&mw, qw, N, K, RW, BK, true) || !make_tma_map_i8(&ma, qa, M, K, NT, BK, true))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(gemv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    const int64_t tiles = (N + RW - 1) / RW;
    const int sms = device_sm_count();
    const int grid = (int)(tiles < sms ? tiles : sms);
    gemv_tc_kernel<<<grid, kThreads, kSmem, stream>>>(mw, ma, (int)M, (int)N, (int)K, ep);
    note_launch();
    return cudaGetLastError();
}

cudaError_t read_and_clear_gemv_tc_error(uint32_t* code) {
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_gemv_error, sizeof(v));
    if (e != cudaSuccess) return e;
    *code = v;
    if (v) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_gemv_error, &zero, sizeof(zero));
    }
    return e;
}

}  // namespace q8
