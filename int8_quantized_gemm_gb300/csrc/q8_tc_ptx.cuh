// PTX building blocks shared by the tcgen05 kernels (mbarriers, TMA, tcgen05
// MMA / TMEM, shared-memory vector access, the exact int8 -> fp16 conversion).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace q8 {

namespace tc {

constexpr long long kTimeoutCycles = 1LL << 31;    // about a second

enum : unsigned {
    kErrProducer = 1u,
    kErrConvFull = 2u,
    kErrConvEmpty = 4u,
    kErrMmaFull = 8u,
    kErrMmaAcc = 16u,
    kErrDrain = 32u,
    kErrRelay = 64u     // CTA pairs: the odd CTA's forwarder of converted stages
};


__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity. Returns false if the
// kernel is aborting (another role gave up) or this wait ran out of time
// (limit clock cycles; the failure-path self-test passes a short one).
// sleep_ns > 0 backs off between polls, leaving issue slots to warps that
// share the SM sub-partition (for waiters that are not latency critical).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned code, unsigned int* err_word, unsigned sleep_ns = 0,
                                          long long limit = kTimeoutCycles) {
    if (mbar_try(bar, parity)) return true;
    long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (sleep_ns) __nanosleep(sleep_ns);
        if (mbar_try(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort_flag) return false;
            if (clock64() - t0 > limit) {
                *abort_flag = 1;
                atomicOr(err_word, code);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes in 8-row atoms of 1024 bytes (stride between atoms 1024 bytes).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;             // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;   // stride byte offset: next 8-row atom
    d |= (uint64_t)1 << 46;             // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;             // 128-byte swizzle
    return d;
}

// Instruction descriptor of kind::f16 with fp16 A and B, both K-major, fp32 D.
constexpr uint32_t idesc_f16(int m, int n) {
    return (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
          "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]),
          "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]),
          "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}

// int8 x 4 (one 32-bit word, bytes x0..x3) -> two fp16x2 words holding exactly
// (x0, x2) and (x1, x3). The K order inside each group of four is permuted
// the same way for A and W, which leaves every dot product unchanged.
// Bits 0x64 | (x ^ 0x80) form the fp16 value 1024 + (x + 128); subtracting
// 1152 (0x6480) leaves x exactly.
__device__ __forceinline__ uint32_t hsub_1152(uint32_t v) {
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;\n" : "=r"(r) : "r"(v), "r"(0x64806480u));
    return r;
}
__device__ __forceinline__ void cvt_word(uint32_t w, uint32_t& lo, uint32_t& hi) {
    lo = hsub_1152((w & 0x00FF00FFu) ^ 0x64806480u);
    hi = hsub_1152(((w >> 8) & 0x00FF00FFu) ^ 0x64806480u);
}

// Block-scaled weights. The E8M0 scale byte e as the fp16 power of two 2^(e - 127) in both
// halves (exact for e = 103 .. 142; e = 0 gives 0).
__device__ __forceinline__ uint32_t scale_f16x2(uint32_t e) {
    const float f = __uint_as_float(e << 23);
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(f), "f"(f));
    return r;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;\n" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// cvt_word with each code times the power of two s (h = s in both halves, c = -1152 s):
// 0x6480 | (byte ^ 0x80) is the fp16 1152 + q, and fma(1152 + q, s, -1152 s) = q s, exact
// while -1152 s is an fp16 value (s <= 32).
__device__ __forceinline__ void cvt_word_scaled(uint32_t w, uint32_t h, uint32_t c, uint32_t& lo, uint32_t& hi) {
    const uint32_t l = (w & 0x00FF00FFu) ^ 0x64806480u, u = ((w >> 8) & 0x00FF00FFu) ^ 0x64806480u;
    asm("fma.rn.f16x2 %0, %1, %2, %3;\n" : "=r"(lo) : "r"(l), "r"(h), "r"(c));
    asm("fma.rn.f16x2 %0, %1, %2, %3;\n" : "=r"(hi) : "r"(u), "r"(h), "r"(c));
}

// cvt_word with a per-row magic m = (E << 10 | 0x80) in both halves and c = m with both sign
// bits set: (x & 0x00FF00FF) ^ m puts (byte ^ 0x80) = q + 128 in the low mantissa bits of the
// fp16 2^(E - 15) (1 + 128 / 1024), i.e. (1152 + q) 2^(E - 25), and adding c = -1152 2^(E - 25)
// leaves q 2^(E - 25), exactly (1 <= E <= 30).
__device__ __forceinline__ void cvt_word_magic(uint32_t w, uint32_t m, uint32_t c, uint32_t& lo, uint32_t& hi) {
    uint32_t l, u;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;\n" : "=r"(l) : "r"(w), "r"(0x00FF00FFu), "r"(m));
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;\n" : "=r"(u) : "r"(w >> 8), "r"(0x00FF00FFu), "r"(m));
    asm("add.rn.f16x2 %0, %1, %2;\n" : "=r"(lo) : "r"(l), "r"(c));
    asm("add.rn.f16x2 %0, %1, %2;\n" : "=r"(hi) : "r"(u), "r"(c));
}

// Two packed int4 bytes (K 4t, 4t+1 | 4t+2, 4t+3 as low/high nibbles) -> fp16x2 of the low
// nibbles (K 4t, 4t+2) and of the high nibbles (K 4t+1, 4t+3): the pairs cvt_word gives for an
// int8 word, so activations and int4 weights share the K order. SEL picks the two bytes of w
// (0x4140: bytes 0, 1; 0x4342: bytes 2, 3) and spreads them to the low byte of each half.
// A nibble n (two's complement) XOR 8 is n + 8. Low nibbles: (x & 0x000F000F) ^ 0x64086408 sets
// the fp16 exponent of 1024 and flips bit 3 in one lop3, giving 1024 + n + 8; minus 1032 is n.
// High nibbles sit four bits up: (x & 0x00F000F0) ^ 0x64806480 is 1024 + 16 (n + 8), and
// (that / 16) - 72 = n, one fp16 FMA with exact operands and an exact result.
template <uint32_t SEL>
__device__ __forceinline__ void cvt_int4x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    uint32_t x, l, h;
    asm("prmt.b32 %0, %1, 0, %2;\n" : "=r"(x) : "r"(w), "n"(SEL));
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;\n" : "=r"(l) : "r"(x), "r"(0x000F000Fu), "r"(0x64086408u));
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;\n" : "=r"(h) : "r"(x), "r"(0x00F000F0u), "r"(0x64806480u));
    asm("sub.rn.f16x2 %0, %1, %2;\n" : "=r"(lo) : "r"(l), "r"(0x64086408u));
    asm("fma.rn.f16x2 %0, %1, %2, %3;\n" : "=r"(hi) : "r"(h), "r"(0x2C002C00u), "r"(0xD480D480u));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, const uint4& v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// Byte offset of fp16 16-byte chunk j (0..7) of row r in a 128B-swizzled K-major tile.
__device__ __forceinline__ uint32_t sw128(int r, int j) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((j ^ (r & 7)) << 4));
}


__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}

// Each thread of the warp writes 32 consecutive 32-bit columns of its TMEM lane (the warp's
// lane quarter, in taddr), then waits until the stores have completed.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
        "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
        "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(slot_smem), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}

// TMA tensor store of a box from shared memory (bulk-group completion), and the waits on
// the issuing thread's bulk groups: ".read" only until the shared-memory source has been read.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];\n" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
}
// The same box added element-wise into global memory (the tensor map's element type, here
// int32: exact and order-independent), for K-split partial sums.
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
    asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];\n" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }

// ------------------------------------------------------------------ CTA pairs (cta_group::2)
// Two CTAs of a cluster share one MMA: the even CTA issues it, A rows and B rows
// are split between the pair's shared memories, and each CTA's tensor memory
// holds the accumulator rows of its own A half.

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}

// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Arrive on an mbarrier of any CTA in the cluster (release at cluster scope).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];\n" ::"r"(cluster_addr) : "memory");
}

// Arrive on an mbarrier of another CTA of the cluster with the instruction's default
// ordering (release at CTA scope). For announcing data that sits in the arriving CTA's
// own shared memory, already made visible to the async proxy (the pair MMA reads each
// CTA's operand half through that CTA's shared memory), or for handing back a buffer.
// A cluster-scope release costs a memory fence of several hundred nanoseconds per
// arrive, which serialises a per-stage hand-off.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];\n" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ bool mbar_try_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\n"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait (as mbar_wait) for a barrier that CTAs of the cluster arrive on.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                  unsigned code, unsigned int* err_word) {
    if (mbar_try_cluster(bar, parity)) return true;
    long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_cluster(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort_flag) return false;
            if (clock64() - t0 > kTimeoutCycles) {
                *abort_flag = 1;
                atomicOr(err_word, code);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void mma_f16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Pair MMA with A from tensor memory: each CTA's A half sits in its own TMEM lanes 0..127
// at column a_tmem (a 32-bit column holds two consecutive fp16 K elements of a row).
__device__ __forceinline__ void mma_f16_pair_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on the barrier at offset `bar` of every CTA in `mask` once the pair's MMAs complete.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n" ::"r"(
            bar),
        "h"(mask)
        : "memory");
}

// Collective over one warp in each CTA of the pair.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(slot_smem), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}

}  // namespace tc

// Host side: TMA descriptor of a row-major int8 [rows, K] matrix with box
// [box_rows, box_k] and zero fill outside; swizzle128 stores each 128-byte box
// row with its 16-byte chunks XOR-permuted by (row % 8) (box_k must be 128).
// False if the driver entry point is missing.
bool make_tma_map_i8(CUtensorMap* map, const int8_t* base, int64_t rows, int64_t K, int box_rows, int box_k,
                     bool swizzle128 = false);
// fp16 [rows, K] row-major, box [box_rows, box_k] (box_k * 2 == 128 bytes), 128-byte swizzle: the
// K-major layout of the UMMA descriptors. False unless the base and row pitch are 16-byte multiples.
bool make_tma_map_f16(CUtensorMap* map, const uint16_t* base, int64_t rows, int64_t K, int box_rows, int box_k);
// Same with box [box_rows, 64] and the 64-byte swizzle: the 16-byte chunk c of row r
// lands at chunk c ^ ((r >> 1) & 3) of its 64-byte row (shared-memory base 512-byte aligned).
bool make_tma_map_i8_sw64(CUtensorMap* map, const int8_t* base, int64_t rows, int64_t K, int box_rows);
// Output map for TMA stores of a row-major [rows, cols] matrix of fp32, int32, bf16 or int8:
// box [32 rows, 128 bytes of columns] with the 128-byte swizzle. False unless the row pitch
// is a multiple of 16 bytes and the base is 16-byte aligned.
enum { kMapF32 = 0, kMapI32 = 1, kMapBF16 = 2, kMapI8 = 3 };
bool make_tma_map_out(CUtensorMap* map, void* base, int kind, int64_t rows, int64_t cols);
int device_sm_count();

}  // namespace q8
