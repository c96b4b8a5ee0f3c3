// The W8A8 layer on host buffers: activations in host memory -> output in host memory,
// with the host <-> device copies overlapped with the device work.
//
// The token rows are processed in slices of R rows. Slice i is copied to the device on
// a copy-in stream, quantized per token and multiplied on the caller's stream, and its
// output copied back on a copy-out stream; slices alternate between two workspace slots,
// so the copy of slice i + 1 in, the GEMM of slice i and the copy of slice i - 1 out run
// at the same time. Per-token quantization acts row by row, so the result is the same
// as one call over all rows.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "q8_internal.h"

namespace {

constexpr int kMaxDevices = 64;

// Per device, created by the first call on it and kept until exit: the two copy streams
// and the events that order the slots (entry, then per slot: copied in, computed, copied out).
struct HostPipe {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t entry = nullptr, ev_in[2] = {}, ev_comp[2] = {}, ev_out[2] = {};
};
HostPipe g_pipes[kMaxDevices];
std::mutex g_pipe_mu;

void destroy_pipe(HostPipe& p) {
    if (p.in) cudaStreamDestroy(p.in);
    if (p.out) cudaStreamDestroy(p.out);
    cudaEvent_t* evs[7] = {&p.entry, &p.ev_in[0], &p.ev_in[1], &p.ev_comp[0], &p.ev_comp[1], &p.ev_out[0],
                           &p.ev_out[1]};
    for (cudaEvent_t* e : evs)
        if (*e) cudaEventDestroy(*e);
    p = HostPipe{};
}

// Called with g_pipe_mu held.
bool pipe_ready(HostPipe& p) {
    if (p.ready) return true;
    bool ok = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) == cudaSuccess;
    cudaEvent_t* evs[7] = {&p.entry, &p.ev_in[0], &p.ev_in[1], &p.ev_comp[0], &p.ev_comp[1], &p.ev_out[0],
                           &p.ev_out[1]};
    for (cudaEvent_t* e : evs) ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        destroy_pipe(p);
        (void)cudaGetLastError();
        return false;
    }
    p.ready = true;
    return true;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int64_t chunk_rows_for(int64_t M, int64_t chunk_rows) {
    if (chunk_rows > 0) return chunk_rows < M ? chunk_rows : M;
    // default: about sixteen slices, whole 256-row GEMM tiles (the first copy in and the last
    // copy out, which nothing overlaps, stay short; at 8192 x 16384 -> 8192, 16 slices took
    // 3.22 ms against 3.62 ms for 4 and 3.31 ms for 32)
    int64_t r = ((M + 15) / 16 + 255) / 256 * 256;
    return r < M ? r : M;
}

struct Slot {
    float* a;
    int8_t* qa;
    float* s_a;
    int32_t* z_a;
    float* y;
};

size_t slot_bytes(int64_t R, int64_t N, int64_t K) {
    return align256((size_t)R * K * 4) + align256((size_t)R * K) + 2 * align256((size_t)R * 4) +
           align256((size_t)R * N * 4);
}

Slot slot_at(void* ws, size_t bytes_per_slot, int64_t R, int64_t N, int64_t K, int i) {
    uint8_t* p = static_cast<uint8_t*>(ws) + (size_t)i * bytes_per_slot;
    Slot s;
    s.a = reinterpret_cast<float*>(p);
    p += align256((size_t)R * K * 4);
    s.qa = reinterpret_cast<int8_t*>(p);
    p += align256((size_t)R * K);
    s.s_a = reinterpret_cast<float*>(p);
    p += align256((size_t)R * 4);
    s.z_a = reinterpret_cast<int32_t*>(p);
    p += align256((size_t)R * 4);
    s.y = reinterpret_cast<float*>(p);
    (void)N;
    return s;
}

q8_status status_of(cudaError_t e) { return e == cudaSuccess ? Q8_OK : Q8_ERR_CUDA; }

}  // namespace

extern "C" size_t q8_linear_host_workspace(int64_t M, int64_t N, int64_t K, int64_t chunk_rows) {
    if (M <= 0 || N < 0 || K < 0 || chunk_rows < 0) return 0;
    const int64_t R = chunk_rows_for(M, chunk_rows);
    return 2 * slot_bytes(R, N, K);
}

// The argument checks of the host-buffer layer (everything but the workspace). Q8_OK with
// *empty set when there is nothing to do.
static q8_status check_host_args(const float* a_host, int64_t M, int64_t K, q8_symmetry sym, const int8_t* qw,
                                 const float* s_w, q8_granularity gw, const int32_t* colsum, int64_t N,
                                 const float* y_host, int64_t chunk_rows, bool* empty) {
    *empty = false;
    if (M < 0 || N < 0 || K < 0 || chunk_rows < 0) return Q8_ERR_INVALID_ARG;
    if (sym != Q8_SYMMETRIC && sym != Q8_ASYMMETRIC) return Q8_ERR_INVALID_ARG;
    if (gw != Q8_PER_TENSOR && gw != Q8_PER_ROW) return Q8_ERR_INVALID_ARG;
    if (K % 16 != 0 || K > (sym == Q8_ASYMMETRIC ? 65792 : 131056)) return Q8_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) {
        *empty = true;
        return Q8_OK;
    }
    if (!a_host && K > 0) return Q8_ERR_INVALID_ARG;
    if (!y_host || !s_w || (K > 0 && !qw)) return Q8_ERR_INVALID_ARG;
    if (sym == Q8_ASYMMETRIC && !colsum) return Q8_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(qw) & 15) != 0 || (reinterpret_cast<uintptr_t>(s_w) & 3) != 0 ||
        (reinterpret_cast<uintptr_t>(colsum) & 3) != 0)
        return Q8_ERR_INVALID_ARG;
    return Q8_OK;
}

extern "C" q8_status q8_linear_host(const float* a_host, int64_t M, int64_t K, q8_symmetry sym, const int8_t* qw,
                                    const float* s_w, q8_granularity gw, const int32_t* colsum, int64_t N,
                                    float* y_host, int64_t chunk_rows, void* workspace, size_t workspace_bytes,
                                    q8_stream_t stream) {
    bool empty = false;
    const q8_status chk = check_host_args(a_host, M, K, sym, qw, s_w, gw, colsum, N, y_host, chunk_rows, &empty);
    if (chk != Q8_OK || empty) return chk;
    const int64_t R = chunk_rows_for(M, chunk_rows);
    const size_t per_slot = slot_bytes(R, N, K);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0 || workspace_bytes < 2 * per_slot)
        return Q8_ERR_INVALID_ARG;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return Q8_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_pipe_mu);   // the device's streams and events serve one call at a time
    HostPipe& p = g_pipes[dev];
    if (!pipe_ready(p)) return Q8_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    // The copy streams start after the work already queued on the caller's stream (an earlier
    // call may still read this workspace).
    cudaError_t e = cudaEventRecord(p.entry, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p.in, p.entry, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p.out, p.entry, 0);
    if (e != cudaSuccess) return Q8_ERR_CUDA;

    const int64_t chunks = (M + R - 1) / R;
    q8_status st = Q8_OK;
    for (int64_t i = 0; i < chunks && st == Q8_OK; ++i) {
        const int b = (int)(i & 1);
        const Slot sl = slot_at(workspace, per_slot, R, N, K, b);
        const int64_t r0 = i * R, rows = (M - r0) < R ? (M - r0) : R;
        // in: slot b's activations are free once the quantizer of slice i - 2 has read them
        if (i >= 2) e = cudaStreamWaitEvent(p.in, p.ev_comp[b], 0);
        if (e == cudaSuccess && K > 0)
            e = cudaMemcpyAsync(sl.a, a_host + r0 * K, (size_t)rows * K * 4, cudaMemcpyHostToDevice, p.in);
        if (e == cudaSuccess) e = cudaEventRecord(p.ev_in[b], p.in);
        // compute: after the copy in, and once slice i - 2's output has left slot b
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, p.ev_in[b], 0);
        if (e == cudaSuccess && i >= 2) e = cudaStreamWaitEvent(s, p.ev_out[b], 0);
        if (e != cudaSuccess) {
            st = Q8_ERR_CUDA;
            break;
        }
        int32_t* z = sym == Q8_ASYMMETRIC ? sl.z_a : nullptr;
        st = q8_linear(sl.a, rows, K, Q8_PER_ROW, sym, sl.qa, sl.s_a, z, qw, s_w, gw, z ? colsum : nullptr, N, sl.y,
                       stream);
        if (st != Q8_OK) break;
        e = cudaEventRecord(p.ev_comp[b], s);
        // out: after the compute of slice i
        if (e == cudaSuccess) e = cudaStreamWaitEvent(p.out, p.ev_comp[b], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(y_host + r0 * N, sl.y, (size_t)rows * N * 4, cudaMemcpyDeviceToHost, p.out);
        if (e == cudaSuccess) e = cudaEventRecord(p.ev_out[b], p.out);
        if (e != cudaSuccess) st = Q8_ERR_CUDA;
    }
    // The caller's stream completes only after every slice's output has reached the host (and,
    // on an error, after whatever was queued on the copy streams).
    cudaError_t e2 = cudaEventRecord(p.ev_in[0], p.in);
    if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(s, p.ev_in[0], 0);
    if (e2 == cudaSuccess) e2 = cudaEventRecord(p.ev_out[0], p.out);
    if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(s, p.ev_out[0], 0);
    if (st == Q8_OK && e2 != cudaSuccess) st = status_of(e2);
    return st;
}

// ------------------------------------------------------------------------------------------
// q8_linear_host_static: q8_linear_host with its workspace in a fixed device array of this
// library instead of caller memory, for callers that must not allocate device memory
// themselves (see include/q8.h). The array is kStaticScratchBytes on every device that loads
// the library, held until the process exits, and shared by all calls.

namespace {

constexpr size_t kStaticScratchBytes = (size_t)64 << 20;   // 64 MiB
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch on the current device (host code only sees a stand-in
// for the array). Looked up on every call, with the device current: the first lookup on a
// device loads the module there, later ones are a table lookup, and an address can never be
// stale after a device reset (the module, and with it the array, is then loaded anew).
q8_status static_scratch(void** out) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) {
        (void)cudaGetLastError();
        return Q8_ERR_CUDA;
    }
    *out = p;
    return Q8_OK;
}

}  // namespace

extern "C" size_t q8_linear_host_static_limit(void) { return kStaticScratchBytes; }

extern "C" q8_status q8_linear_host_static(const float* a_host, int64_t M, int64_t K, q8_symmetry sym,
                                           const int8_t* qw, const float* s_w, q8_granularity gw,
                                           const int32_t* colsum, int64_t N, float* y_host, int64_t chunk_rows,
                                           q8_stream_t stream) {
    // the same checks, in the same order, as q8_linear_host, before the size check
    bool empty = false;
    const q8_status chk = check_host_args(a_host, M, K, sym, qw, s_w, gw, colsum, N, y_host, chunk_rows, &empty);
    if (chk != Q8_OK || empty) return chk;
    int64_t R = chunk_rows;
    if (R == 0) {
        // the largest slice whose two workspace slots fit in the array (whole 256-row tiles when
        // at least one tile fits)
        if (q8_linear_host_workspace(M, N, K, 1) > kStaticScratchBytes) return Q8_ERR_UNSUPPORTED;
        int64_t lo = 1, hi = M;
        while (lo < hi) {
            const int64_t mid = lo + (hi - lo + 1) / 2;
            if (q8_linear_host_workspace(M, N, K, mid) <= kStaticScratchBytes) lo = mid;
            else hi = mid - 1;
        }
        R = lo >= 256 ? lo / 256 * 256 : lo;
    } else if (q8_linear_host_workspace(M, N, K, R) > kStaticScratchBytes) {
        return Q8_ERR_UNSUPPORTED;
    }
    void* scratch = nullptr;
    const q8_status st = static_scratch(&scratch);
    if (st != Q8_OK) return st;
    return q8_linear_host(a_host, M, K, sym, qw, s_w, gw, colsum, N, y_host, R, scratch, kStaticScratchBytes,
                          stream);
}
