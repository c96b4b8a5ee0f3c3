// Check of the division used by the fused RMSNorm quantizer (test tool, not part of the library):
// q0 = RN(x r) with r = RN(1 / d), then q1 = RN(q0 + RN(x - q0 d) r) by two FMAs (Markstein's
// correction), compared bit for bit with CUDA's IEEE division __fdiv_rn(x, d) for significand
// pairs x, d in [1, 2) (scaling either by a power of two scales every step exactly while all
// values stay normal). Usage: markstein_check [divisor_stride]: every x significand (2^23) against
// the divisor significands 0, stride, 2 stride, ... (stride 1: all 2^46 pairs). Prints the number
// of checks and of mismatches; exits 0 iff there is none.
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cuda_runtime.h>

__global__ void sweep(uint32_t d_first, uint32_t d_stride, uint32_t d_count, unsigned long long* cnt) {
    unsigned long long bad = 0, checks = 0;
    const uint64_t total = (uint64_t)d_count << 23;
    for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < total; i += (uint64_t)gridDim.x * blockDim.x) {
        const uint32_t dm = d_first + d_stride * (uint32_t)(i >> 23);
        const float d = __uint_as_float(0x3F800000u | (dm & 0x7FFFFFu));
        const float x = __uint_as_float(0x3F800000u | (uint32_t)(i & 0x7FFFFFu));
        const float r = __fdiv_rn(1.0f, d);
        const float q0 = __fmul_rn(x, r);
        const float q1 = __fmaf_rn(__fmaf_rn(-q0, d, x), r, q0);
        bad += __float_as_uint(q1) != __float_as_uint(__fdiv_rn(x, d));
        ++checks;
    }
    atomicAdd(&cnt[0], checks);
    atomicAdd(&cnt[1], bad);
}

int main(int argc, char** argv) {
    const uint32_t stride = argc > 1 ? (uint32_t)strtoul(argv[1], nullptr, 10) : 4096u;
    if (stride == 0 || stride > (1u << 23)) return 2;
    const uint32_t n_div = ((1u << 23) + stride - 1) / stride;
    unsigned long long* cnt = nullptr;
    if (cudaMalloc(&cnt, 2 * sizeof(unsigned long long)) != cudaSuccess) return 2;
    cudaMemset(cnt, 0, 2 * sizeof(unsigned long long));
    const uint32_t per = 1024;   // divisors per launch
    for (uint32_t k = 0; k < n_div; k += per) {
        const uint32_t count = n_div - k < per ? n_div - k : per;
        sweep<<<152 * 16, 256>>>(k * stride, stride, count, cnt);
    }
    const cudaError_t err = cudaDeviceSynchronize();
    unsigned long long h[2] = {0, 0};
    cudaMemcpy(h, cnt, sizeof(h), cudaMemcpyDeviceToHost);
    printf("%s checks %llu mismatches %llu\n", cudaGetErrorString(err), h[0], h[1]);
    return (err == cudaSuccess && h[1] == 0 && h[0] == ((unsigned long long)n_div << 23)) ? 0 : 1;
}
