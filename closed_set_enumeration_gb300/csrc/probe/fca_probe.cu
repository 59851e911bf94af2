// Roofline probes: LOP3 issue rate and buffer read bandwidth (see include/fca_probe.h).
#include <cuda_runtime.h>

#include <cstdint>

#include "fca_probe.h"

namespace {

constexpr int CHAINS = 8;
constexpr int ROUNDS = 4096;

__device__ __forceinline__ uint32_t lop3_maj(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t r;
    asm volatile("lop3.b32 %0, %1, %2, %3, 0xE8;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

__global__ void __launch_bounds__(256) lop3_kernel(uint32_t *out, uint32_t s0, uint32_t s1)
{
    uint32_t x[CHAINS];
#pragma unroll
    for (int k = 0; k < CHAINS; ++k) x[k] = s0 ^ (threadIdx.x * 2654435761u + k * 40503u + blockIdx.x);
    const uint32_t c0 = s1, c1 = s1 * 3u + 1u;
    for (int i = 0; i < ROUNDS; ++i) {
#pragma unroll
        for (int k = 0; k < CHAINS; ++k) x[k] = lop3_maj(x[k], x[(k + 1) % CHAINS], (k & 1) ? c1 : c0);
    }
    uint32_t acc = 0;
#pragma unroll
    for (int k = 0; k < CHAINS; ++k) acc ^= x[k];
    out[(size_t)blockIdx.x * blockDim.x + threadIdx.x] = acc;
}

__global__ void __launch_bounds__(512) read_kernel(const uint4 *__restrict__ buf, size_t n4, int reps, uint32_t *out)
{
    uint32_t acc = 0;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (int r = 0; r < reps; ++r)
        for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
            const uint4 v = __ldcg(buf + i);
            acc ^= v.x ^ v.y ^ v.z ^ v.w;
        }
    if (acc == 0x9e3779b9u) out[0] = acc;   // practically never taken; keeps the loads alive
}

}  // namespace

extern "C" int fca_probe_lop3(double *ops_per_s, double *ms)
{
    int dev = 0, sms = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return (int)e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return (int)e;
    const int threads = 256, blocks = sms * 8;
    uint32_t *out = nullptr;
    if ((e = cudaMalloc(&out, (size_t)blocks * threads * 4)) != cudaSuccess) return (int)e;
    cudaEvent_t a, b;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    lop3_kernel<<<blocks, threads>>>(out, 12345u, 777u);   // warm-up
    float best = 1e30f;
    for (int r = 0; r < 3; ++r) {
        cudaEventRecord(a);
        lop3_kernel<<<blocks, threads>>>(out, 12345u + r, 777u);
        cudaEventRecord(b);
        cudaEventSynchronize(b);
        float t = 0.f;
        cudaEventElapsedTime(&t, a, b);
        if (t < best) best = t;
    }
    e = cudaGetLastError();
    cudaEventDestroy(a);
    cudaEventDestroy(b);
    cudaFree(out);
    if (e != cudaSuccess) return (int)e;
    const double ops = (double)blocks * threads * CHAINS * ROUNDS;
    if (ms) *ms = best;
    if (ops_per_s) *ops_per_s = ops / (best * 1e-3);
    return 0;
}

extern "C" int fca_probe_read_bw(uint64_t bytes, int reps, double *gbps)
{
    int dev = 0, sms = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return (int)e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return (int)e;
    const size_t n4 = bytes / 16;
    uint4 *buf = nullptr;
    uint32_t *out = nullptr;
    if ((e = cudaMalloc(&buf, n4 * 16)) != cudaSuccess) return (int)e;
    if ((e = cudaMalloc(&out, 16)) != cudaSuccess) { cudaFree(buf); return (int)e; }
    cudaMemset(buf, 1, n4 * 16);
    cudaEvent_t a, b;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    const int threads = 512, blocks = sms * 4;
    const int passes = 8;                              // the buffer is read 8 times per launch
    read_kernel<<<blocks, threads>>>(buf, n4, 1, out);   // warm-up: brings the buffer into L2
    float best = 1e30f;
    for (int r = 0; r < (reps > 0 ? reps : 1); ++r) {
        cudaEventRecord(a);
        read_kernel<<<blocks, threads>>>(buf, n4, passes, out);
        cudaEventRecord(b);
        cudaEventSynchronize(b);
        float t = 0.f;
        cudaEventElapsedTime(&t, a, b);
        if (t < best) best = t;
    }
    e = cudaGetLastError();
    cudaEventDestroy(a);
    cudaEventDestroy(b);
    cudaFree(buf);
    cudaFree(out);
    if (e != cudaSuccess) return (int)e;
    if (gbps) *gbps = (double)(n4 * 16) * passes / (best * 1e-3) / 1e9;
    return 0;
}
