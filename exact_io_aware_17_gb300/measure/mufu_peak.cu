// Throughput of the exponential unit: ex2.approx.f32 (the instruction the softmax uses), issued from
// every SM with enough independent work to keep the unit busy.  A measurement program, not part of
// libfa.so: exact_io_aware_17_gb300/mufu_peak.py compiles and runs it.
//
// Each thread runs kChains independent chains x <- -ex2(x); with x in [-1, -0.5] every value stays in
// range.  The result is written out so that nothing is optimised away.
#include <cstdio>
#include <cuda_runtime.h>

constexpr int kChains = 8;

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__global__ void __launch_bounds__(256) ex2_loop(int iters, float* out, long long* cycles) {
    float x[kChains];
#pragma unroll
    for (int c = 0; c < kChains; ++c) x[c] = -0.5f - 0.05f * (float)c - 1e-4f * (float)(threadIdx.x & 7);
    const long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int c = 0; c < kChains; ++c) x[c] = -ex2_approx(x[c]);
    }
    const long long t1 = clock64();
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < kChains; ++c) s += x[c];
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

int main() {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int blocks = sms * 8, threads = 256, iters = 4096;
    float* out;
    long long* cyc;
    cudaMalloc(&out, sizeof(float) * blocks * threads);
    cudaMalloc(&cyc, sizeof(long long) * blocks);
    cudaEvent_t a, b;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    ex2_loop<<<blocks, threads>>>(iters, out, cyc);   // warm-up
    float best_ms = 1e30f;
    for (int rep = 0; rep < 5; ++rep) {
        cudaEventRecord(a);
        ex2_loop<<<blocks, threads>>>(iters, out, cyc);
        cudaEventRecord(b);
        cudaEventSynchronize(b);
        float ms = 0.f;
        cudaEventElapsedTime(&ms, a, b);
        best_ms = ms < best_ms ? ms : best_ms;
    }
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        printf("{\"error\": \"%s\"}\n", cudaGetErrorString(e));
        return 1;
    }
    long long* h = new long long[blocks];
    cudaMemcpy(h, cyc, sizeof(long long) * blocks, cudaMemcpyDeviceToHost);
    double mean_cycles = 0;
    for (int i = 0; i < blocks; ++i) mean_cycles += (double)h[i];
    mean_cycles /= blocks;
    const double ex2_total = (double)blocks * threads * iters * kChains;
    // 8 blocks of 256 threads per SM run together (2048 threads): per-SM rate = that SM's ex2 / cycles.
    const double per_sm_clk = (double)8 * threads * iters * kChains / mean_cycles;
    printf("{\"ex2_per_s\": %.6e, \"ex2_per_sm_per_clk\": %.2f, \"sms\": %d, \"ms\": %.4f}\n",
           ex2_total / (best_ms * 1e-3), per_sm_clk, sms, best_ms);
    delete[] h;
    return 0;
}
