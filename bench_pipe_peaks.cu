// bench_pipe_peaks.cu -- measurement probe for bench.py, not part of libmsc.
//
// Measures the per-SM throughput of the pipes the S6 scan is bound by, on the
// GPU it runs on: MUFU ex2 (ex2.approx.ftz.f32), MUFU rcp, FP32 FFMA and the
// packed FFMA2 (fma.rn.f32x2).  Each thread runs 8 independent dependency
// chains so the pipe, not latency, limits the rate; every SM holds 32 warps.
// bench.py uses the results as the SFU / FP32 roofline denominators.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr int kChains = 8;

template <int kOp>
__global__ void __launch_bounds__(256) pipe_kernel(float* sink, unsigned long long* cycles, int iters,
                                                   float seed) {
    float x[kChains];
#pragma unroll
    for (int c = 0; c < kChains; ++c) x[c] = seed + 0.001f * (threadIdx.x + c);
    uint64_t xv[kChains];
    if (kOp == 2) {
#pragma unroll
        for (int c = 0; c < kChains; ++c)
            asm("mov.b64 %0, {%1, %2};" : "=l"(xv[c]) : "f"(x[c]), "f"(x[c] + 0.5f));
    }
    uint64_t av, bv;
    asm("mov.b64 %0, {%1, %2};" : "=l"(av) : "f"(0.999f), "f"(0.998f));
    asm("mov.b64 %0, {%1, %2};" : "=l"(bv) : "f"(1e-3f), "f"(2e-3f));
    __syncthreads();
    unsigned long long t0 = clock64();
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int c = 0; c < kChains; ++c) {
            if (kOp == 0) {
                // x in [0.5, 1] stays there: ex2(-x) in [0.5, 0.71]
                asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(x[c]) : "f"(-x[c]));
            } else if (kOp == 1) {
                asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(x[c]) : "f"(0.999f), "f"(1e-3f));
            } else if (kOp == 2) {
                asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(xv[c]) : "l"(av), "l"(bv));
            } else {
                // x <- rcp(x + 1): x in [0.5, 1] stays in [0.5, 0.67]; the add keeps
                // the chain from being an involution (rcp of rcp) that folds away
                asm volatile("add.f32 %0, %0, 0f3F800000;\n\trcp.approx.ftz.f32 %0, %0;" : "+f"(x[c]));
            }
        }
    }
    unsigned long long t1 = clock64();
    __syncthreads();
    float acc = 0.f;
    if (kOp == 2) {
#pragma unroll
        for (int c = 0; c < kChains; ++c) {
            float a, b;
            asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(xv[c]));
            acc += a + b;
        }
    } else {
#pragma unroll
        for (int c = 0; c < kChains; ++c) acc += x[c];
    }
    if (acc == 12345.678f) sink[threadIdx.x] = acc;  // keeps the chains alive
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

}  // namespace

extern "C" {

// results[4 * op + 0] = operations per second (whole GPU)
// results[4 * op + 1] = operations per SM per clock (from clock64 of the CTAs)
// results[4 * op + 2] = kernel milliseconds,  results[4 * op + 3] = SM count
// op: 0 = ex2, 1 = ffma, 2 = ffma2 (counted as 2 FMAs), 3 = rcp.
// Returns 0 on success, else the CUDA error code.
int msc_probe_pipe_peaks(float* results, int iters) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int blocks = sms * 8, threads = 256;
    float* sink = nullptr;
    unsigned long long* cyc = nullptr;
    cudaError_t e = cudaMalloc(&sink, threads * sizeof(float));
    if (e != cudaSuccess) return (int)e;
    e = cudaMalloc(&cyc, blocks * sizeof(unsigned long long));
    if (e != cudaSuccess) { cudaFree(sink); return (int)e; }
    cudaEvent_t a, b;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    unsigned long long* hcyc = new unsigned long long[blocks];
    for (int op = 0; op < 4; ++op) {
        for (int rep = 0; rep < 3; ++rep) {
            cudaEventRecord(a);
            switch (op) {
                case 0: pipe_kernel<0><<<blocks, threads>>>(sink, cyc, iters, 0.7f); break;
                case 1: pipe_kernel<1><<<blocks, threads>>>(sink, cyc, iters, 0.7f); break;
                case 2: pipe_kernel<2><<<blocks, threads>>>(sink, cyc, iters, 0.7f); break;
                default: pipe_kernel<3><<<blocks, threads>>>(sink, cyc, iters, 0.7f); break;
            }
            cudaEventRecord(b);
        }
        e = cudaEventSynchronize(b);
        if (e != cudaSuccess) break;
        float ms = 0.f;
        cudaEventElapsedTime(&ms, a, b);
        cudaMemcpy(hcyc, cyc, blocks * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
        double maxc = 0;
        for (int i = 0; i < blocks; ++i) maxc = hcyc[i] > maxc ? (double)hcyc[i] : maxc;
        const double per_thread = (double)iters * kChains * (op == 2 ? 2.0 : 1.0);
        const double total = per_thread * blocks * threads;
        results[4 * op + 0] = (float)(total / (ms * 1e-3));
        // 8 CTAs of 256 threads share one SM concurrently
        results[4 * op + 1] = (float)(per_thread * threads * 8 / maxc);
        results[4 * op + 2] = ms;
        results[4 * op + 3] = (float)sms;
    }
    delete[] hcyc;
    cudaEventDestroy(a);
    cudaEventDestroy(b);
    cudaFree(sink);
    cudaFree(cyc);
    return (int)e;
}

}  // extern "C"
