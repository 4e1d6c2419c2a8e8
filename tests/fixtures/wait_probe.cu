// wait_probe.cu -- test fixture (failure detection), not part of libmsc.
//
// Exercises the library's bounded mbarrier wait (msc::wait_bounded, the wait
// every TMA and tensor-core pipeline of libmsc uses) on the GPU without a hang:
// one CTA waits on a barrier that nothing completes, the wait gives up after
// about one second by the global timer, the CTA records MSC_ERR_TIMEOUT in a
// status word and returns, and the context stays usable.  With `arrive` set a
// thread arrives first and the wait completes at once.
#include <cuda_runtime.h>
#include <stdint.h>

#include "msc.h"
#include "msc_tma.cuh"

namespace {

__global__ void __launch_bounds__(32) wait_probe_kernel(unsigned* status, unsigned long long* ns, int arrive) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        msc::mbar_init(&bar, 1);
        msc::fence_barrier_init();
    }
    __syncthreads();
    if (arrive && threadIdx.x == 0) msc::mbar_arrive(&bar);  // completes phase 0
    unsigned long long t0, t1;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    const bool ok = msc::wait_bounded(&bar, 0u);
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
    // every thread takes the same branch (no thread is left at a barrier)
    const bool failed = __syncthreads_or(!ok);
    if (threadIdx.x == 0) {
        status[0] = failed ? (unsigned)MSC_ERR_TIMEOUT : 0u;
        ns[0] = t1 - t0;
    }
}

}  // namespace

extern "C" {

// Runs the probe once.  *status_out: 0 when the wait completed, MSC_ERR_TIMEOUT
// when it gave up; *seconds_out: how long the wait took.  Returns 0 or the CUDA
// error code.
int msc_probe_wait_timeout(int arrive, unsigned* status_out, double* seconds_out) {
    unsigned* d_status = nullptr;
    unsigned long long* d_ns = nullptr;
    cudaError_t e = cudaMalloc(&d_status, sizeof(unsigned));
    if (e != cudaSuccess) return (int)e;
    e = cudaMalloc(&d_ns, sizeof(unsigned long long));
    if (e != cudaSuccess) {
        cudaFree(d_status);
        return (int)e;
    }
    wait_probe_kernel<<<1, 32>>>(d_status, d_ns, arrive);
    e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    unsigned st = 0;
    unsigned long long ns = 0;
    if (e == cudaSuccess) e = cudaMemcpy(&st, d_status, sizeof(st), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(&ns, d_ns, sizeof(ns), cudaMemcpyDeviceToHost);
    cudaFree(d_status);
    cudaFree(d_ns);
    if (e != cudaSuccess) return (int)e;
    *status_out = st;
    *seconds_out = (double)ns * 1e-9;
    return 0;
}

}  // extern "C"
