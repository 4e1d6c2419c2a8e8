// msc_noalloc.cu -- the S6 forward for callers that cannot allocate device memory.
//
// Some callers cannot hand the library a workspace: a plugin loaded into a host
// framework that owns every device allocation and exposes no allocator to it,
// or a latency-critical serving loop that must not call cudaMalloc on its hot
// path (cudaMalloc can synchronise the device and stall unrelated work).  For
// them msc_selective_scan_fwd_noalloc() runs the same kernels as
// msc_selective_scan_fwd() with the segment scratch of long sequences taken
// from a fixed array in device global memory that this file owns.
//
// The array (MSC_STATIC_SCRATCH_BYTES) exists on every device that loads the
// library and stays there until the process exits.  Host code cannot pass the
// array's name to a kernel -- on the host it is only a stand-in for the device
// symbol -- so the device address is looked up once per device with
// cudaGetSymbolAddress, the first time the entry point runs on that device,
// and cached.  Every call shares the array: calls that overlap on the GPU (on
// different streams, or from different host threads) race on it.
#include <cuda_runtime.h>

#include <mutex>

#include "msc.h"
#include "msc_common.cuh"
#include "msc_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[MSC_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 128;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

}  // namespace

extern "C" msc_status msc_selective_scan_fwd_noalloc(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                                     msc_dtype in_dtype, const void* u, const void* delta,
                                                     const float* A, const void* B, const void* C, const float* D,
                                                     const void* z, const float* delta_bias, const float* h0,
                                                     float* y, float* h_last, void* stream) {
    msc_host::clear_error();
    // Only the segment scratch of long sequences with few rows is required: the
    // plan picks its segment count among those whose scratch fits the array
    // (with none, it runs the sequence unsegmented), so `need` stays within it;
    // the check below guards that.  The chained schedule's optional scratch is
    // used when it fits.
    size_t need = 0;
    if (batch >= 1 && dim >= 1 && seqlen >= 1 && dstate >= 1 && dstate <= MSC_S6_FWD_MAX_DSTATE) {
        const msc_host::S6Plan plan =
            msc_host::s6_fwd_plan(batch, dim, seqlen, dstate, (size_t)MSC_STATIC_SCRATCH_BYTES);
        if (plan.workspace_required) need = plan.workspace;
    }
    if (need > (size_t)MSC_STATIC_SCRATCH_BYTES)
        return msc_host::fail(MSC_ERR_WORKSPACE,
                              "this problem needs %zu bytes of scratch; the allocation-free entry point has %u",
                              need, (unsigned)MSC_STATIC_SCRATCH_BYTES);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return msc_host::fail(MSC_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return msc_host::fail(MSC_ERR_UNSUPPORTED, "device ordinal %d too large", dev);
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (g_scratch_addr[dev] == nullptr) {
            // set-up on this device (current here): device address of the array
            void* ptr = nullptr;
            e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
            if (e != cudaSuccess)
                return msc_host::fail(MSC_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
            g_scratch_addr[dev] = ptr;
        }
        scratch = g_scratch_addr[dev];
    }
    // Nothing in the scratch has to start at zero: every value the kernels read
    // from it was written earlier in the same call.
    return msc_host::s6_fwd_entry(batch, dim, seqlen, dstate, in_dtype, (int)MSC_DISC_EULER, u, delta, A, B, C, D,
                                  z, delta_bias, h0, y, h_last, scratch, (size_t)MSC_STATIC_SCRATCH_BYTES, stream,
                                  (size_t)MSC_STATIC_SCRATCH_BYTES);
}
