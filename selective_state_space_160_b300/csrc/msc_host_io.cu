// msc_host_io.cu -- S6 forward from and to host memory, with the copies
// overlapped with the scan (a chunked, three-stream pipeline over the batch).
//
// Chunk c (cb batch entries) goes through: upload of u, delta, z, B, C into
// staging slot c % 2 (upload stream), the forward on that slot (the caller's
// stream), download of y (download stream).  The upload of chunk c + 1 and the
// download of chunk c - 1 run while chunk c is scanned.  A slot is refilled
// only after the scan of its previous chunk (its inputs) and the download of
// its previous y are done.  The caller's stream waits for the last download,
// so synchronising it makes y complete.  Rows are independent, so the result
// equals one forward over the whole batch (with the same segment plan).
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "msc.h"
#include "msc_common.cuh"

namespace {

size_t a256(size_t x) { return (x + 255) / 256 * 256; }

struct SlotLayout {
    size_t u, delta, z, B, C, y, ws, bytes;  // offsets within one slot, and its size
};

SlotLayout slot_layout(int64_t cb, int64_t dim, int64_t L, int64_t N, size_t es, bool has_z) {
    SlotLayout s{};
    const size_t rows = (size_t)(cb * dim) * (size_t)L, bc = (size_t)(cb * N) * (size_t)L;
    size_t off = 0;
    s.u = off; off += a256(rows * es);
    s.delta = off; off += a256(rows * es);
    s.z = off; off += has_z ? a256(rows * es) : 0;
    s.B = off; off += a256(bc * es);
    s.C = off; off += a256(bc * es);
    s.y = off; off += a256(rows * 4);
    s.ws = off; off += a256(msc_selective_scan_fwd_workspace_size(cb, dim, L, N));
    s.bytes = off;
    return s;
}

// Two non-blocking streams per device (upload, download), made once.
struct IoStreams {
    cudaStream_t up = nullptr, down = nullptr;
};
IoStreams g_streams[64];
std::once_flag g_streams_once[64];

cudaError_t io_streams(IoStreams** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    IoStreams& s = g_streams[dev & 63];
    std::call_once(g_streams_once[dev & 63], [&]() {
        if (cudaStreamCreateWithFlags(&s.up, cudaStreamNonBlocking) != cudaSuccess) s.up = nullptr;
        if (cudaStreamCreateWithFlags(&s.down, cudaStreamNonBlocking) != cudaSuccess) s.down = nullptr;
    });
    if (!s.up || !s.down) return cudaErrorInitializationError;
    *out = &s;
    return cudaSuccess;
}

}  // namespace

extern "C" {

size_t msc_selective_scan_fwd_host_staging_size(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                                msc_dtype in_dtype, int has_z, int64_t chunk_batch) {
    if (batch < 1 || dim < 1 || seqlen < 1 || dstate < 1 || dstate > MSC_S6_FWD_MAX_DSTATE || chunk_batch < 1) return 0;
    if (in_dtype != MSC_F32 && in_dtype != MSC_BF16) return 0;
    const int64_t cb = chunk_batch < batch ? chunk_batch : batch;
    const size_t es = in_dtype == MSC_BF16 ? 2 : 4;
    return 2 * slot_layout(cb, dim, seqlen, dstate, es, has_z != 0).bytes;
}

msc_status msc_selective_scan_fwd_host(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                                       msc_dtype in_dtype, const void* u, const void* delta, const float* A,
                                       const void* B, const void* C, const float* D, const void* z,
                                       const float* delta_bias, float* y, int64_t chunk_batch, void* staging,
                                       size_t staging_bytes, void* stream) {
    msc_host::clear_error();
    if (batch < 1 || dim < 1 || seqlen < 1 || dstate < 1 || chunk_batch < 1)
        return msc_host::fail(MSC_ERR_INVALID_ARG, "batch, dim, seqlen, dstate and chunk_batch must be >= 1");
    if (in_dtype != MSC_F32 && in_dtype != MSC_BF16)
        return msc_host::fail(MSC_ERR_INVALID_ARG, "in_dtype must be MSC_F32 or MSC_BF16");
    if (!u || !delta || !B || !C || !y || !A)
        return msc_host::fail(MSC_ERR_INVALID_ARG, "u, delta, A, B, C and y must not be NULL");
    const int64_t cb = chunk_batch < batch ? chunk_batch : batch;
    const size_t es = in_dtype == MSC_BF16 ? 2 : 4;
    const SlotLayout lay = slot_layout(cb, dim, seqlen, dstate, es, z != nullptr);
    if (staging == nullptr || staging_bytes < 2 * lay.bytes)
        return msc_host::fail(MSC_ERR_WORKSPACE, "staging of %zu bytes required (got %zu)", 2 * lay.bytes,
                              staging ? staging_bytes : (size_t)0);
    if ((reinterpret_cast<uintptr_t>(staging) & 255u) != 0)
        return msc_host::fail(MSC_ERR_INVALID_ARG, "staging must be 256-byte aligned");

    IoStreams* io = nullptr;
    cudaError_t e = io_streams(&io);
    if (e != cudaSuccess) return msc_host::fail(MSC_ERR_CUDA, "io streams: %s", cudaGetErrorString(e));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // events: start, and per slot the last upload, scan and download
    cudaEvent_t ev[7];
    for (int i = 0; i < 7; ++i) {
        e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
        if (e != cudaSuccess) {
            for (int k = 0; k < i; ++k) cudaEventDestroy(ev[k]);
            return msc_host::fail(MSC_ERR_CUDA, "event: %s", cudaGetErrorString(e));
        }
    }
    cudaEvent_t ev_start = ev[0], *ev_up = ev + 1, *ev_scan = ev + 3, *ev_down = ev + 5;
    msc_status res = MSC_OK;
    const size_t row_in = (size_t)dim * (size_t)seqlen * es, bc_in = (size_t)dstate * (size_t)seqlen * es;
    const size_t row_out = (size_t)dim * (size_t)seqlen * 4;
    char* stage = static_cast<char*>(staging);
    const char* hu = static_cast<const char*>(u);
    const char* hd = static_cast<const char*>(delta);
    const char* hz = static_cast<const char*>(z);
    const char* hB = static_cast<const char*>(B);
    const char* hC = static_cast<const char*>(C);
    char* hy = reinterpret_cast<char*>(y);

    // the pipeline starts after the caller's earlier work on its stream
    e = cudaEventRecord(ev_start, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(io->up, ev_start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(io->down, ev_start, 0);
    const int64_t nchunks = (batch + cb - 1) / cb;
    for (int64_t c = 0; c < nchunks && e == cudaSuccess && res == MSC_OK; ++c) {
        const int s = (int)(c & 1);
        const int64_t b0 = c * cb, nb = (batch - b0) < cb ? (batch - b0) : cb;
        char* slot = stage + (size_t)s * lay.bytes;
        // upload: the slot's inputs are free once the scan of chunk c - 2 is done
        if (c >= 2) e = cudaStreamWaitEvent(io->up, ev_scan[s], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(slot + lay.u, hu + b0 * row_in, nb * row_in, cudaMemcpyHostToDevice, io->up);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(slot + lay.delta, hd + b0 * row_in, nb * row_in, cudaMemcpyHostToDevice, io->up);
        if (e == cudaSuccess && z)
            e = cudaMemcpyAsync(slot + lay.z, hz + b0 * row_in, nb * row_in, cudaMemcpyHostToDevice, io->up);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(slot + lay.B, hB + b0 * bc_in, nb * bc_in, cudaMemcpyHostToDevice, io->up);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(slot + lay.C, hC + b0 * bc_in, nb * bc_in, cudaMemcpyHostToDevice, io->up);
        if (e == cudaSuccess) e = cudaEventRecord(ev_up[s], io->up);
        // scan: after the upload, and once the download of chunk c - 2 has read the slot's y
        if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev_up[s], 0);
        if (e == cudaSuccess && c >= 2) e = cudaStreamWaitEvent(st, ev_down[s], 0);
        if (e != cudaSuccess) break;
        res = msc_selective_scan_fwd(nb, dim, seqlen, dstate, in_dtype, slot + lay.u, slot + lay.delta, A,
                                     slot + lay.B, slot + lay.C, D, z ? slot + lay.z : nullptr, delta_bias, nullptr,
                                     reinterpret_cast<float*>(slot + lay.y), nullptr, slot + lay.ws,
                                     lay.bytes - lay.ws, stream);
        if (res != MSC_OK) break;
        e = cudaEventRecord(ev_scan[s], st);
        // download
        if (e == cudaSuccess) e = cudaStreamWaitEvent(io->down, ev_scan[s], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(hy + b0 * row_out, slot + lay.y, nb * row_out, cudaMemcpyDeviceToHost, io->down);
        if (e == cudaSuccess) e = cudaEventRecord(ev_down[s], io->down);
    }
    // the caller's stream completes with the last downloads
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev_down[0], 0);
    if (e == cudaSuccess && nchunks > 1) e = cudaStreamWaitEvent(st, ev_down[1], 0);
    for (int i = 0; i < 7; ++i) cudaEventDestroy(ev[i]);
    if (res != MSC_OK) return res;
    if (e != cudaSuccess) return msc_host::fail(MSC_ERR_CUDA, "host pipeline: %s", cudaGetErrorString(e));
    return MSC_OK;
}

}  // extern "C"
