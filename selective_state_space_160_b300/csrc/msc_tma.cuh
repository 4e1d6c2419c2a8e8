// msc_tma.cuh -- TMA (cp.async.bulk.tensor) and mbarrier helpers for sm_103a,
// written as inline PTX, plus the host-side tensor-map encoder.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "msc_common.cuh"

namespace msc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async (TMA / tensor core) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Arrive once and announce `bytes` of transaction data (TMA completions).
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// The same test, but a thread whose phase is not complete is suspended until it
// completes or about `hint_ns` nanoseconds pass, instead of returning at once
// (a waiting warp then takes no issue slots from the warps it waits for).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Bounded wait on phase `parity`: returns false if it did not complete within
// `max_iters` polls (each poll may suspend the warp for a short while).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t max_iters) {
    for (uint32_t i = 0; i < max_iters; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// Wait for phase `parity` of `bar`, giving up after about one second (by the
// global timer), or as soon as *abort becomes non-zero when abort is given, so
// that one role's timeout does not cascade through the others of the block.
// sleep_ns > 0: after a few polls the waiting thread is suspended between tests
// (for roles that wait long, such as an MMA issuer or an epilogue); 0 keeps
// polling (for short waits inside a tight pipeline).
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity,
                                             const volatile uint32_t* abort = nullptr, uint32_t sleep_ns = 0) {
    if (mbar_wait(bar, parity, sleep_ns ? 4u : 256u)) return true;
    uint64_t t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    while (true) {
        if (sleep_ns ? mbar_try_wait_sleep(bar, parity, sleep_ns) : mbar_try_wait(bar, parity)) return true;
        if (abort && *abort) return false;
        uint64_t t1;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
        if (t1 - t0 > 1000000000ull) return false;
    }
}

// cp.async.bulk global -> shared (16-byte aligned addresses, size a multiple of
// 16), completion counted on `bar`
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// 32-byte streaming store of 8 floats (sm_100+ 256-bit global access); p is
// 32-byte aligned
__device__ __forceinline__ void st_cs_v8(float* p, const float* v) {
    asm volatile("st.global.cs.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "f"(v[0]), "f"(v[1]),
                 "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
                 : "memory");
}

// 3-D tiled TMA load into shared memory, completion counted on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0,
                                            int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0,
                                            int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Byte offset of 16-byte chunk `c` of row `r` in a tile of 64-byte rows written
// by TMA with CU_TENSOR_MAP_SWIZZLE_64B (address bits [4,6) ^= bits [7,9)).
__device__ __forceinline__ uint32_t sw64(uint32_t r, uint32_t c) {
    return r * 64u + ((c ^ ((r >> 1) & 3u)) << 4);
}

// -------------------------------------------------------- packed fp32 pairs
// fma/mul on two fp32 lanes at once (sm_100+): one issue slot for two results.
__device__ __forceinline__ uint64_t pk2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void upk2(uint64_t r, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t ex2_2(uint64_t x) {
    float a, b;
    upk2(x, a, b);
    float ra, rb;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(ra) : "f"(a));
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(rb) : "f"(b));
    return pk2(ra, rb);
}
__device__ __forceinline__ uint64_t rcp_2(uint64_t x) {
    float a, b;
    upk2(x, a, b);
    float ra, rb;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(ra) : "f"(a));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rb) : "f"(b));
    return pk2(ra, rb);
}

// softplus of two values, each half exactly as softplus_f (msc_common.cuh):
// max(x, 0) + ln2 log2(1 + e^{-|x|}), the log term by MUFU lg2 (a series for
// e^{-|x|} < 2^-6).
__device__ __forceinline__ uint64_t softplus_2(uint64_t x) {
    float x0, x1;
    upk2(x, x0, x1);
    float w0, w1;
    upk2(ex2_2(pk2(-fabsf(x0) * MSC_LOG2E, -fabsf(x1) * MSC_LOG2E)), w0, w1);
    return fma2(pk2(log2_1p_unit(w0), log2_1p_unit(w1)), pk2(MSC_LN2, MSC_LN2), pk2(fmaxf(x0, 0.f), fmaxf(x1, 0.f)));
}

// silu of two values: z / (1 + e^-z)
__device__ __forceinline__ uint64_t silu_2(uint64_t z) {
    float z0, z1;
    upk2(z, z0, z1);
    const uint64_t e = ex2_2(pk2(-z0 * MSC_LOG2E, -z1 * MSC_LOG2E));
    return mul2(z, rcp_2(add2(e, pk2(1.f, 1.f))));
}

}  // namespace msc

namespace msc_host {
// Encodes a tiled tensor map (driver entry point resolved at run time, so the
// library does not link libcuda).  dims/strides are innermost first; strides
// are in bytes for dims 1..rank-1.  Returns false (with msc_last_error set) on
// failure.
bool encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                 const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                 CUtensorMapSwizzle swizzle);
}  // namespace msc_host
