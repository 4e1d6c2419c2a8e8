// msc_common.cuh -- device helpers shared by the libmsc kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "msc.h"

#define MSC_LOG2E 1.4426950408889634f
#define MSC_LN2 0.6931471805599453f

namespace msc {

// ---------------------------------------------------------------- SFU helpers
// ex2.approx on the special-function unit: one MUFU op, flushes denormals.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// log2(1 + w) for w in [0, 1]: MUFU lg2 of 1 + w for w >= 2^-6; below, where
// lg2's absolute error and the rounding of 1 + w are large against the
// result, the series log2(e) (w - w^2/2 + w^3/3), whose first omitted term
// (w^4/4) is below 3e-7 of the result there.
__device__ __forceinline__ float log2_1p_unit(float w) {
    const float l = lg2_approx(1.f + w);
    const float s = w * fmaf(w, fmaf(w, MSC_LOG2E / 3.f, -0.5f * MSC_LOG2E), MSC_LOG2E);
    return w < 0x1p-6f ? s : l;
}

// softplus(x) = log(1 + e^x) = max(x, 0) + ln2 log2(1 + w), w = e^{-|x|} in (0, 1].
// The log1p term takes MUFU lg2 and a few ALU ops rather than a long FMA-pipe
// series, which leaves the FMA pipe to the recurrence.  For x > 20 the term is
// below half an ulp of x, so the sum rounds to x exactly.  softplus_2 in
// msc_tma.cuh runs the same operations on each half of a pair, so the two give
// identical bits.
__device__ __forceinline__ float softplus_f(float x) {
    const float w = ex2_approx(-fabsf(x) * MSC_LOG2E);
    return fmaf(log2_1p_unit(w), MSC_LN2, fmaxf(x, 0.f));
}

// logistic sigmoid 1 / (1 + e^-x); for x -> -inf, e^-x -> inf and rcp -> 0.
__device__ __forceinline__ float sigmoid_f(float x) {
    return rcp_approx(1.f + ex2_approx(-x * MSC_LOG2E));
}

__device__ __forceinline__ float silu_f(float x) { return x * sigmoid_f(x); }

// ------------------------------------------------------------------ bf16 bits
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

// Load element i of a row that is fp32 (kBF16 = false) or bf16 bits (true).
template <bool kBF16>
__device__ __forceinline__ float ld_elem(const void* p, int64_t i) {
    if constexpr (kBF16) {
        return bf16_to_f(__ldg(reinterpret_cast<const uint16_t*>(p) + i));
    } else {
        return __ldg(reinterpret_cast<const float*>(p) + i);
    }
}

// Load 8 consecutive elements starting at element i (16-byte aligned for bf16,
// 32-byte span for fp32 -- two 16-byte loads) into out[0..7].
template <bool kBF16>
__device__ __forceinline__ void ld8(const void* p, int64_t i, float* out) {
    if constexpr (kBF16) {
        uint4 v = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p) + i));
        out[0] = bf16lo(v.x); out[1] = bf16hi(v.x);
        out[2] = bf16lo(v.y); out[3] = bf16hi(v.y);
        out[4] = bf16lo(v.z); out[5] = bf16hi(v.z);
        out[6] = bf16lo(v.w); out[7] = bf16hi(v.w);
    } else {
        const float4* q = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p) + i);
        float4 a = __ldg(q), b = __ldg(q + 1);
        out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
        out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
    }
}

}  // namespace msc

// ------------------------------------------------------------- host helpers
namespace msc_host {
// Records a message for msc_last_error() on this thread and returns `st`.
msc_status fail(msc_status st, const char* fmt, ...);
// Clears the thread's last error.
void clear_error();
// Checks cudaGetLastError() after a launch; returns MSC_OK or MSC_ERR_CUDA.
msc_status check_launch(const char* what);
int num_sms();
// This thread's current device as one bit (devices 0..63), for launch sites
// that set a kernel attribute once per device.
inline uint64_t device_bit() {
    int d = 0;
    cudaGetDevice(&d);
    return 1ull << (d & 63);
}
}  // namespace msc_host
