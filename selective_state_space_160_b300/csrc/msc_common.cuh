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

// softplus(x) = log(1 + e^x) = max(x, 0) + log1p(w), w = e^{-|x|} in (0, 1].
// log1p(w) = 2 atanh(s) with s = w / (2 + w) in (0, 1/3], summed as the odd
// series 2 (s + s^3/3 + ... + s^13/13); the first omitted term is below 2e-8 of
// the result, so the value is good to a few fp32 ulps for every x.  For x > 20
// the log1p term is below 2.1e-9 and x itself is returned.
__device__ __forceinline__ float softplus_f(float x) {
    if (x > 20.f) return x;
    float w = ex2_approx(-fabsf(x) * MSC_LOG2E);
    float s = w * rcp_approx(2.f + w);
    float s2 = s * s;
    float p = fmaf(s2, 1.f / 13.f, 1.f / 11.f);
    p = fmaf(s2, p, 1.f / 9.f);
    p = fmaf(s2, p, 1.f / 7.f);
    p = fmaf(s2, p, 1.f / 5.f);
    p = fmaf(s2, p, 1.f / 3.f);
    p = fmaf(s2, p, 1.f);
    return fmaxf(x, 0.f) + 2.f * s * p;
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
