// s6_step.cu -- S6 decode step on sm_103a: one token per channel row, the state
// updated in place.
//
// What it computes, per row (b, d) ("Mamba — 选择性状态空间模型", 实践案例 1: reading
// one token updates the fixed-size state once and reads it out):
//   Delta = softplus(delta + Delta_bias[d])
//   h_n  <- exp(Delta A[d, n]) h_n + Delta B[b, n] u          (exponential Euler)
//   y     = (sum_n C[b, n] h_n + D[d] u) * silu(z)
//
// Design.  The step is bound by HBM: per row the fp32 state (dstate floats) is
// read and written once, u / delta / z are a few bytes, and A (shared across the
// batch) and B, C (shared across channels) are served from L2 and L1.  kLanes
// threads share a row (2 up to 16 states, 4 up to 32, 8 up to 64): thread j
// owns states [8 j, 8 j + 8), so a warp moves 32 / kLanes consecutive rows =
// one contiguous 1 KB block of state per 16-byte access (dstate 16, 32 or 64;
// other sizes take scalar accesses).  The readout partial sums meet in a
// shuffle butterfly; thread 0 of the row applies skip and gate and stores y.
// dstate exps per row ride on the MUFU pipe, far below the bytes.
#include <cuda_runtime.h>

#include "msc_common.cuh"
#include "msc_internal.h"

namespace {

struct StepParams {
    const void* u;
    const void* delta;
    const void* z;
    const void* B;
    const void* C;
    const float* A;
    const float* D;
    const float* delta_bias;
    float* state;
    float* y;
    int64_t rows, dim;
    int N;
};

// kVec: dstate == 8 kLanes (every row and 8-state slice 16-byte aligned)
template <bool kBF16, bool kVec, int kLanes>
__global__ void __launch_bounds__(256) s6_step_kernel(const StepParams p) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int j = threadIdx.x & (kLanes - 1);
    const int64_t row_raw = idx / kLanes;
    const bool row_ok = row_raw < p.rows;
    const int64_t row = row_ok ? row_raw : p.rows - 1;  // out-of-range pairs compute on the last row, store nothing
    const int64_t b = row / p.dim, d = row % p.dim;
    const int N = p.N;
    const int n0 = 8 * j;

    const float uu = msc::ld_elem<kBF16>(p.u, row);
    const float xv = msc::ld_elem<kBF16>(p.delta, row) + (p.delta_bias ? __ldg(p.delta_bias + d) : 0.f);
    const float dt = msc::softplus_f(xv);
    const float dtu = dt * uu;

    float h[8], a[8], bv[8], cv[8];
    float* st = p.state + row * N + n0;
    if constexpr (kVec) {
        const float4 h0 = *reinterpret_cast<const float4*>(st);
        const float4 h1 = *reinterpret_cast<const float4*>(st + 4);
        h[0] = h0.x; h[1] = h0.y; h[2] = h0.z; h[3] = h0.w;
        h[4] = h1.x; h[5] = h1.y; h[6] = h1.z; h[7] = h1.w;
        const float4 a0 = __ldg(reinterpret_cast<const float4*>(p.A + d * N + n0));
        const float4 a1 = __ldg(reinterpret_cast<const float4*>(p.A + d * N + n0) + 1);
        a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w;
        a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
        msc::ld8<kBF16>(p.B, b * N + n0, bv);
        msc::ld8<kBF16>(p.C, b * N + n0, cv);
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const bool on = n0 + k < N;
            h[k] = on ? st[k] : 0.f;
            a[k] = on ? __ldg(p.A + d * N + n0 + k) : 0.f;
            bv[k] = on ? msc::ld_elem<kBF16>(p.B, b * N + n0 + k) : 0.f;
            cv[k] = on ? msc::ld_elem<kBF16>(p.C, b * N + n0 + k) : 0.f;
        }
    }
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        h[k] = fmaf(msc::ex2_approx(dt * a[k] * MSC_LOG2E), h[k], dtu * bv[k]);
        if (k & 1)
            acc1 = fmaf(cv[k], h[k], acc1);
        else
            acc0 = fmaf(cv[k], h[k], acc0);
    }
    float acc = acc0 + acc1;
#pragma unroll
    for (int m = 1; m < kLanes; m *= 2) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (!row_ok) return;
    if (kVec) {
        *reinterpret_cast<float4*>(st) = make_float4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<float4*>(st + 4) = make_float4(h[4], h[5], h[6], h[7]);
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (n0 + k < N) st[k] = h[k];
    }
    if (j == 0) {
        float yv = acc + (p.D ? __ldg(p.D + d) : 0.f) * uu;
        if (p.z) yv *= msc::silu_f(msc::ld_elem<kBF16>(p.z, row));
        p.y[row] = yv;
    }
}

template <bool kBF16, int kLanes>
msc_status launch_lanes(const StepParams& p, cudaStream_t st) {
    const int64_t blocks = (kLanes * p.rows + 255) / 256;
    if (blocks > 0x7FFFFFFF) return msc_host::fail(MSC_ERR_UNSUPPORTED, "batch * dim too large for one launch");
    const unsigned grid = (unsigned)blocks;
    if (p.N == 8 * kLanes)
        s6_step_kernel<kBF16, true, kLanes><<<grid, 256, 0, st>>>(p);
    else
        s6_step_kernel<kBF16, false, kLanes><<<grid, 256, 0, st>>>(p);
    return msc_host::check_launch("s6_step");
}

template <bool kBF16>
msc_status launch(const StepParams& p, cudaStream_t st) {
    if (p.N <= 16) return launch_lanes<kBF16, 2>(p, st);
    if (p.N <= 32) return launch_lanes<kBF16, 4>(p, st);
    return launch_lanes<kBF16, 8>(p, st);
}

}  // namespace

namespace msc_host {

msc_status s6_step_launch(const S6StepArgs& a, cudaStream_t st) {
    StepParams p{};
    p.u = a.u; p.delta = a.delta; p.z = a.z; p.B = a.B; p.C = a.C;
    p.A = a.A; p.D = a.D; p.delta_bias = a.delta_bias; p.state = a.state; p.y = a.y;
    p.rows = a.batch * a.dim; p.dim = a.dim; p.N = a.N;
    return a.bf16 ? launch<true>(p, st) : launch<false>(p, st);
}

}  // namespace msc_host
