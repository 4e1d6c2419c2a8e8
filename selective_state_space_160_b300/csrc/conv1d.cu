// conv1d.cu -- causal depthwise conv1d + SiLU front end of the Mamba block on sm_103a.
//
// What it computes (bqwf survey sec. 3.1: each Mamba block runs a causal 1-D
// convolution for local context before the selective SSM):
//   out[b, d, t] = silu(bias[d] + sum_{k < K} w[d, k] x[b, d, t - (K - 1) + k]),  x = 0 before t = 0
// and its decode step, which keeps the last K - 1 inputs of every row (study
// note "Mamba — 选择性状态空间模型", 踩过的坑: the convolution still keeps the
// last few inputs when there is no attention cache).
//
// Design.  Both are bound by HBM: per element the sequence kernel reads x once
// (2 or 4 bytes) and writes out once; the K <= 8 weights of a channel and its
// bias are read through L1.  One thread produces 16 consecutive outputs of a
// row: it loads its own two 8-step chunks and the chunk before them (the
// K - 1 halo inputs; the neighbouring thread loads the same chunk, so that
// load hits L1), so a warp reads and writes whole contiguous row segments with
// three 16-byte (bf16) loads in flight per thread.  Rows whose length is not a
// multiple of 8 take element-wise accesses.
#include <cuda_runtime.h>

#include "msc_common.cuh"
#include "msc_internal.h"

namespace {

struct ConvParams {
    const void* x;
    const float* w;
    const float* bias;
    void* out;
    float* state;
    int64_t rows, dim, L, nchunks;
    int K;
    int silu;
};

__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float finish(float acc, int silu) { return silu ? msc::silu_f(acc) : acc; }

template <bool kOutBF16>
__device__ __forceinline__ void store1(void* out, int64_t i, float v) {
    if constexpr (kOutBF16) {
        const uint32_t w = pack_bf16x2_rn(v, 0.f);
        reinterpret_cast<uint16_t*>(out)[i] = (uint16_t)(w & 0xFFFFu);
    } else {
        reinterpret_cast<float*>(out)[i] = v;
    }
}

// One thread makes 16 consecutive outputs.  kVec: L % 8 == 0, so every 8-step
// chunk is 16-byte aligned in x and out; a thread whose 16 steps run past the
// row end (or any thread when L % 8 != 0) takes element-wise accesses.
template <bool kInBF16, bool kOutBF16, bool kVec>
__global__ void __launch_bounds__(256) conv1d_fwd_kernel(const ConvParams p) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= p.rows * p.nchunks) return;
    const int64_t row = idx / p.nchunks;
    const int64_t c = idx - row * p.nchunks;
    const int64_t d = row % p.dim;
    const int64_t t0 = 16 * c;
    const int K = p.K;
    const bool vec = kVec && t0 + 16 <= p.L;

    // xv[0..8): the 8 steps before (halo), xv[8..24): this thread's 16 steps
    float xv[24];
    if (vec) {
        msc::ld8<kInBF16>(p.x, row * p.L + t0, xv + 8);
        msc::ld8<kInBF16>(p.x, row * p.L + t0 + 8, xv + 16);
        if (c > 0) {
            msc::ld8<kInBF16>(p.x, row * p.L + t0 - 8, xv);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) xv[i] = 0.f;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 24; ++i) {
            const int64_t t = t0 - 8 + i;
            xv[i] = (t >= 0 && t < p.L) ? msc::ld_elem<kInBF16>(p.x, row * p.L + t) : 0.f;
        }
    }
    // weights right-aligned in an 8-tap window: ws[m] = w[m - (8 - K)], zero
    // before; output t0 + i = sum_m ws[m] x[t0 + i - 7 + m] = sum_m ws[m] xv[i + 1 + m]
    float ws[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) ws[m] = (m + K >= 8) ? __ldg(p.w + d * K + (m + K - 8)) : 0.f;
    const float b0 = p.bias ? __ldg(p.bias + d) : 0.f;

    float o[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float acc = b0;
#pragma unroll
        for (int m = 0; m < 8; ++m) acc = fmaf(ws[m], xv[i + 1 + m], acc);
        o[i] = finish(acc, p.silu);
    }
    if (vec) {
        if constexpr (kOutBF16) {
            uint4* q = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.out) + row * p.L + t0);
            q[0] = make_uint4(pack_bf16x2_rn(o[0], o[1]), pack_bf16x2_rn(o[2], o[3]), pack_bf16x2_rn(o[4], o[5]),
                              pack_bf16x2_rn(o[6], o[7]));
            q[1] = make_uint4(pack_bf16x2_rn(o[8], o[9]), pack_bf16x2_rn(o[10], o[11]),
                              pack_bf16x2_rn(o[12], o[13]), pack_bf16x2_rn(o[14], o[15]));
        } else {
            float4* q = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + row * p.L + t0);
#pragma unroll
            for (int e = 0; e < 4; ++e) q[e] = make_float4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            if (t0 + i < p.L) store1<kOutBF16>(p.out, row * p.L + t0 + i, o[i]);
    }
}

// One thread per row: state holds the previous K - 1 inputs, oldest first.
template <bool kInBF16, bool kOutBF16>
__global__ void __launch_bounds__(256) conv1d_update_kernel(const ConvParams p) {
    const int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (row >= p.rows) return;
    const int64_t d = row % p.dim;
    const int K = p.K;
    float s[8];
    float* st = p.state + row * (K - 1);
#pragma unroll
    for (int k = 0; k < 7; ++k) s[k] = k < K - 1 ? st[k] : 0.f;
    const float xn = msc::ld_elem<kInBF16>(p.x, row);
    float acc = p.bias ? __ldg(p.bias + d) : 0.f;
#pragma unroll
    for (int k = 0; k < 7; ++k)
        if (k < K - 1) acc = fmaf(__ldg(p.w + d * K + k), s[k], acc);
    acc = fmaf(__ldg(p.w + d * K + K - 1), xn, acc);
    store1<kOutBF16>(p.out, row, finish(acc, p.silu));
#pragma unroll
    for (int k = 0; k < 7; ++k) {
        if (k < K - 2) st[k] = s[k + 1];
        else if (k == K - 2) st[k] = xn;
    }
}

template <bool kIn, bool kOut>
msc_status launch_fwd(const ConvParams& p, bool vec, cudaStream_t st) {
    const int64_t n = p.rows * p.nchunks;
    const int64_t blocks = (n + 255) / 256;
    if (blocks > 0x7FFFFFFF) return msc_host::fail(MSC_ERR_UNSUPPORTED, "problem too large for one launch");
    if (vec)
        conv1d_fwd_kernel<kIn, kOut, true><<<(unsigned)blocks, 256, 0, st>>>(p);
    else
        conv1d_fwd_kernel<kIn, kOut, false><<<(unsigned)blocks, 256, 0, st>>>(p);
    return msc_host::check_launch("conv1d_fwd");
}

template <bool kIn, bool kOut>
msc_status launch_update(const ConvParams& p, cudaStream_t st) {
    const int64_t blocks = (p.rows + 255) / 256;
    if (blocks > 0x7FFFFFFF) return msc_host::fail(MSC_ERR_UNSUPPORTED, "problem too large for one launch");
    conv1d_update_kernel<kIn, kOut><<<(unsigned)blocks, 256, 0, st>>>(p);
    return msc_host::check_launch("conv1d_update");
}

}  // namespace

namespace msc_host {

msc_status conv1d_fwd_launch(const Conv1dArgs& a, cudaStream_t st) {
    ConvParams p{};
    p.x = a.x; p.w = a.weight; p.bias = a.bias; p.out = a.out;
    p.rows = a.batch * a.dim; p.dim = a.dim; p.L = a.L; p.nchunks = (a.L + 15) / 16;
    p.K = a.K; p.silu = a.silu;
    const bool vec = (a.L % 8) == 0;
    if (a.in_bf16)
        return a.out_bf16 ? launch_fwd<true, true>(p, vec, st) : launch_fwd<true, false>(p, vec, st);
    return a.out_bf16 ? launch_fwd<false, true>(p, vec, st) : launch_fwd<false, false>(p, vec, st);
}

msc_status conv1d_update_launch(const Conv1dArgs& a, cudaStream_t st) {
    ConvParams p{};
    p.x = a.x; p.w = a.weight; p.bias = a.bias; p.out = a.out; p.state = a.state;
    p.rows = a.batch * a.dim; p.dim = a.dim; p.L = 1; p.nchunks = 1;
    p.K = a.K; p.silu = a.silu;
    if (a.in_bf16) return a.out_bf16 ? launch_update<true, true>(p, st) : launch_update<true, false>(p, st);
    return a.out_bf16 ? launch_update<false, true>(p, st) : launch_update<false, false>(p, st);
}

}  // namespace msc_host
