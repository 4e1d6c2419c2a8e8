// conv1d.cu -- causal depthwise conv1d + SiLU front end of the Mamba block on sm_103a.
//
// What it computes (bqwf survey sec. 3.1: each Mamba block runs a causal 1-D
// convolution for local context before the selective SSM):
//   out[b, d, t] = silu(bias[d] + sum_{k < K} w[d, k] x[b, d, t - (K - 1) + k]),  x = 0 before t = 0
// its decode step, which keeps the last K - 1 inputs of every row (study
// note "Mamba — 选择性状态空间模型", 踩过的坑: the convolution still keeps the
// last few inputs when there is no attention cache), and its backward.
//
// Design.  Both are bound by HBM: per element the sequence kernel reads x once
// (2 or 4 bytes) and writes out once; the K <= 8 weights of a channel and its
// bias are read through L1.  For K <= 4 (Mamba's width) and L % 8 == 0 the
// forward and backward are persistent kernels whose warps walk 512-step units
// of a row, lane l taking 16 consecutive steps: halos and look-ahead pass
// between neighbouring lanes by shuffle, one lane per warp prefetches the unit
// two ahead into L2 with a bulk request, and the taps run on packed f32x2
// arithmetic.  Other widths and lengths take one thread per 16 consecutive
// outputs: it loads its own two 8-step chunks and the chunk before them (the
// K - 1 halo inputs; the neighbouring thread loads the same chunk, so that
// load hits L1), with element-wise accesses where L is not a multiple of 8.
#include <cuda_runtime.h>

#include "msc_common.cuh"
#include "msc_tma.cuh"
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

// silu'(x) = s (1 + x (1 - s)), s = sigmoid(x)
__device__ __forceinline__ float dsilu_f(float x) {
    const float sg = msc::sigmoid_f(x);
    return sg * (1.f + x * (1.f - sg));
}
__device__ __forceinline__ uint64_t dsilu_2(uint64_t x) {
    float x0, x1;
    msc::upk2(x, x0, x1);
    const uint64_t e = msc::ex2_2(msc::pk2(-x0 * MSC_LOG2E, -x1 * MSC_LOG2E));
    const uint64_t sg = msc::rcp_2(msc::add2(e, msc::pk2(1.f, 1.f)));
    const uint64_t one_m = msc::fma2(sg, msc::pk2(-1.f, -1.f), msc::pk2(1.f, 1.f));
    return msc::mul2(sg, msc::fma2(x, one_m, msc::pk2(1.f, 1.f)));
}

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

// K <= 4 (the width Mamba uses) and L % 8 == 0: a persistent kernel whose
// warps walk units of one row's 512 consecutive steps, lane l taking steps
// 16 l .. 16 l + 15 of the unit.  The three inputs before a lane's first step
// are the last three of the lane before it (a shuffle); a unit's first lane
// loads them.  The first lane also prefetches, into L2 with one bulk request,
// the unit the warp takes two sweeps later, so DRAM reads run ahead of the
// loads without holding registers.  Taps are right-aligned in a 4-tap window;
// output pairs use packed f32x2 arithmetic.
constexpr int kUnitSteps = 512;
constexpr int kPrefetchAhead = 2;  // units (sweeps of the grid) prefetched ahead

// Position of a unit: row, 512-step segment, channel.
struct UnitPos {
    int64_t row, d;
    int seg;
};

__device__ __forceinline__ void advance(UnitPos& q, int64_t sq, int sr, int64_t sqd, int nseg, int64_t dim) {
    q.row += sq;
    q.d += sqd;
    q.seg += sr;
    if (q.seg >= nseg) { q.seg -= nseg; ++q.row; ++q.d; }
    if (q.d >= dim) q.d -= dim;
}

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// One unit's inputs (512 steps, or the row's rest) into L2.
template <int kES>
__device__ __forceinline__ void prefetch_unit(const void* x, const UnitPos& q, int64_t L) {
    const int64_t s0 = (int64_t)q.seg * kUnitSteps;
    const int64_t n = L - s0 < kUnitSteps ? L - s0 : kUnitSteps;
    prefetch_l2(reinterpret_cast<const uint8_t*>(x) + (q.row * L + s0) * kES, (uint32_t)(n * kES));
}

template <bool kInBF16, bool kOutBF16>
__global__ void __launch_bounds__(256) conv1d_fwd_w4_kernel(const ConvParams p, int64_t units, int nseg) {
    constexpr int kES = kInBF16 ? 2 : 4;
    const int lane = threadIdx.x & 31;
    const int64_t wstep = (int64_t)gridDim.x * (blockDim.x >> 5);  // units per sweep of the grid
    int64_t u = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (u >= units) return;  // warp-uniform
    const int64_t sq = wstep / nseg;
    const int sr = (int)(wstep - sq * nseg);
    const int64_t sqd = sq % p.dim;
    UnitPos cur;
    cur.row = u / nseg;
    cur.seg = (int)(u - cur.row * nseg);
    cur.d = cur.row % p.dim;
    // the unit prefetched next: kPrefetchAhead sweeps ahead of the current one
    UnitPos pf = cur;
    int64_t upf = u;
    for (int k = 0; k <= kPrefetchAhead; ++k) {
        if (k > 0) { advance(pf, sq, sr, sqd, nseg, p.dim); upf += wstep; }
        if (lane == 0 && upf < units) prefetch_unit<kES>(p.x, pf, p.L);
    }

    for (; u < units; u += wstep, advance(cur, sq, sr, sqd, nseg, p.dim)) {
        advance(pf, sq, sr, sqd, nseg, p.dim);
        upf += wstep;
        if (lane == 0 && upf < units) prefetch_unit<kES>(p.x, pf, p.L);

        const int64_t t0 = (int64_t)cur.seg * kUnitSteps + 16 * lane;
        const int nv = t0 >= p.L ? 0 : (p.L - t0 >= 16 ? 16 : (int)(p.L - t0));
        const int64_t base = cur.row * p.L + t0;
        // xs[0..3) = x[t0 - 3 .. t0), xs[3..19) = x[t0 .. t0 + 16)
        float xs[19];
        if constexpr (kInBF16) {
            const uint4* q = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p.x) + base);
            const uint4 a = nv > 0 ? __ldg(q) : make_uint4(0u, 0u, 0u, 0u);
            const uint4 b = nv > 8 ? __ldg(q + 1) : make_uint4(0u, 0u, 0u, 0u);
            // x[t0 - 4 .. t0) as two bf16 pairs (8-byte aligned: t0 is a multiple of 16)
            const uint2 hv = (lane == 0 && t0 > 0)
                                 ? __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(p.x) + base - 4))
                                 : make_uint2(0u, 0u);
            const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                xs[3 + 2 * k] = msc::bf16lo(w[k]);
                xs[4 + 2 * k] = msc::bf16hi(w[k]);
            }
            const uint32_t s6 = __shfl_up_sync(0xffffffffu, w[6], 1);
            const uint32_t s7 = __shfl_up_sync(0xffffffffu, w[7], 1);
            const uint32_t h0 = lane == 0 ? hv.x : s6, h1 = lane == 0 ? hv.y : s7;
            xs[0] = msc::bf16hi(h0);
            xs[1] = msc::bf16lo(h1);
            xs[2] = msc::bf16hi(h1);
        } else {
            const float4* q = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p.x) + base);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 v = nv > 4 * e ? __ldg(q + e) : make_float4(0.f, 0.f, 0.f, 0.f);
                xs[3 + 4 * e] = v.x; xs[4 + 4 * e] = v.y; xs[5 + 4 * e] = v.z; xs[6 + 4 * e] = v.w;
            }
            // x[t0 - 4 .. t0) (16-byte aligned); the last three are the halo
            const float4 hv = (lane == 0 && t0 > 0) ? __ldg(q - 1) : make_float4(0.f, 0.f, 0.f, 0.f);
            const float hl[3] = {hv.y, hv.z, hv.w};
#pragma unroll
            for (int m = 0; m < 3; ++m) {
                const float s = __shfl_up_sync(0xffffffffu, xs[16 + m], 1);
                xs[m] = lane == 0 ? hl[m] : s;
            }
        }
        if (t0 == 0) xs[0] = xs[1] = xs[2] = 0.f;
        uint64_t w2[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float w = (m + p.K >= 4) ? __ldg(p.w + cur.d * p.K + (m + p.K - 4)) : 0.f;
            w2[m] = msc::pk2(w, w);
        }
        const float bv = p.bias ? __ldg(p.bias + cur.d) : 0.f;
        const uint64_t b2 = msc::pk2(bv, bv);
        // output t0 + i = sum_m w4[m] x[t0 + i - 3 + m] = sum_m w4[m] xs[i + m]
        uint32_t ob[8];
        uint64_t of[8];
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
            uint64_t acc = b2;
#pragma unroll
            for (int m = 0; m < 4; ++m) acc = msc::fma2(w2[m], msc::pk2(xs[i + m], xs[i + 1 + m]), acc);
            if (p.silu) acc = msc::silu_2(acc);
            float lo, hi;
            msc::upk2(acc, lo, hi);
            if constexpr (kOutBF16) ob[i / 2] = pack_bf16x2_rn(lo, hi);
            else of[i / 2] = acc;
        }
        if (nv > 0) {
            if constexpr (kOutBF16) {
                uint4* q = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.out) + base);
                q[0] = make_uint4(ob[0], ob[1], ob[2], ob[3]);
                if (nv > 8) q[1] = make_uint4(ob[4], ob[5], ob[6], ob[7]);
            } else {
                ulonglong2* q = reinterpret_cast<ulonglong2*>(reinterpret_cast<float*>(p.out) + base);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (nv > 4 * e) q[e] = make_ulonglong2(of[2 * e], of[2 * e + 1]);
            }
        }
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

// Backward, one thread per 16 consecutive steps of a row (the forward's tiling):
// with pre the pre-activation and g = dout silu'(pre) (dout without the
// activation), dx[s] = sum_k w[k] g[s + K - 1 - k], dw[k] += sum_t g[t] x[t - K + 1 + k],
// db += sum_t g[t].  The thread recomputes pre over its 16 steps and the 8 after
// (an 8-step halo of x before them), so it needs x of steps t0 - 8 .. t0 + 24
// and dout of t0 .. t0 + 24.  dw and db: a butterfly over the warp when all 32
// lanes hold chunks of one row, else per-thread atomics.
// kW: the tap window (4 when K <= 4, as in Mamba, else 8), weights right-aligned.
template <bool kInBF16, bool kVec, int kW>
__global__ void __launch_bounds__(256) conv1d_bwd_kernel(const ConvParams p, const float* dout, float* dx,
                                                         float* dw, float* db) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const bool live = idx < p.rows * p.nchunks;
    const int64_t row = live ? idx / p.nchunks : 0;
    const int64_t c = live ? idx - row * p.nchunks : 0;
    const int64_t d = row % p.dim;
    const int64_t t0 = 16 * c;
    const int K = p.K;
    const int lane = threadIdx.x & 31;
    // xv[i] = x[t0 - 8 + i] (i < 32), gv[i] = dout[t0 + i] (i < 24), 0 outside [0, L)
    float xv[32], gv[24];
    const bool vec = kVec && live && t0 + 24 <= p.L;
    if (vec) {
        if (c > 0) msc::ld8<kInBF16>(p.x, row * p.L + t0 - 8, xv);
        else {
#pragma unroll
            for (int i = 0; i < 8; ++i) xv[i] = 0.f;
        }
#pragma unroll
        for (int q = 0; q < 3; ++q) {
            msc::ld8<kInBF16>(p.x, row * p.L + t0 + 8 * q, xv + 8 + 8 * q);
            msc::ld8<false>(dout, row * p.L + t0 + 8 * q, gv + 8 * q);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int64_t t = t0 - 8 + i;
            xv[i] = (live && t >= 0 && t < p.L) ? msc::ld_elem<kInBF16>(p.x, row * p.L + t) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < 24; ++i) {
            const int64_t t = t0 + i;
            gv[i] = (live && t < p.L) ? dout[row * p.L + t] : 0.f;
        }
    }
    float ws[kW];
#pragma unroll
    for (int m = 0; m < kW; ++m) ws[m] = (live && m + K >= kW) ? __ldg(p.w + d * K + (m + K - kW)) : 0.f;
    const float b0 = (live && p.bias) ? __ldg(p.bias + d) : 0.f;
    // g over steps t0 .. t0 + 15 + kW - 1
    // (pre[t0 + i] = sum_m ws[m] x[t0 + i - kW + 1 + m] = sum_m ws[m] xv[i + 9 - kW + m])
    constexpr int kG = 16 + kW - 1;
    if (p.silu) {
#pragma unroll
        for (int i = 0; i < kG; ++i) {
            float pre = b0;
#pragma unroll
            for (int m = 0; m < kW; ++m) pre = fmaf(ws[m], xv[i + 9 - kW + m], pre);
            const float sg = msc::sigmoid_f(pre);
            gv[i] *= sg * (1.f + pre * (1.f - sg));
        }
    }
    // dx[t0 + s] = sum_m ws[m] g[t0 + s + kW - 1 - m]
    if (live) {
        float o[16];
#pragma unroll
        for (int s2 = 0; s2 < 16; ++s2) {
            float acc = 0.f;
#pragma unroll
            for (int m = 0; m < kW; ++m) acc = fmaf(ws[m], gv[s2 + kW - 1 - m], acc);
            o[s2] = acc;
        }
        if (kVec && t0 + 16 <= p.L) {
            float4* q = reinterpret_cast<float4*>(dx + row * p.L + t0);
#pragma unroll
            for (int e = 0; e < 4; ++e) q[e] = make_float4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
        } else {
#pragma unroll
            for (int s2 = 0; s2 < 16; ++s2)
                if (t0 + s2 < p.L) dx[row * p.L + t0 + s2] = o[s2];
        }
    }
    // partial dw (tap m of the window) and db over this thread's own steps
    float part[kW + 1];
#pragma unroll
    for (int m = 0; m <= kW; ++m) part[m] = 0.f;
#pragma unroll
    for (int s2 = 0; s2 < 16; ++s2) {
        const float gg = (t0 + s2 < p.L) ? gv[s2] : 0.f;
#pragma unroll
        for (int m = 0; m < kW; ++m) part[m] = fmaf(gg, xv[s2 + 9 - kW + m], part[m]);
        part[kW] += gg;
    }
    const int64_t row0 = __shfl_sync(0xffffffffu, row, 0);
    const bool one_row = __all_sync(0xffffffffu, live && row == row0);
    if (one_row) {
#pragma unroll
        for (int m = 0; m <= kW; ++m)
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) part[m] += __shfl_xor_sync(0xffffffffu, part[m], off);
        if (lane != 0) return;
    } else if (!live) {
        return;
    }
#pragma unroll
    for (int m = 0; m < kW; ++m)
        if (m + K >= kW) atomicAdd(dw + d * K + (m + K - kW), part[m]);
    if (db) atomicAdd(db + d, part[kW]);
}

// Backward for K <= 4 and L % 8 == 0.  A warp takes whole rows, one 512-step
// segment after another, lane l taking steps 16 l .. 16 l + 15 of a segment
// (the forward's tiling).  With pre the pre-activation and g = dout silu'(pre)
// (dout without the activation):
//   dx[s] = sum_m w4[m] g[s + 3 - m],  dw4[m] += sum_t g[t] x[t - 3 + m],  db += sum_t g[t]
// (w4: the taps right-aligned in a 4-tap window).  A lane's three inputs before
// its first step come from the lane before it, the three g after its last step
// from the lane after it (shuffles); the segment's first lane loads its halo, the
// last lane loads the three inputs and output gradients after the segment and
// forms their g itself.  dw and db accumulate in registers over the row and are
// reduced over the warp once per row.  Lane 0 prefetches into L2, with bulk
// requests, the segment the warp takes two segments later (x and dout).
// Issues the L2 prefetch of segment (pf_row, pf_seg) of x and dout (lane 0) and
// moves the cursor to the warp's next segment.
template <int kES>
__device__ __forceinline__ void bwd_prefetch(const void* x, const float* dout, int64_t rows, int64_t L, int nseg,
                                             int64_t nwarps, int lane, int64_t& pf_row, int& pf_seg) {
    if (lane == 0 && pf_row < rows) {
        const int64_t s0 = (int64_t)pf_seg * kUnitSteps;
        const int64_t n = L - s0 < kUnitSteps ? L - s0 : kUnitSteps;
        prefetch_l2(reinterpret_cast<const uint8_t*>(x) + (pf_row * L + s0) * kES, (uint32_t)(n * kES));
        prefetch_l2(dout + pf_row * L + s0, (uint32_t)(n * 4));
    }
    if (++pf_seg == nseg) {
        pf_seg = 0;
        pf_row += nwarps;
    }
}

template <bool kInBF16>
__global__ void __launch_bounds__(256) conv1d_bwd_w4_kernel(const ConvParams p, const float* __restrict__ dout,
                                                            float* __restrict__ dx, float* dw, float* db, int nseg) {
    constexpr int kES = kInBF16 ? 2 : 4;
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= p.rows) return;  // warp-uniform
    const int64_t L = p.L;
    // prefetch cursor, two segments ahead of the one being computed
    int64_t pf_row = row;
    int pf_seg = 0;
    bwd_prefetch<kES>(p.x, dout, p.rows, L, nseg, nwarps, lane, pf_row, pf_seg);
    bwd_prefetch<kES>(p.x, dout, p.rows, L, nseg, nwarps, lane, pf_row, pf_seg);

    for (; row < p.rows; row += nwarps) {
        const int64_t d = row % p.dim;
        float ws[4];
        uint64_t w2[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            ws[m] = (m + p.K >= 4) ? __ldg(p.w + d * p.K + (m + p.K - 4)) : 0.f;
            w2[m] = msc::pk2(ws[m], ws[m]);
        }
        const float bv = p.bias ? __ldg(p.bias + d) : 0.f;
        const uint64_t b2 = msc::pk2(bv, bv);
        uint64_t dw2[4] = {0ull, 0ull, 0ull, 0ull};
        uint64_t db2 = 0ull;
        for (int seg = 0; seg < nseg; ++seg) {
            bwd_prefetch<kES>(p.x, dout, p.rows, L, nseg, nwarps, lane, pf_row, pf_seg);
            const int64_t t0 = (int64_t)seg * kUnitSteps + 16 * lane;
            const int nv = t0 >= L ? 0 : (L - t0 >= 16 ? 16 : (int)(L - t0));
            const int64_t base = row * L + t0;
            // xs[0..3) = x[t0 - 3 .. t0), xs[3..19) = x[t0 .. t0 + 16), xs[19..22) = x[t0 + 16 .. t0 + 19)
            float xs[22];
            float gv[16];
            // x after the lane's steps, and dout there (the last lane of the segment)
            const bool tail = lane == 31 && t0 + 16 < L;
            float xt[3] = {0.f, 0.f, 0.f}, gt[3] = {0.f, 0.f, 0.f};
            if constexpr (kInBF16) {
                const uint4* q = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p.x) + base);
                const uint4 a = nv > 0 ? __ldg(q) : make_uint4(0u, 0u, 0u, 0u);
                const uint4 b = nv > 8 ? __ldg(q + 1) : make_uint4(0u, 0u, 0u, 0u);
                const uint2 hv = (lane == 0 && t0 > 0)
                                     ? __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(p.x) + base - 4))
                                     : make_uint2(0u, 0u);
                const uint2 tv = tail ? __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(p.x) + base + 16))
                                      : make_uint2(0u, 0u);
                const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    xs[3 + 2 * k] = msc::bf16lo(w[k]);
                    xs[4 + 2 * k] = msc::bf16hi(w[k]);
                }
                const uint32_t s6 = __shfl_up_sync(0xffffffffu, w[6], 1);
                const uint32_t s7 = __shfl_up_sync(0xffffffffu, w[7], 1);
                const uint32_t h0 = lane == 0 ? hv.x : s6, h1 = lane == 0 ? hv.y : s7;
                xs[0] = msc::bf16hi(h0);
                xs[1] = msc::bf16lo(h1);
                xs[2] = msc::bf16hi(h1);
                xt[0] = msc::bf16lo(tv.x);
                xt[1] = msc::bf16hi(tv.x);
                xt[2] = msc::bf16lo(tv.y);
            } else {
                const float4* q = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p.x) + base);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float4 v = nv > 4 * e ? __ldg(q + e) : make_float4(0.f, 0.f, 0.f, 0.f);
                    xs[3 + 4 * e] = v.x; xs[4 + 4 * e] = v.y; xs[5 + 4 * e] = v.z; xs[6 + 4 * e] = v.w;
                }
                const float4 hv = (lane == 0 && t0 > 0) ? __ldg(q - 1) : make_float4(0.f, 0.f, 0.f, 0.f);
                const float4 tv = tail ? __ldg(q + 4) : make_float4(0.f, 0.f, 0.f, 0.f);
                const float hl[3] = {hv.y, hv.z, hv.w};
#pragma unroll
                for (int m = 0; m < 3; ++m) {
                    const float sv = __shfl_up_sync(0xffffffffu, xs[16 + m], 1);
                    xs[m] = lane == 0 ? hl[m] : sv;
                }
                xt[0] = tv.x; xt[1] = tv.y; xt[2] = tv.z;
            }
            if (t0 == 0) xs[0] = xs[1] = xs[2] = 0.f;
            {
                const float4* q = reinterpret_cast<const float4*>(dout + base);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float4 v = nv > 4 * e ? __ldg(q + e) : make_float4(0.f, 0.f, 0.f, 0.f);
                    gv[4 * e] = v.x; gv[4 * e + 1] = v.y; gv[4 * e + 2] = v.z; gv[4 * e + 3] = v.w;
                }
                const float4 tg = tail ? __ldg(q + 4) : make_float4(0.f, 0.f, 0.f, 0.f);
                gt[0] = tg.x; gt[1] = tg.y; gt[2] = tg.z;
            }
            // the inputs after the lane's steps (used by the last lane only)
            xs[19] = xt[0]; xs[20] = xt[1]; xs[21] = xt[2];
            // g over the lane's 16 steps (pairs), and over the three after it on the last lane
            // (pre[t0 + i] = sum_m w4[m] xs[i + m])
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
                uint64_t pre = b2;
#pragma unroll
                for (int m = 0; m < 4; ++m) pre = msc::fma2(w2[m], msc::pk2(xs[i + m], xs[i + 1 + m]), pre);
                uint64_t g = msc::pk2(gv[i], gv[i + 1]);
                if (p.silu) g = msc::mul2(g, dsilu_2(pre));
                msc::upk2(g, gv[i], gv[i + 1]);
            }
            float ga[3];
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                float pre = bv;
#pragma unroll
                for (int m = 0; m < 4; ++m) pre = fmaf(ws[m], xs[16 + j + m], pre);
                const float gl = p.silu ? gt[j] * dsilu_f(pre) : gt[j];
                const float sv = __shfl_down_sync(0xffffffffu, gv[j], 1);
                ga[j] = lane == 31 ? gl : sv;
            }
            // past the row end g is 0 (dout there is not read)
            if (nv < 16) {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    if (i >= nv) gv[i] = 0.f;
            }
            if (t0 + 16 >= L) ga[0] = ga[1] = ga[2] = 0.f;
            // dx[t0 + s] = sum_m w4[m] g[t0 + s + 3 - m]; g index k = s + 3 - m in 0 .. 18
            float gg[19];
#pragma unroll
            for (int i = 0; i < 16; ++i) gg[i] = gv[i];
            gg[16] = ga[0]; gg[17] = ga[1]; gg[18] = ga[2];
            uint64_t o[8];
#pragma unroll
            for (int s2 = 0; s2 < 16; s2 += 2) {
                uint64_t acc = 0ull;
#pragma unroll
                for (int m = 0; m < 4; ++m) acc = msc::fma2(w2[m], msc::pk2(gg[s2 + 3 - m], gg[s2 + 4 - m]), acc);
                o[s2 / 2] = acc;
            }
            if (nv > 0) {
                ulonglong2* q = reinterpret_cast<ulonglong2*>(dx + base);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (nv > 4 * e) q[e] = make_ulonglong2(o[2 * e], o[2 * e + 1]);
            }
            // dw4[m] += g[t0 + s] x[t0 + s - 3 + m] = gv[s] xs[s + m]; db += g
#pragma unroll
            for (int s2 = 0; s2 < 16; s2 += 2) {
                const uint64_t g2 = msc::pk2(gv[s2], gv[s2 + 1]);
#pragma unroll
                for (int m = 0; m < 4; ++m) dw2[m] = msc::fma2(g2, msc::pk2(xs[s2 + m], xs[s2 + 1 + m]), dw2[m]);
                db2 = msc::add2(db2, g2);
            }
        }
        // the row's dw and db: sum the pair halves, then over the warp
        float part[5];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            float lo, hi;
            msc::upk2(dw2[m], lo, hi);
            part[m] = lo + hi;
        }
        {
            float lo, hi;
            msc::upk2(db2, lo, hi);
            part[4] = lo + hi;
        }
#pragma unroll
        for (int m = 0; m < 5; ++m)
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) part[m] += __shfl_xor_sync(0xffffffffu, part[m], off);
        if (lane == 0) {
#pragma unroll
            for (int m = 0; m < 4; ++m)
                if (m + p.K >= 4) atomicAdd(dw + d * p.K + (m + p.K - 4), part[m]);
            if (db) atomicAdd(db + d, part[4]);
        }
    }
}

template <bool kIn>
msc_status launch_bwd(const ConvParams& p, bool vec, const float* dout, float* dx, float* dw, float* db,
                      cudaStream_t st) {
    if (vec && p.K <= 4) {
        if (p.rows == 0) return MSC_OK;
        const int nseg = (int)((p.L + kUnitSteps - 1) / kUnitSteps);
        static std::atomic<int> per_sm[64];  // resident CTAs per SM, once per device (0: not yet)
        int dev = 0;
        cudaGetDevice(&dev);
        std::atomic<int>& occ = per_sm[dev & 63];
        if (occ.load() == 0) {
            int n = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, conv1d_bwd_w4_kernel<kIn>, 256, 0) != cudaSuccess ||
                n < 1)
                n = 1;
            occ.store(n);
        }
        const int64_t want = (p.rows + 7) / 8;
        const int64_t cap = (int64_t)msc_host::num_sms() * occ.load();
        const unsigned blocks = (unsigned)(want < cap ? want : cap);
        conv1d_bwd_w4_kernel<kIn><<<blocks, 256, 0, st>>>(p, dout, dx, dw, db, nseg);
        return msc_host::check_launch("conv1d_bwd");
    }
    const int64_t n = p.rows * p.nchunks;
    const int64_t blocks = (n + 255) / 256;
    if (blocks > 0x7FFFFFFF) return msc_host::fail(MSC_ERR_UNSUPPORTED, "problem too large for one launch");
    if (p.K <= 4) {
        if (vec)
            conv1d_bwd_kernel<kIn, true, 4><<<(unsigned)blocks, 256, 0, st>>>(p, dout, dx, dw, db);
        else
            conv1d_bwd_kernel<kIn, false, 4><<<(unsigned)blocks, 256, 0, st>>>(p, dout, dx, dw, db);
    } else {
        if (vec)
            conv1d_bwd_kernel<kIn, true, 8><<<(unsigned)blocks, 256, 0, st>>>(p, dout, dx, dw, db);
        else
            conv1d_bwd_kernel<kIn, false, 8><<<(unsigned)blocks, 256, 0, st>>>(p, dout, dx, dw, db);
    }
    return msc_host::check_launch("conv1d_bwd");
}

template <bool kIn, bool kOut>
msc_status launch_fwd(const ConvParams& p, bool vec, cudaStream_t st) {
    if (vec && p.K <= 4) {
        const int nseg = (int)((p.L + kUnitSteps - 1) / kUnitSteps);
        const int64_t units = p.rows * nseg;
        if (units == 0) return MSC_OK;
        static std::atomic<int> per_sm[64];  // resident CTAs per SM, once per device (0: not yet)
        int dev = 0;
        cudaGetDevice(&dev);
        std::atomic<int>& occ = per_sm[dev & 63];
        if (occ.load() == 0) {
            int n = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, conv1d_fwd_w4_kernel<kIn, kOut>, 256, 0) !=
                    cudaSuccess || n < 1)
                n = 1;
            occ.store(n);
        }
        const int64_t want = (units + 7) / 8;
        const int64_t cap = (int64_t)msc_host::num_sms() * occ.load();
        const unsigned blocks = (unsigned)(want < cap ? want : cap);
        conv1d_fwd_w4_kernel<kIn, kOut><<<blocks, 256, 0, st>>>(p, units, nseg);
        return msc_host::check_launch("conv1d_fwd");
    }
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

msc_status conv1d_bwd_launch(const Conv1dArgs& a, const float* dout, float* dx, float* dweight, float* dbias,
                             cudaStream_t st) {
    ConvParams p{};
    p.x = a.x; p.w = a.weight; p.bias = a.bias;
    p.rows = a.batch * a.dim; p.dim = a.dim; p.L = a.L; p.nchunks = (a.L + 15) / 16;
    p.K = a.K; p.silu = a.silu;
    cudaError_t e = cudaMemsetAsync(dweight, 0, (size_t)a.dim * a.K * sizeof(float), st);
    if (e == cudaSuccess && dbias) e = cudaMemsetAsync(dbias, 0, (size_t)a.dim * sizeof(float), st);
    if (e != cudaSuccess) return fail(MSC_ERR_CUDA, "conv1d bwd memset: %s", cudaGetErrorString(e));
    const bool vec = (a.L % 8) == 0;
    return a.in_bf16 ? launch_bwd<true>(p, vec, dout, dx, dweight, dbias, st)
                     : launch_bwd<false>(p, vec, dout, dx, dweight, dbias, st);
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
