// ssd_fwd.cu -- Mamba-2 SSD (scalar-A, multi-head) chunked forward on sm_103a.
//
// What it computes, per batch entry b and head h (bqwf survey sec. 3.2: scalar
// A_t = alpha_t I makes the SSM a masked linear attention; "Mamba 解密" sec. 6.2:
// Y = M (X . B^T) C with M_ij = a_{j+1} ... a_i for i >= j):
//   Delta_t = softplus(delta_t + bias_h),  a_t = exp(Delta_t A_h)
//   y_t = sum_{s <= t} (a_{s+1} ... a_t) (C_t . B_s) Delta_s x_s  (+ D_h x_t) (* silu z_t)
// By the block decomposition, with chunks of Q steps and cs_i the in-chunk
// inclusive cumulative sum of Delta A (so a_{j+1}...a_i = exp(cs_i - cs_j)):
//   Y_diag[i, p] = sum_{j <= i} exp(cs_i - cs_j) (C_i . B_j) Delta_j x_j[p]      (tensor cores)
//   Y_off[i, p]  = exp(cs_i) sum_n C_i[n] Hin[p, n]                             (tensor cores)
//   S_c[p, n]    = sum_j exp(cs_last - cs_j) Delta_j x_j[p] B_j[n]              (tensor cores)
//   Hin_{c+1}    = exp(cs_last(c)) Hin_c + S_c                                  (CUDA cores)
// Four launches: (1) ssd_prep_kernel: Delta and cs; (2) ssd_state_kernel: S_c
// on tcgen05 with the TMA tiles of B and x as MN-major operands; (3)
// ssd_pass_kernel: Hin of every chunk and the final state; (4)
// ssd_scan_kernel: G = C B^T once per (chunk, row block, head block) into
// tensor memory, then per head the masked decay matrix (L . G scaled by Delta)
// is written to shared memory by CUDA cores, a 64-column quarter at a time
// while the tensor cores consume the previous quarter, and Y_diag, Y_off
// accumulate in tensor memory, read back by tcgen05.ld for the epilogue.
//
// Precision: C, B and x enter the tensor cores as the bf16 values they are, so
// G is exact up to fp32 accumulation.  Every operand the CUDA cores form in
// fp32 -- the intra-chunk M'[i, j] = G[i, j] exp(cs_i - cs_j) Delta_j, the
// weighted x of the chunk states and the carried state Hin -- is split into two
// bf16 terms (hi + lo, 16 significant bits) and both terms are multiplied on
// the tensor cores; every product accumulates in fp32.  A single bf16 rounding
// of those operands is not enough: Y_diag and Y_off can be large and cancel at
// chunk boundaries.
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstdlib>

#include "msc_common.cuh"
#include "msc_internal.h"
#include "msc_tc.cuh"
#include "msc_tma.cuh"

namespace {

constexpr uint32_t kSleepNs = 20000;  // suspend hint of the blocks' mbarrier waits

constexpr int kP = 64;    // head dimension
constexpr int kN = 128;   // state size
constexpr int kHB = 16;   // heads per CTA of the state and scan kernels

using msc::bulk_g2s;
using msc::pack_bf16x2;
using msc::split_bf16x2;
using msc::split_bf16x2_packed;
using msc::st_cs_v8;

__device__ unsigned int g_ssd_status[2];

__device__ __forceinline__ void record_timeout(unsigned int site) {
    if (atomicCAS(&g_ssd_status[0], 0u, (unsigned int)MSC_ERR_TIMEOUT) == 0u) g_ssd_status[1] = site;
}

struct SsdParams {
    const uint16_t* x;      // [b, L, H, P] bf16
    const uint16_t* delta;  // [b, L, H] bf16
    const uint16_t* B;      // [b, L, G, N] bf16
    const uint16_t* C;      // [b, L, G, N] bf16
    const uint16_t* z;      // [b, L, H, P] bf16 or null
    const float* A;         // [H]
    const float* D;         // [H] or null
    const float* bias;      // [H] or null
    float* y;               // [b, L, H, P]
    float* final_state;     // [b, H, P, N] or null
    float* dt;              // [b, H, Lp]
    float* cs;              // [b, H, Lp]
    float* S;               // [b, nc, H, P, N]
    uint16_t* Hin;          // [b, nc, H] pairs (hi, lo) of 64 x 128 bf16 K-major SW128 tile images
    float* Hin32;           // [b, nc, H, P, N] fp32 copy of the same states, or null
    int64_t L, Lp;
    int batch, H, G, hpg, Q, nc;
};

__device__ __forceinline__ float bf(uint16_t v) { return __uint_as_float(((uint32_t)v) << 16); }

// ------------------------------------------------------------------ (1) prep
// One CTA per (chunk, head, batch), one thread per step: Delta and the in-chunk
// inclusive prefix sum of Delta A (zero past the sequence end).
__global__ void __launch_bounds__(256) ssd_prep_kernel(const SsdParams p) {
    __shared__ float s_w[8];
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t t = (int64_t)c * p.Q + tid;
    float dt = 0.f;
    if (tid < p.Q && t < p.L) {
        const float xv = bf(p.delta[((int64_t)b * p.L + t) * p.H + h]) + (p.bias ? p.bias[h] : 0.f);
        dt = msc::softplus_f(xv);
    }
    float v = dt * p.A[h];
    // inclusive scan: warp shuffles, then warp totals
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) s_w[warp] = v;
    __syncthreads();
    float add = 0.f;
    for (int w = 0; w < warp; ++w) add += s_w[w];
    v += add;
    if (tid < p.Q) {
        const size_t o = ((size_t)b * p.H + h) * p.Lp + (size_t)c * p.Q + tid;
        p.dt[o] = dt;
        p.cs[o] = v;
    }
}




constexpr int kHBS = 8;  // heads per CTA of the state kernel

// ------------------------------------------------------ (2) chunk states
// S_c^T[n, p] = sum_j B_j[n] Xw_j[p], Xw_j = exp(cs_last - cs_j) Delta_j x_j, as
// a tcgen05 GEMM (M = 128 states, N = 64, K = Q steps) whose operands are the
// TMA tiles themselves, used MN-major: B [Q j][128 n] as A (two 64-wide n
// blocks) and x [Q j][64 p], scaled in place by the step weights and split
// into bf16 hi + lo tiles, as B.  x tiles (with the head's Delta and cs rows)
// are double-buffered: the load of head h + 1 is issued as soon as the MMAs of
// head h - 1 have released its buffer, and the epilogue of head h - 1 runs
// while the MMAs of head h do.
struct StateSmem {
    uint8_t* sB;
    uint8_t* sX;
    uint8_t* sL;
    float* s_dc;  // [2 buffers][Delta, cs][256]
    uint64_t* bars;  // 0: B, 1-2: x buffers, 3-4: MMA of a buffer
};

__device__ __forceinline__ void state_issue_head(const StateSmem m, const CUtensorMap* tmX, const CUtensorMap* tmZ,
                                                 const SsdParams& p, int h, int s, int c, int b) {
    const int Q = p.Q;
    const uint32_t tile = (uint32_t)Q * 128u;
    const size_t dbase = ((size_t)b * p.H + h) * p.Lp + (size_t)c * Q;
    msc::mbar_arrive_expect_tx(&m.bars[1 + s], (tmZ ? 2u : 1u) * tile + 8u * (uint32_t)Q);
    msc::tma_load_3d(m.sX + s * tile, tmX, &m.bars[1 + s], h * kP, c * Q, b);
    if (tmZ) msc::tma_load_3d(m.sL + s * tile, tmZ, &m.bars[1 + s], h * kP, c * Q, b);
    bulk_g2s(m.s_dc + s * 512, p.dt + dbase, 4u * (uint32_t)Q, &m.bars[1 + s]);
    bulk_g2s(m.s_dc + s * 512 + 256, p.cs + dbase, 4u * (uint32_t)Q, &m.bars[1 + s]);
}

// kMode 0: the chunk states above.  The same product with other operands gives
// the backward's U_c^T[n, p] = sum_i C_i[n] exp(cs_i) g_i[p] (the gradient that
// reaches the state entering chunk c from the chunk's own outputs): tmB maps C,
// tmX maps dy, and with kMode 2 tmZ maps z, which lands in the lo buffer and
// gates g = dy silu(z) before the split; the result goes to p.S.
template <int kMode>
__global__ void __launch_bounds__(256) ssd_state_kernel(const __grid_constant__ CUtensorMap tmB,
                                                        const __grid_constant__ CUtensorMap tmX,
                                                        const __grid_constant__ CUtensorMap tmZ, const SsdParams p) {
    extern __shared__ uint8_t s_dyn[];
    uint8_t* base = s_dyn + ((1024u - (msc::smem_u32(s_dyn) & 1023u)) & 1023u);  // 1024-aligned, still a shared address
    const int Q = p.Q;
    const uint32_t tile = (uint32_t)Q * 128u;  // bytes of one [Q][64] bf16 tile
    StateSmem m;
    m.sB = base;                // 2 tiles (n blocks)
    m.sX = m.sB + 2 * tile;     // 2 buffers: x, then Xw hi in place
    m.sL = m.sX + 2 * tile;     // 2 buffers: Xw lo
    m.s_dc = reinterpret_cast<float*>(m.sL + 2 * tile);
    m.bars = reinterpret_cast<uint64_t*>(m.s_dc + 1024);
    uint32_t* slot = reinterpret_cast<uint32_t*>(m.bars + 5);

    const int c = blockIdx.x, hb = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h0 = hb * kHBS;
    const int nh = min(kHBS, p.H - h0);
    const int g = h0 / p.hpg;

    if (warp == 0) {
        msc::tmem_alloc(slot, 128);
        msc::tmem_relinquish();
    }
    if (tid == 0) {
        for (int k = 0; k < 5; ++k) msc::mbar_init(&m.bars[k], 1);
        msc::fence_barrier_init();
        msc::prefetch_tmap(&tmB);
        msc::prefetch_tmap(&tmX);
        msc::mbar_arrive_expect_tx(&m.bars[0], 2 * tile);
        for (int nb = 0; nb < 2; ++nb) msc::tma_load_3d(m.sB + nb * tile, &tmB, &m.bars[0], g * kN + nb * 64, c * Q, b);
        if (kMode == 2) msc::prefetch_tmap(&tmZ);
        for (int it = 0; it < 2 && it < nh; ++it) state_issue_head(m, &tmX, kMode == 2 ? &tmZ : nullptr, p, h0 + it, it, c, b);
    }
    __syncthreads();
    const uint32_t tmem = *slot;
    const uint32_t idesc = msc::idesc_f16(true, 128, kP, true, true);
    bool ok = msc::wait_bounded(&m.bars[0], 0, nullptr, kSleepNs);
    bool failed = false;

    // S of head hp from accumulator buffer sp: lane = n, column = p; warps w and
    // w + 4 read lanes 32 (w % 4) .. and split the 64 columns
    auto epilogue = [&](int hp, int sp) {
        const int lq = warp & 3, c0 = 32 * (warp >> 2);
        float* dst = p.S + ((((size_t)b * p.nc + c) * p.H + hp) * kP) * kN + (32 * lq + lane);
        float v[32];
        msc::tmem_ld16(tmem + 64 * sp + ((uint32_t)(32 * lq) << 16) + (uint32_t)c0, v);
        msc::tmem_ld16(tmem + 64 * sp + ((uint32_t)(32 * lq) << 16) + (uint32_t)(c0 + 16), v + 16);
        msc::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) __stcs(dst + (size_t)(c0 + i) * kN, v[i]);
        msc::tc_fence_before();
    };

    for (int it = 0; it < nh; ++it) {
        const int s = it & 1;
        if (it >= 1) {
            // MMAs of head it - 1 done: its x buffer takes head it + 1
            ok = msc::wait_bounded(&m.bars[3 + (s ^ 1)], (uint32_t)(((it - 1) >> 1) & 1), nullptr, kSleepNs) && ok;
            if (__syncthreads_or(!ok)) {
                if (tid == 0) record_timeout(20);
                failed = true;
                break;
            }
            if (tid == 0 && it + 1 < nh)
                state_issue_head(m, &tmX, kMode == 2 ? &tmZ : nullptr, p, h0 + it + 1, s ^ 1, c, b);
        }
        ok = msc::wait_bounded(&m.bars[1 + s], (uint32_t)((it >> 1) & 1), nullptr, kSleepNs) && ok;
        if (__syncthreads_or(!ok)) {
            if (tid == 0) record_timeout(21);
            failed = true;
            break;
        }
        // Xw = w_j x_j, split into hi (in place) and lo; row j of the tile is
        // 128 bytes (64 p), the swizzle only permutes chunks within the row
        {
            uint8_t* xs = m.sX + s * tile;
            uint8_t* ls = m.sL + s * tile;
            const float* s_dt = m.s_dc + s * 512;
            const float* s_cs = s_dt + 256;
            const float cs_last = s_cs[Q - 1];
            for (int u = tid; u < Q * 8; u += 256) {
                const int j = u >> 3;
                const float wj = kMode == 0 ? msc::ex2_approx((cs_last - s_cs[j]) * MSC_LOG2E) * s_dt[j]
                                            : msc::ex2_approx(s_cs[j] * MSC_LOG2E);
                uint4 v = *reinterpret_cast<const uint4*>(xs + u * 16);
                uint32_t w[4] = {v.x, v.y, v.z, v.w}, hi[4], lo[4];
                const uint64_t wj2 = msc::pk2(wj, wj);
                if (kMode == 2) {
                    const uint4 zv = *reinterpret_cast<const uint4*>(ls + u * 16);
                    const uint32_t zw[4] = {zv.x, zv.y, zv.z, zv.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        split_bf16x2_packed(msc::mul2(msc::mul2(wj2, msc::pk2(msc::bf16lo(w[e]), msc::bf16hi(w[e]))),
                                                      msc::silu_2(msc::pk2(msc::bf16lo(zw[e]), msc::bf16hi(zw[e])))),
                                            hi[e], lo[e]);
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        split_bf16x2_packed(msc::mul2(wj2, msc::pk2(msc::bf16lo(w[e]), msc::bf16hi(w[e]))), hi[e], lo[e]);
                }
                *reinterpret_cast<uint4*>(xs + u * 16) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4*>(ls + u * 16) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            msc::fence_proxy_async_smem();
            msc::tc_fence_before();
            __syncthreads();
            msc::tc_fence_after();
            if (tid == 0) {
                const uint32_t aB = msc::smem_u32(m.sB), aX = msc::smem_u32(xs), aL = msc::smem_u32(ls);
                for (int k = 0; k < Q / 16; ++k) {
                    const uint64_t ad = msc::sdesc_sw128_mn(aB + k * 2048, tile);
                    msc::mma_f16(tmem + 64 * s, ad, msc::sdesc_sw128_mn(aX + k * 2048, tile), idesc, k > 0 ? 1u : 0u);
                    msc::mma_f16(tmem + 64 * s, ad, msc::sdesc_sw128_mn(aL + k * 2048, tile), idesc, 1u);
                }
                msc::mma_commit(&m.bars[3 + s]);
            }
        }
        if (it >= 1) epilogue(h0 + it - 1, s ^ 1);  // its MMAs were waited for above
    }
    if (!failed && nh > 0) {
        const int it = nh - 1;
        ok = msc::wait_bounded(&m.bars[3 + (it & 1)], (uint32_t)((it >> 1) & 1), nullptr, kSleepNs);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) record_timeout(22);
        } else {
            msc::tc_fence_after();
            epilogue(h0 + it, it & 1);
        }
    }
    msc::tc_fence_before();
    __syncthreads();
    if (warp == 0) msc::tmem_dealloc(tmem, 128);
}

// ------------------------------------------------------------ (3) state pass
// One thread per (b, h, p, 8 consecutive n): Hin of every chunk (also in fp32
// when Hin32 is set, for the backward) as bf16 hi + lo
// tile images (K-major [64 p][128 n], 128-byte swizzle: one 16-byte chunk per
// thread and chunk) for the scan kernel's tensor cores, and the final state.
// The chunk states are loaded eight chunks ahead of the dependent chain.
__global__ void __launch_bounds__(256) ssd_pass_kernel(const SsdParams p) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int b = blockIdx.y;
    constexpr int kN8 = kN / 8;
    if (idx >= (int64_t)p.H * kP * kN8) return;
    const int n0 = (int)(idx % kN8) * 8;
    const int pp = (int)((idx / kN8) % kP);
    const int h = (int)(idx / (kN8 * kP));
    const size_t dbase = ((size_t)b * p.H + h) * p.Lp;
    const uint32_t off = msc::sw128_offset(pp, n0, kP);
    float run[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) run[e] = 0.f;
    for (int c0 = 0; c0 < p.nc; c0 += 8) {
        float4 sv[8][2];
        float dv[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int c = c0 + k;
            if (c < p.nc) {
                const float4* src = reinterpret_cast<const float4*>(
                    p.S + ((((size_t)b * p.nc + c) * p.H + h) * kP + pp) * kN + n0);
                sv[k][0] = __ldcs(src);
                sv[k][1] = __ldcs(src + 1);
                dv[k] = p.cs[dbase + (size_t)c * p.Q + p.Q - 1];
            } else {
                sv[k][0] = sv[k][1] = make_float4(0.f, 0.f, 0.f, 0.f);
                dv[k] = 0.f;
            }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int c = c0 + k;
            if (c >= p.nc) break;
            uint8_t* tile = reinterpret_cast<uint8_t*>(p.Hin + (((size_t)b * p.nc + c) * p.H + h) * (2 * kP * kN));
            if (p.Hin32) {
                float4* dst = reinterpret_cast<float4*>(p.Hin32 + ((((size_t)b * p.nc + c) * p.H + h) * kP + pp) * kN + n0);
                dst[0] = make_float4(run[0], run[1], run[2], run[3]);
                dst[1] = make_float4(run[4], run[5], run[6], run[7]);
            }
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) split_bf16x2(run[2 * e], run[2 * e + 1], hi[e], lo[e]);
            *reinterpret_cast<uint4*>(tile + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(tile + kP * kN * 2 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            const float a = msc::ex2_approx(dv[k] * MSC_LOG2E);
            const float s8[8] = {sv[k][0].x, sv[k][0].y, sv[k][0].z, sv[k][0].w,
                                 sv[k][1].x, sv[k][1].y, sv[k][1].z, sv[k][1].w};
#pragma unroll
            for (int e = 0; e < 8; ++e) run[e] = fmaf(a, run[e], s8[e]);
        }
    }
    if (p.final_state) {
        float4* dst = reinterpret_cast<float4*>(p.final_state + (((size_t)b * p.H + h) * kP + pp) * kN + n0);
        dst[0] = make_float4(run[0], run[1], run[2], run[3]);
        dst[1] = make_float4(run[4], run[5], run[6], run[7]);
    }
}

// ------------------------------------------------------------ (4) chunk scan
struct ScanMaps {
    CUtensorMap C, B, xs, xq;
};

constexpr int kScanCompute = 16;                       // warps forming M' and running the epilogue
constexpr int kWarpLoad = kScanCompute;                // warp streaming x, Delta, cs and Hin
constexpr int kWarpMma = kScanCompute + 1;             // warp issuing the tensor-core MMAs
constexpr int kScanThreads = (kScanCompute + 2) * 32;


// CTA = (chunk c, row block ib of 128 rows, block of kHB heads, batch b), in
// three roles that hand work over through mbarriers:
//  * load warp: streams, one head ahead, the x tile with the head's Delta and
//    cs rows (double-buffered) and the Hin hi + lo images (reloaded as soon as
//    the head's Y_off MMAs have read them);
//  * MMA warp: G = C B^T once (bf16 K-major TMA tiles, into tensor memory),
//    then per head Y_off = C Hin^T and Y_diag = M' x, one 64-column quarter of
//    M' at a time, into one of two accumulator pairs;
//  * 16 compute warps: warp w owns rows 32 (w % 4) + lane (its TMEM lanes) and
//    16 columns of every quarter.  They form M'[i, j] = G[i, j] exp(cs_i -
//    cs_j) Delta_j for j <= i, plus D on the diagonal so that D x_i comes out
//    of the same product, split into bf16 hi + lo, into two alternating
//    quarter buffers; blocks above the diagonal are written as zeros without
//    arithmetic.  The epilogue of head h (y = Y_diag + exp(cs_i) Y_off, times
//    silu(z)) runs after the quarters of head h + 1 have been handed over, so
//    the tensor cores are never waited for.
__global__ void __launch_bounds__(kScanThreads, 1) ssd_scan_kernel(const __grid_constant__ CUtensorMap tmC,
                                                                   const __grid_constant__ CUtensorMap tmB,
                                                                   const __grid_constant__ CUtensorMap tmX,
                                                                   const SsdParams p) {
    extern __shared__ uint8_t s_dyn[];
    uint8_t* base = s_dyn + ((1024u - (msc::smem_u32(s_dyn) & 1023u)) & 1023u);  // 1024-aligned, still a shared address
    const int Q = p.Q;
    const int nib = (Q + 127) / 128;
    const int c = blockIdx.x / nib, ib = blockIdx.x % nib;
    const int hb = blockIdx.y, b = blockIdx.z;
    const int Qi = min(Q, (ib + 1) * 128);       // columns j of this row block: [0, Qi)
    const int rows_valid = min(128, Q - ib * 128);
    const int xrows = min(Q, 128);               // rows of one x box
    const int nq = Qi / 64;
    uint8_t* sC = base;                          // [2 kb][128 i][128 B], K-major
    uint8_t* sBM = sC + 32768;                   // B [2 kb][Q j][128 B] for G, then 2 x (hi, lo) quarter buffers
    uint8_t* sX = sBM + 65536;                   // 2 x: x [Qi j][64 p], MN-major
    uint8_t* sH = sX + 65536;                    // Hin hi [2 kb][64 p][128 B], then lo
    float* s_dc = reinterpret_cast<float*>(sH + 32768);  // [2 buffers][Delta, cs][256]
    float* s_w = s_dc + 1024;                    // per compute warp: log2(Delta_j), then -cs_j, 64 columns each
    float* s_D = s_w + kScanCompute * 128;       // D of the block's heads
    uint64_t* bars = reinterpret_cast<uint64_t*>(s_D + 64);
    // 0 C+B loaded, 1 G done, 2-3 x full, 4 Hin full, 5 Y_off done, 6-7 quarter built (16 arrivals),
    // 8-9 quarter consumed, 10-11 x free, 12-13 head done, 14-15 accumulator free (16 arrivals), 16 drain
    uint32_t* slot = reinterpret_cast<uint32_t*>(bars + 17);
    volatile uint32_t* abort = slot + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h0 = hb * kHB;
    const int nh = min(kHB, p.H - h0);
    const int g = h0 / p.hpg;
    const int64_t tc0 = (int64_t)c * Q;
    const uint32_t tG = 0;
    const uint32_t xbytes = (uint32_t)Qi * 128u;

    if (warp == 0) {
        msc::tmem_alloc(slot, 512);
        msc::tmem_relinquish();
    }
    if (tid == 0) {
        for (int k = 0; k < 17; ++k) msc::mbar_init(&bars[k], (k == 6 || k == 7 || k == 14 || k == 15) ? kScanCompute : 1);
        msc::fence_barrier_init();
        *abort = 0u;
    }
    if (tid < kHB) s_D[tid] = (p.D && tid < nh) ? p.D[h0 + tid] : 0.f;
    __syncthreads();
    const uint32_t tmem = *slot;

    if (warp == kWarpLoad) {
        // ---------------------------------------------------------- loads
        if (lane == 0) {
            msc::prefetch_tmap(&tmC);
            msc::prefetch_tmap(&tmB);
            msc::prefetch_tmap(&tmX);
            msc::mbar_arrive_expect_tx(&bars[0], 2u * 128u * 128u + 2u * (uint32_t)Q * 128u);
            for (int kb = 0; kb < 2; ++kb) {
                msc::tma_load_3d(sC + kb * 16384, &tmC, &bars[0], g * kN + kb * 64, (int)(tc0 + ib * 128), b);
                msc::tma_load_3d(sBM + kb * Q * 128, &tmB, &bars[0], g * kN + kb * 64, (int)tc0, b);
            }
        }
        bool pok = true;
        int nx0 = 0, nx1 = 0, nhin = 0;
        for (int it = 0; it < nh; ++it) {
            const int s = it & 1, h = h0 + it;
            if (it >= 2) {
                pok = __all_sync(0xffffffffu, msc::wait_bounded(&bars[10 + s], (uint32_t)(((it - 2) >> 1) & 1), abort, kSleepNs));
                if (!pok) break;
            }
            if (lane == 0) {
                const size_t dbase = ((size_t)b * p.H + h) * p.Lp + (size_t)tc0;
                msc::mbar_arrive_expect_tx(&bars[2 + s], xbytes + 8u * (uint32_t)Qi);
                for (int r = 0; r < Qi; r += xrows)
                    msc::tma_load_3d(sX + s * 32768 + r * 128, &tmX, &bars[2 + s], h * kP, (int)(tc0 + r), b);
                bulk_g2s(s_dc + s * 512, p.dt + dbase, 4u * (uint32_t)Qi, &bars[2 + s]);
                bulk_g2s(s_dc + s * 512 + 256, p.cs + dbase, 4u * (uint32_t)Qi, &bars[2 + s]);
            }
            if (s == 0) ++nx0; else ++nx1;
            if (it >= 1) {
                pok = __all_sync(0xffffffffu, msc::wait_bounded(&bars[5], (uint32_t)((it - 1) & 1), abort, kSleepNs));
                if (!pok) break;
            }
            if (lane == 0) {
                msc::mbar_arrive_expect_tx(&bars[4], 32768u);
                bulk_g2s(sH, p.Hin + (((size_t)b * p.nc + c) * p.H + h) * (2 * kP * kN), 32768u, &bars[4]);
            }
            ++nhin;
        }
        if (!pok && lane == 0) {
            record_timeout(50);
            *abort = 1u;
        }
        // every load issued lands before the block ends (they have all been
        // consumed already unless the block gives up)
        bool dok = true;
        if (nx0 > 0) dok = msc::wait_bounded(&bars[2], (uint32_t)((nx0 - 1) & 1), nullptr, kSleepNs) && dok;
        if (nx1 > 0) dok = msc::wait_bounded(&bars[3], (uint32_t)((nx1 - 1) & 1), nullptr, kSleepNs) && dok;
        if (nhin > 0) dok = msc::wait_bounded(&bars[4], (uint32_t)((nhin - 1) & 1), nullptr, kSleepNs) && dok;
        if (!dok && lane == 0) record_timeout(51);
    } else if (warp == kWarpMma) {
        // ---------------------------------------------------------- MMA issue
        if (lane == 0) {
            const uint32_t id64 = msc::idesc_f16(true, 128, kP);                // A, B K-major
            const uint32_t id64x = msc::idesc_f16(true, 128, kP, false, true);  // B MN-major (x)
            bool mok = msc::wait_bounded(&bars[0], 0, abort, kSleepNs);
            if (mok) {
                msc::tc_fence_after();
                const uint32_t idesc = msc::idesc_f16(true, 128, Qi);
                for (int k = 0; k < 8; ++k) {
                    const uint32_t koff = (uint32_t)((k & 3) * 32);
                    const uint64_t ad = msc::sdesc_sw128(msc::smem_u32(sC + (k >> 2) * 16384) + koff);
                    const uint64_t bd = msc::sdesc_sw128(msc::smem_u32(sBM + (k >> 2) * Q * 128) + koff);
                    msc::mma_f16(tmem + tG, ad, bd, idesc, k > 0 ? 1u : 0u);
                }
                msc::mma_commit(&bars[1]);
            }
            for (int it = 0; it < nh && mok; ++it) {
                const int s = it & 1;
                const uint32_t tYd = 256u + 128u * (uint32_t)s, tYo = tYd + 64u;
                mok = msc::wait_bounded(&bars[2 + s], (uint32_t)((it >> 1) & 1), abort, kSleepNs) &&
                      msc::wait_bounded(&bars[4], (uint32_t)(it & 1), abort, kSleepNs);
                if (mok && it >= 2) mok = msc::wait_bounded(&bars[14 + s], (uint32_t)(((it - 2) >> 1) & 1), abort, kSleepNs);
                if (!mok) break;
                msc::tc_fence_after();
                const uint32_t aC = msc::smem_u32(sC), aH = msc::smem_u32(sH);
                for (int k = 0; k < kN / 16; ++k) {
                    const uint32_t koff = (uint32_t)((k >> 2) * 16384 + (k & 3) * 32);
                    const uint32_t hoff = (uint32_t)((k >> 2) * kP * 128 + (k & 3) * 32);
                    msc::mma_f16(tmem + tYo, msc::sdesc_sw128(aC + koff), msc::sdesc_sw128(aH + hoff), id64,
                                 k > 0 ? 1u : 0u);
                    msc::mma_f16(tmem + tYo, msc::sdesc_sw128(aC + koff), msc::sdesc_sw128(aH + 16384 + hoff), id64, 1u);
                }
                msc::mma_commit(&bars[5]);
                const uint32_t aX = msc::smem_u32(sX + s * 32768);
                for (int q = 0; q < nq; ++q) {
                    const int u = it * nq + q, bq = u & 1;
                    mok = msc::wait_bounded(&bars[6 + bq], (uint32_t)((u >> 1) & 1), abort, kSleepNs);
                    if (!mok) break;
                    msc::tc_fence_after();
                    const uint32_t aHi = msc::smem_u32(sBM + bq * 32768), aLo = aHi + 16384u;
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t bd = msc::sdesc_sw128_mn(aX + (uint32_t)(64 * q + 16 * k) * 128u, 32768u);
                        msc::mma_f16(tmem + tYd, msc::sdesc_sw128(aHi + k * 32), bd, id64x, (q > 0 || k > 0) ? 1u : 0u);
                        msc::mma_f16(tmem + tYd, msc::sdesc_sw128(aLo + k * 32), bd, id64x, 1u);
                    }
                    msc::mma_commit(&bars[8 + bq]);
                }
                if (!mok) break;
                msc::mma_commit(&bars[10 + s]);
                msc::mma_commit(&bars[12 + s]);
            }
            if (!mok) {
                record_timeout(46);
                *abort = 1u;
            }
            // every MMA issued completes before the tensor memory is released
            msc::mma_commit(&bars[16]);
            if (!msc::wait_bounded(&bars[16], 0, nullptr, kSleepNs)) record_timeout(47);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ M' quarters and epilogue
        const int lq = warp & 3, cslot = warp >> 2;
        const int i_loc = 32 * lq + lane;
        const int i_chk = ib * 128 + i_loc;
        const int row_lo = ib * 128 + 32 * lq;     // first row of this warp
        const uint32_t lane_off = (uint32_t)(32 * lq) << 16;
        float* my_w = s_w + warp * 128;  // log2(Delta_j)
        float* my_c = my_w + 64;         // -cs_j
        bool ok = __all_sync(0xffffffffu, msc::wait_bounded(&bars[1], 0, abort, kSleepNs));
        msc::tc_fence_after();
        float csi_prev = 0.f;
        uint4 z_prev[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
        // y of head hp (row scale csi_prev, gate z_prev); `release` hands the
        // accumulator pair back to the MMA warp once it has been read
        auto epilogue = [&](int hp, bool release) -> bool {
            const int sp = hp & 1;
            if (!__all_sync(0xffffffffu, msc::wait_bounded(&bars[12 + sp], (uint32_t)((hp >> 1) & 1), abort, kSleepNs)))
                return false;
            msc::tc_fence_after();
            float yd[16], yo[16];
            const uint32_t tYd = 256u + 128u * (uint32_t)sp;
            msc::tmem_ld16(tmem + tYd + lane_off + (uint32_t)(16 * cslot), yd);
            msc::tmem_ld16(tmem + tYd + 64u + lane_off + (uint32_t)(16 * cslot), yo);
            msc::tmem_ld_wait();
            msc::tc_fence_before();
            __syncwarp();
            if (release && lane == 0) msc::mbar_arrive(&bars[14 + sp]);
            const int64_t t = tc0 + i_chk;
            if (i_loc < rows_valid && t < p.L) {
                const float e_i = msc::ex2_approx(csi_prev * MSC_LOG2E);
                float out[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) out[e] = fmaf(e_i, yo[e], yd[e]);
                if (p.z) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const uint32_t zw[4] = {z_prev[e].x, z_prev[e].y, z_prev[e].z, z_prev[e].w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            out[8 * e + 2 * k] *= msc::silu_f(msc::bf16lo(zw[k]));
                            out[8 * e + 2 * k + 1] *= msc::silu_f(msc::bf16hi(zw[k]));
                        }
                    }
                }
                float* yrow = p.y + (((int64_t)b * p.L + t) * p.H + h0 + hp) * kP + 16 * cslot;
                st_cs_v8(yrow, out);
                st_cs_v8(yrow + 8, out + 8);
            }
            return true;
        };
        for (int it = 0; it <= nh && ok; ++it) {
            if (it < nh) {
                const int s = it & 1;
                ok = __all_sync(0xffffffffu, msc::wait_bounded(&bars[2 + s], (uint32_t)((it >> 1) & 1), abort, kSleepNs));
                if (!ok) break;
                const float* s_dt = s_dc + s * 512;
                const float* s_cs = s_dt + 256;
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int idx = lane + 32 * r;
                    const int j = 64 * (idx >> 4) + 16 * cslot + (idx & 15);
                    float wv = 0.f, cv = 0.f;
                    if (j < Qi) {
                        const float dtj = s_dt[j];
                        wv = dtj > 0.f ? __log2f(dtj) : -INFINITY;
                        cv = -s_cs[j];
                    }
                    my_w[idx] = wv;
                    my_c[idx] = cv;
                }
                // the decay exponent is formed as (cs_i - cs_j) log2(e) + log2(Delta_j):
                // the difference of two nearby cumulative sums is exact, so the
                // decays near the diagonal, where they are close to 1, keep full
                // precision however large cs grows along the chunk
                const float csi = s_cs[i_chk < Qi ? i_chk : 0];
                const float Dh = s_D[it];
                __syncwarp();
                for (int q = 0; q < nq; ++q) {
                    // quarter u alternates between buffers u % 2; before refilling
                    // one, wait for the MMAs of its previous use (u - 2)
                    const int u = it * nq + q, bq = u & 1;
                    if (u >= 2) {
                        ok = __all_sync(0xffffffffu,
                                        msc::wait_bounded(&bars[8 + bq], (uint32_t)(((u >> 1) - 1) & 1), abort, kSleepNs));
                        if (!ok) break;
                    }
                    const int j0 = 64 * q + 16 * cslot;
                    uint32_t ph[8], pl[8];
                    if (j0 > row_lo + 31 || row_lo >= Qi) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) ph[e] = pl[e] = 0u;
                    } else {
                        float gv[16];
                        msc::tmem_ld16(tmem + tG + lane_off + (uint32_t)j0, gv);
                        float wv[16], cv[16];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float4 w4 = reinterpret_cast<const float4*>(my_w + 16 * q)[e];
                            const float4 c4 = reinterpret_cast<const float4*>(my_c + 16 * q)[e];
                            wv[4 * e] = w4.x; wv[4 * e + 1] = w4.y; wv[4 * e + 2] = w4.z; wv[4 * e + 3] = w4.w;
                            cv[4 * e] = c4.x; cv[4 * e + 1] = c4.y; cv[4 * e + 2] = c4.z; cv[4 * e + 3] = c4.w;
                        }
                        msc::tmem_ld_wait();
                        if (j0 + 15 <= row_lo) {
                            // every column at or below every row of the warp: packed
                            // pair arithmetic, no masks
                            const uint64_t csi2 = msc::pk2(csi, csi);
                            const uint64_t l2e2 = msc::pk2(MSC_LOG2E, MSC_LOG2E);
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const uint64_t x = msc::fma2(msc::add2(csi2, msc::pk2(cv[2 * e], cv[2 * e + 1])), l2e2,
                                                             msc::pk2(wv[2 * e], wv[2 * e + 1]));
                                const uint64_t v = msc::mul2(msc::ex2_2(x), msc::pk2(gv[2 * e], gv[2 * e + 1]));
                                split_bf16x2_packed(v, ph[e], pl[e]);
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const int ja = j0 + 2 * e, jb = ja + 1;
                                float va = (ja <= i_chk)
                                               ? gv[2 * e] * msc::ex2_approx(fmaf(csi + cv[2 * e], MSC_LOG2E, wv[2 * e]))
                                               : 0.f;
                                float vb = (jb <= i_chk)
                                               ? gv[2 * e + 1] * msc::ex2_approx(fmaf(csi + cv[2 * e + 1], MSC_LOG2E, wv[2 * e + 1]))
                                               : 0.f;
                                if (ja == i_chk) va += Dh;
                                if (jb == i_chk) vb += Dh;
                                split_bf16x2(va, vb, ph[e], pl[e]);
                            }
                        }
                    }
                    uint8_t* bh = sBM + bq * 32768;
                    const uint32_t o0 = msc::sw128_offset(i_loc, 16 * cslot, 128);
                    const uint32_t o1 = msc::sw128_offset(i_loc, 16 * cslot + 8, 128);
                    *reinterpret_cast<uint4*>(bh + o0) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
                    *reinterpret_cast<uint4*>(bh + o1) = make_uint4(ph[4], ph[5], ph[6], ph[7]);
                    *reinterpret_cast<uint4*>(bh + 16384 + o0) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
                    *reinterpret_cast<uint4*>(bh + 16384 + o1) = make_uint4(pl[4], pl[5], pl[6], pl[7]);
                    msc::fence_proxy_async_smem();
                    msc::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) msc::mbar_arrive(&bars[6 + bq]);
                }
                if (!ok) break;
                // epilogue of head it - 1, then keep this head's row scale and gate
                if (it >= 1) {
                    ok = epilogue(it - 1, true);
                    if (!ok) break;
                }
                csi_prev = csi;
                {
                    const int64_t t = tc0 + i_chk;
                    if (p.z && i_loc < rows_valid && t < p.L) {
                        const uint4* zrow = reinterpret_cast<const uint4*>(
                            p.z + (((int64_t)b * p.L + t) * p.H + h0 + it) * kP + 16 * cslot);
                        z_prev[0] = __ldcs(zrow);
                        z_prev[1] = __ldcs(zrow + 1);
                    }
                }
            } else {
                ok = epilogue(nh - 1, false);  // the last head
            }
        }
        if (!ok && lane == 0) {
            record_timeout(42);
            *abort = 1u;
        }
    }
    msc::tc_fence_before();
    __syncthreads();
    if (warp == 0) msc::tmem_dealloc(tmem, 512);
}

size_t a256(size_t x) { return (x + 255) / 256 * 256; }

constexpr int kScanSmem = 1024 + 32768 + 65536 + 65536 + 32768 + 4096 + 8192 + 256 + 17 * 8 + 8;

int state_smem(int Q) { return 1024 + 6 * Q * 128 + 4096 + 64; }

}  // namespace

namespace msc_host {

size_t ssd_workspace(int64_t batch, int64_t L, int64_t H, int64_t P, int64_t N, int64_t G, int64_t Q) {
    (void)G;
    const int64_t nc = (L + Q - 1) / Q, Lp = nc * Q;
    size_t ws = a256((size_t)batch * H * Lp * 4) * 2;               // dt, cs
    ws += a256((size_t)batch * nc * H * P * N * 4);                  // S
    ws += a256((size_t)batch * nc * H * P * N * 2 * 2);              // Hin images (hi, lo)
    return ws + 1024;
}

msc_status ssd_launch(const SsdArgs& a, cudaStream_t st) {
    SsdParams p{};
    p.x = static_cast<const uint16_t*>(a.x);
    p.delta = static_cast<const uint16_t*>(a.delta);
    p.B = static_cast<const uint16_t*>(a.B);
    p.C = static_cast<const uint16_t*>(a.C);
    p.z = static_cast<const uint16_t*>(a.z);
    p.A = a.A; p.D = a.D; p.bias = a.delta_bias; p.y = a.y; p.final_state = a.final_state;
    p.Hin32 = a.Hin32;
    p.L = a.L; p.batch = (int)a.batch; p.H = (int)a.H; p.G = (int)a.G; p.hpg = (int)(a.H / a.G); p.Q = (int)a.Q;
    p.nc = (int)((a.L + a.Q - 1) / a.Q);
    p.Lp = (int64_t)p.nc * a.Q;
    if (p.hpg % kHB != 0 && p.G != 1) return fail(MSC_ERR_UNSUPPORTED, "heads per group must be a multiple of %d", kHB);
    char* ws = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(a.workspace) + 1023) & ~uintptr_t(1023));
    p.dt = reinterpret_cast<float*>(ws); ws += a256((size_t)a.batch * a.H * p.Lp * 4);
    p.cs = reinterpret_cast<float*>(ws); ws += a256((size_t)a.batch * a.H * p.Lp * 4);
    p.S = reinterpret_cast<float*>(ws); ws += a256((size_t)a.batch * p.nc * a.H * kP * kN * 4);
    p.Hin = reinterpret_cast<uint16_t*>(ws);

    // (1) Delta, cs
    ssd_prep_kernel<<<dim3(p.nc, p.H, (unsigned)a.batch), 256, 0, st>>>(p);
    msc_status s = check_launch("ssd_prep");
    if (s != MSC_OK) return s;
    // tensor maps: x [b, L, H * P] and B, C [b, L, G * N], boxes of 64 elements
    ScanMaps m;
    {
        const uint64_t bcd[3] = {(uint64_t)(a.G * kN), (uint64_t)a.L, (uint64_t)a.batch};
        const uint64_t bcs[2] = {(uint64_t)(a.G * kN * 2), (uint64_t)(a.L * a.G * kN * 2)};
        const uint32_t cbox[3] = {64, 128, 1};
        const uint32_t qbox[3] = {64, (uint32_t)p.Q, 1};
        const uint32_t sbox[3] = {64, (uint32_t)std::min(p.Q, 128), 1};
        const uint64_t xd[3] = {(uint64_t)(a.H * kP), (uint64_t)a.L, (uint64_t)a.batch};
        const uint64_t xs[2] = {(uint64_t)(a.H * kP * 2), (uint64_t)(a.L * a.H * kP * 2)};
        if (!encode_tmap(&m.C, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.C, bcd, bcs, cbox, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_tmap(&m.B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.B, bcd, bcs, qbox, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_tmap(&m.xq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.x, xd, xs, qbox, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_tmap(&m.xs, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.x, xd, xs, sbox, CU_TENSOR_MAP_SWIZZLE_128B))
            return MSC_ERR_CUDA;
    }
    // (2) chunk states
    {
        static std::atomic<uint64_t> configured{0};  // one bit per device on which the attribute is set
        if (!(configured & msc_host::device_bit())) {
            cudaError_t e = cudaFuncSetAttribute(ssd_state_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, state_smem(256));
            if (e != cudaSuccess) return fail(MSC_ERR_CUDA, "ssd_state smem attribute: %s", cudaGetErrorString(e));
            configured |= msc_host::device_bit();
        }
        ssd_state_kernel<0><<<dim3(p.nc, (p.H + kHBS - 1) / kHBS, (unsigned)a.batch), 256, state_smem(p.Q), st>>>(
            m.B, m.xq, m.xq, p);
        if ((s = check_launch("ssd_state")) != MSC_OK) return s;
    }
    // (3) inter-chunk state pass
    {
        const int64_t per_b = (int64_t)p.H * kP * kN;
        ssd_pass_kernel<<<dim3((unsigned)((per_b / 8 + 255) / 256), (unsigned)a.batch), 256, 0, st>>>(p);
        if ((s = check_launch("ssd_pass")) != MSC_OK) return s;
    }
    // (4) chunk scan
    {
        const int nib = (p.Q + 127) / 128;
        static std::atomic<uint64_t> configured{0};  // one bit per device on which the attribute is set
        if (!(configured & msc_host::device_bit())) {
            cudaError_t e = cudaFuncSetAttribute(ssd_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kScanSmem);
            if (e != cudaSuccess) return fail(MSC_ERR_CUDA, "ssd_scan smem attribute: %s", cudaGetErrorString(e));
            configured |= msc_host::device_bit();
        }
        ssd_scan_kernel<<<dim3(p.nc * nib, (p.H + kHB - 1) / kHB, (unsigned)a.batch), kScanThreads, kScanSmem, st>>>(
            m.C, m.B, m.xs, p);
        if ((s = check_launch("ssd_scan")) != MSC_OK) return s;
    }
    return MSC_OK;
}

msc_status ssd_states(const SsdArgs& a, float* dt, float* cs, float* S, float* Hin32, uint16_t* Himg,
                      cudaStream_t st) {
    SsdParams p{};
    p.x = static_cast<const uint16_t*>(a.x);
    p.delta = static_cast<const uint16_t*>(a.delta);
    p.B = static_cast<const uint16_t*>(a.B);
    p.C = static_cast<const uint16_t*>(a.C);
    p.A = a.A; p.bias = a.delta_bias;
    p.L = a.L; p.batch = (int)a.batch; p.H = (int)a.H; p.G = (int)a.G; p.hpg = (int)(a.H / a.G); p.Q = (int)a.Q;
    p.nc = (int)((a.L + a.Q - 1) / a.Q);
    p.Lp = (int64_t)p.nc * a.Q;
    if (p.hpg % kHBS != 0 && p.G != 1) return fail(MSC_ERR_UNSUPPORTED, "heads per group must be a multiple of %d", kHBS);
    p.dt = dt; p.cs = cs; p.S = S;
    ssd_prep_kernel<<<dim3(p.nc, p.H, (unsigned)a.batch), 256, 0, st>>>(p);
    msc_status s = check_launch("ssd_prep");
    if (s != MSC_OK) return s;
    CUtensorMap mB, mX;
    {
        const uint64_t bcd[3] = {(uint64_t)(a.G * kN), (uint64_t)a.L, (uint64_t)a.batch};
        const uint64_t bcs[2] = {(uint64_t)(a.G * kN * 2), (uint64_t)(a.L * a.G * kN * 2)};
        const uint32_t qbox[3] = {64, (uint32_t)p.Q, 1};
        const uint64_t xd[3] = {(uint64_t)(a.H * kP), (uint64_t)a.L, (uint64_t)a.batch};
        const uint64_t xs[2] = {(uint64_t)(a.H * kP * 2), (uint64_t)(a.L * a.H * kP * 2)};
        if (!encode_tmap(&mB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.B, bcd, bcs, qbox, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_tmap(&mX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.x, xd, xs, qbox, CU_TENSOR_MAP_SWIZZLE_128B))
            return MSC_ERR_CUDA;
    }
    {
        static std::atomic<uint64_t> configured{0};  // one bit per device on which the attribute is set
        if (!(configured & msc_host::device_bit())) {
            cudaError_t e = cudaFuncSetAttribute(ssd_state_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, state_smem(256));
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(ssd_state_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, state_smem(256));
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(ssd_state_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, state_smem(256));
            if (e != cudaSuccess) return fail(MSC_ERR_CUDA, "ssd_state smem attribute: %s", cudaGetErrorString(e));
            configured |= msc_host::device_bit();
        }
        ssd_state_kernel<0><<<dim3(p.nc, (p.H + kHBS - 1) / kHBS, (unsigned)a.batch), 256, state_smem(p.Q), st>>>(
            mB, mX, mX, p);
        if ((s = check_launch("ssd_state")) != MSC_OK) return s;
    }
    // one pass writes the states entering every chunk in fp32 and as the images
    const int64_t per_b = (int64_t)p.H * kP * kN;
    p.Hin = Himg;
    p.Hin32 = Hin32;
    p.final_state = nullptr;
    ssd_pass_kernel<<<dim3((unsigned)((per_b / 8 + 255) / 256), (unsigned)a.batch), 256, 0, st>>>(p);
    return check_launch("ssd_pass");
}

msc_status ssd_ugrad(const SsdArgs& a, const void* dy, const float* cs, float* U, cudaStream_t st) {
    SsdParams p{};
    p.L = a.L; p.batch = (int)a.batch; p.H = (int)a.H; p.G = (int)a.G; p.hpg = (int)(a.H / a.G); p.Q = (int)a.Q;
    p.nc = (int)((a.L + a.Q - 1) / a.Q);
    p.Lp = (int64_t)p.nc * a.Q;
    if (p.hpg % kHBS != 0 && p.G != 1) return fail(MSC_ERR_UNSUPPORTED, "heads per group must be a multiple of %d", kHBS);
    p.cs = const_cast<float*>(cs);
    p.dt = const_cast<float*>(cs);  // read into shared memory with cs; unused by the U weights
    p.S = U;
    CUtensorMap mC, mDy, mZ;
    const uint64_t bcd[3] = {(uint64_t)(a.G * kN), (uint64_t)a.L, (uint64_t)a.batch};
    const uint64_t bcs[2] = {(uint64_t)(a.G * kN * 2), (uint64_t)(a.L * a.G * kN * 2)};
    const uint32_t qbox[3] = {64, (uint32_t)p.Q, 1};
    const uint64_t xd[3] = {(uint64_t)(a.H * kP), (uint64_t)a.L, (uint64_t)a.batch};
    const uint64_t xs[2] = {(uint64_t)(a.H * kP * 2), (uint64_t)(a.L * a.H * kP * 2)};
    if (!encode_tmap(&mC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.C, bcd, bcs, qbox, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tmap(&mDy, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, dy, xd, xs, qbox, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tmap(&mZ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.z ? a.z : dy, xd, xs, qbox, CU_TENSOR_MAP_SWIZZLE_128B))
        return MSC_ERR_CUDA;
    {
        static std::atomic<uint64_t> configured{0};  // one bit per device on which the attribute is set
        if (!(configured & msc_host::device_bit())) {
            cudaError_t e = cudaFuncSetAttribute(ssd_state_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, state_smem(256));
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(ssd_state_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, state_smem(256));
            if (e != cudaSuccess) return fail(MSC_ERR_CUDA, "ssd_state smem attribute: %s", cudaGetErrorString(e));
            configured |= msc_host::device_bit();
        }
    }
    const dim3 grid(p.nc, (p.H + kHBS - 1) / kHBS, (unsigned)a.batch);
    if (a.z)
        ssd_state_kernel<2><<<grid, 256, state_smem(p.Q), st>>>(mC, mDy, mZ, p);
    else
        ssd_state_kernel<1><<<grid, 256, state_smem(p.Q), st>>>(mC, mDy, mZ, p);
    return check_launch("ssd_ugrad");
}

msc_status ssd_take_status(unsigned int* code, unsigned int* site) {
    unsigned int w[2] = {0, 0};
    cudaError_t e = cudaMemcpyFromSymbol(w, g_ssd_status, sizeof(w));
    if (e != cudaSuccess) return fail(MSC_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
    if (w[0] != 0) {
        const unsigned int zz[2] = {0, 0};
        e = cudaMemcpyToSymbol(g_ssd_status, zz, sizeof(zz));
        if (e != cudaSuccess) return fail(MSC_ERR_CUDA, "status clear: %s", cudaGetErrorString(e));
    }
    *code = w[0];
    *site = w[1];
    return MSC_OK;
}

}  // namespace msc_host
