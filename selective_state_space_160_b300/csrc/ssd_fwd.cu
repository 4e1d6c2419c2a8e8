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
// on tcgen05; (3) ssd_pass_kernel: Hin of every chunk and the final state;
// (4) ssd_scan_kernel: G = C B^T once per (chunk, row block, head group) into
// tensor memory, then per head the masked decay matrix (L . G scaled by Delta)
// and x are written to shared memory by CUDA cores and Y_diag, Y_off
// accumulate in tensor memory, read back by tcgen05.ld for the epilogue.
//
// Precision: G is exact from bf16 C, B with fp32 accumulation.  Every operand
// the CUDA cores form in fp32 -- the intra-chunk M'[i, j] = G[i, j]
// exp(cs_i - cs_j) Delta_j, the weighted x of the chunk states and the carried
// state Hin -- is split into two fp16 terms (hi + lo, ~22 significant bits)
// and both terms are multiplied on the tensor cores, while C, B and x convert
// from bf16 to fp16 exactly; every product accumulates in fp32.  A single fp16
// rounding (11-bit significand) measured up to 6.9e-3 relative error on seeded
// inputs: Y_diag and Y_off can be large and cancel at chunk boundaries.
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstdlib>

#include "msc_common.cuh"
#include "msc_internal.h"
#include "msc_tc.cuh"
#include "msc_tma.cuh"

namespace {

constexpr int kP = 64;    // head dimension
constexpr int kN = 128;   // state size
constexpr int kHB = 16;   // heads per CTA of the state and scan kernels

__device__ unsigned int g_ssd_status[2];

__device__ __forceinline__ void record_timeout(unsigned int site) {
    if (atomicCAS(&g_ssd_status[0], 0u, (unsigned int)MSC_ERR_TIMEOUT) == 0u) g_ssd_status[1] = site;
}

// Wait for phase `parity` of `bar`, giving up after about one second.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity) {
    if (msc::mbar_wait(bar, parity, 256)) return true;
    uint64_t t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    while (true) {
        if (msc::mbar_try_wait(bar, parity)) return true;
        uint64_t t1;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
        if (t1 - t0 > 1000000000ull) return false;
    }
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
    uint16_t* Hin;          // [b, nc, H] pairs (hi, lo) of 64 x 128 fp16 K-major SW128 tile images
    int64_t L, Lp;
    int H, G, hpg, Q, nc;
};

// fp32 -> fp16 bit pattern, round to nearest even
__device__ __forceinline__ uint16_t f2h_bits(float v) {
    uint16_t r;
    asm("cvt.rn.f16.f32 %0, %1;" : "=h"(r) : "f"(v));
    return r;
}
__device__ __forceinline__ float bf(uint16_t v) { return __uint_as_float(((uint32_t)v) << 16); }
__device__ __forceinline__ float h2f(uint16_t v) {
    float r;
    asm("cvt.f32.f16 %0, %1;" : "=f"(r) : "h"(v));
    return r;
}

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

// ------------------------------------------------------ (2) chunk states
// S_c^T[n, p] = sum_j B_j[n] * (exp(cs_last - cs_j) Delta_j x_j[p]) as a
// tcgen05 GEMM: M = 128 (n), N = 64 (p), K = Q (j).  A = B^T and B = Xw^T are
// transposed into K-major SW128 tiles by the CUDA cores.
__global__ void __launch_bounds__(128) ssd_state_kernel(const SsdParams p) {
    extern __shared__ uint8_t s_dyn[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(s_dyn) + 1023) & ~uintptr_t(1023));
    const int Q = p.Q;
    uint8_t* sBt = base;                   // [128 n][Q j] fp16
    uint8_t* sXw = base + kN * Q * 2;      // [64 p][Q j] fp16, hi term
    uint8_t* sXl = sXw + kP * Q * 2;       // [64 p][Q j] fp16, lo term
    uint64_t* bar = reinterpret_cast<uint64_t*>(sXl + kP * Q * 2);
    uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 1);
    float* s_w = reinterpret_cast<float*>(slot + 4);  // [Q] weights

    const int c = blockIdx.x, hb = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h0 = hb * kHB;
    const int g = h0 / p.hpg;
    const int64_t tc0 = (int64_t)c * Q;

    if (warp == 0) {
        msc::tmem_alloc(slot, 64);
        msc::tmem_relinquish();
    }
    if (tid == 0) {
        msc::mbar_init(bar, 1);
        msc::fence_barrier_init();
    }
    // B^T of this chunk (shared by the group's heads): unit = (j, 8 consecutive n)
    for (int u = tid; u < Q * (kN / 8); u += 128) {
        const int j = u >> 4, n0 = (u & 15) * 8;
        const int64_t t = tc0 + j;
        uint4 raw = make_uint4(0, 0, 0, 0);
        if (t < p.L) raw = __ldg(reinterpret_cast<const uint4*>(p.B + (((int64_t)b * p.L + t) * p.G + g) * kN + n0));
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            *reinterpret_cast<uint16_t*>(sBt + msc::sw128_offset(n0 + 2 * e, j, kN)) = f2h_bits(msc::bf16lo(w[e]));
            *reinterpret_cast<uint16_t*>(sBt + msc::sw128_offset(n0 + 2 * e + 1, j, kN)) = f2h_bits(msc::bf16hi(w[e]));
        }
    }
    __syncthreads();
    const uint32_t tmem = *slot;
    const uint32_t idesc = msc::idesc_f16(false, 128, kP);
    bool ok = true;
    const int hend = min(h0 + kHB, p.H);
    for (int h = h0, it = 0; h < hend; ++h, ++it) {
        const size_t dbase = ((size_t)b * p.H + h) * p.Lp + (size_t)tc0;
        const float cs_last = p.cs[dbase + Q - 1];
        for (int j = tid; j < Q; j += 128) s_w[j] = msc::ex2_approx((cs_last - p.cs[dbase + j]) * MSC_LOG2E) * p.dt[dbase + j];
        __syncthreads();
        // Xw^T[p][j] = w_j x_j[p]: unit = (j, 8 consecutive p)
        for (int u = tid; u < Q * (kP / 8); u += 128) {
            const int j = u >> 3, p0 = (u & 7) * 8;
            const int64_t t = tc0 + j;
            uint4 raw = make_uint4(0, 0, 0, 0);
            if (t < p.L) raw = __ldg(reinterpret_cast<const uint4*>(p.x + (((int64_t)b * p.L + t) * p.H + h) * kP + p0));
            const float wj = s_w[j];
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
#pragma unroll
                for (int f = 0; f < 2; ++f) {
                    const float v = wj * (f ? msc::bf16hi(w[e]) : msc::bf16lo(w[e]));
                    const uint16_t hb = f2h_bits(v);
                    const uint32_t off = msc::sw128_offset(p0 + 2 * e + f, j, kP);
                    *reinterpret_cast<uint16_t*>(sXw + off) = hb;
                    *reinterpret_cast<uint16_t*>(sXl + off) = f2h_bits(v - h2f(hb));
                }
            }
        }
        msc::fence_proxy_async_smem();
        __syncthreads();
        msc::tc_fence_after();
        if (tid == 0) {
            for (int k = 0; k < Q / 16; ++k) {
                const uint32_t koff = (uint32_t)((k & 3) * 32);
                const uint64_t ad = msc::sdesc_sw128(msc::smem_u32(sBt + (k >> 2) * kN * 128) + koff);
                const uint64_t bh = msc::sdesc_sw128(msc::smem_u32(sXw + (k >> 2) * kP * 128) + koff);
                const uint64_t bl = msc::sdesc_sw128(msc::smem_u32(sXl + (k >> 2) * kP * 128) + koff);
                msc::mma_f16(tmem, ad, bh, idesc, k > 0 ? 1u : 0u);
                msc::mma_f16(tmem, ad, bl, idesc, 1u);
            }
            msc::mma_commit(bar);
        }
        const bool w_ok = wait_phase(bar, (uint32_t)(it & 1));
        if (__syncthreads_or(!w_ok)) {
            if (tid == 0) record_timeout(20);
            ok = false;
            break;
        }
        msc::tc_fence_after();
        // thread = state n (TMEM lane); 64 columns = p
        float* dst = p.S + ((((size_t)b * p.nc + c) * p.H + h) * kP) * kN + (32 * warp + lane);
#pragma unroll
        for (int c16 = 0; c16 < kP; c16 += 16) {
            float v[16];
            msc::tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)c16, v);
            msc::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) dst[(size_t)(c16 + i) * kN] = v[i];
        }
        msc::tc_fence_before();
        __syncthreads();
    }
    (void)ok;
    msc::tc_fence_before();
    __syncthreads();
    if (warp == 0) msc::tmem_dealloc(tmem, 64);
}

// ------------------------------------------------------------ (3) state pass
// One thread per (b, h, p, n): Hin of every chunk (fp16 tile images for the
// scan kernel's tensor cores) and the final state.
__global__ void __launch_bounds__(256) ssd_pass_kernel(const SsdParams p) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t total = (int64_t)gridDim.y * p.H * kP * kN;  // gridDim.y = batch
    (void)total;
    const int b = blockIdx.y;
    if (idx >= (int64_t)p.H * kP * kN) return;
    const int n = (int)(idx % kN);
    const int pp = (int)((idx / kN) % kP);
    const int h = (int)(idx / (kN * kP));
    float run = 0.f;
    const size_t dbase = ((size_t)b * p.H + h) * p.Lp;
    for (int c = 0; c < p.nc; ++c) {
        // hi image, then lo image (the rounding residual), 16 KB each
        uint8_t* tile = reinterpret_cast<uint8_t*>(p.Hin + (((size_t)b * p.nc + c) * p.H + h) * (2 * kP * kN));
        const uint16_t hb = f2h_bits(run);
        *reinterpret_cast<uint16_t*>(tile + msc::sw128_offset(pp, n, kP)) = hb;
        *reinterpret_cast<uint16_t*>(tile + kP * kN * 2 + msc::sw128_offset(pp, n, kP)) = f2h_bits(run - h2f(hb));
        const float decay = msc::ex2_approx(p.cs[dbase + (size_t)c * p.Q + p.Q - 1] * MSC_LOG2E);
        run = fmaf(decay, run, p.S[((((size_t)b * p.nc + c) * p.H + h) * kP + pp) * kN + n]);
    }
    if (p.final_state) p.final_state[(((size_t)b * p.H + h) * kP + pp) * kN + n] = run;
}

// ------------------------------------------------------------ (4) chunk scan
struct ScanMaps {
    CUtensorMap C, B;
};

// Releases the block's tensor memory (every thread calls it once, at the end).
__device__ __forceinline__ void scan_finish(uint32_t tmem, int warp) {
    msc::tc_fence_before();
    __syncthreads();
    if (warp == 0) msc::tmem_dealloc(tmem, 512);
}

// CTA = (chunk c, row block ib of 128 rows, head block, batch b); 256 threads.
// Warps w and w + 4 share TMEM lanes 32 (w % 4) .. (rows) and split columns.
__global__ void __launch_bounds__(256) ssd_scan_kernel(const __grid_constant__ CUtensorMap tmC,
                                                       const __grid_constant__ CUtensorMap tmB, const SsdParams p) {
    extern __shared__ uint8_t s_dyn[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(s_dyn) + 1023) & ~uintptr_t(1023));
    const int Q = p.Q;
    const int c = blockIdx.x / ((Q + 127) / 128), ib = blockIdx.x % ((Q + 127) / 128);
    const int hb = blockIdx.y, b = blockIdx.z;
    const int Qi = min(Q, (ib + 1) * 128);      // columns j of this row block: [0, Qi)
    const int rows_valid = min(128, Q - ib * 128);
    uint8_t* sC = base;                          // [128 i][128 n]  (2 x 16 KB)
    uint8_t* sBM = sC + 32768;                   // B [Q j][128 n] for G, then M'_hi [128 i][Qi j]
    uint8_t* sML = sBM + 65536;                  // M'_lo [128 i][Qi j]
    uint8_t* sXd = sML + 65536;                  // x [64 p][Qi j] fp16
    uint8_t* sH = sXd + 32768;                   // Hin [64 p][128 n] fp16: hi tile, then lo tile
    float* s_w = reinterpret_cast<float*>(sH + 32768);  // log2(Delta_j) - cs_j log2(e)
    uint64_t* bars = reinterpret_cast<uint64_t*>(s_w + 256);  // 0: loads, 1: G, 2: Hin, 3: head MMAs
    uint32_t* slot = reinterpret_cast<uint32_t*>(bars + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int i_loc = 32 * quarter + lane;        // row of this thread within the block
    const int i_chk = ib * 128 + i_loc;           // row within the chunk
    const int h0 = hb * kHB;
    const int g = h0 / p.hpg;
    const int64_t tc0 = (int64_t)c * Q;
    const uint32_t tG = 0, tYd = 256, tYo = 320;

    if (warp == 0) {
        msc::tmem_alloc(slot, 512);
        msc::tmem_relinquish();
    }
    if (tid == 0) {
        for (int k = 0; k < 4; ++k) msc::mbar_init(&bars[k], 1);
        msc::fence_barrier_init();
        msc::prefetch_tmap(&tmC);
        msc::prefetch_tmap(&tmB);
        // C rows of this block and B rows [0, Qi) of the chunk, 128-byte swizzled, K = n in 2 blocks
        // (the B box is Q rows: the G GEMM of this block uses its first Qi)
        const uint32_t bytes = 2u * 128u * 128u + 2u * (uint32_t)Q * 128u;
        msc::mbar_arrive_expect_tx(&bars[0], bytes);
        for (int kb = 0; kb < 2; ++kb) {
            msc::tma_load_3d(sC + kb * 16384, &tmC, &bars[0], g * kN + kb * 64, (int)(tc0 + ib * 128), b);
            msc::tma_load_3d(sBM + kb * Q * 128, &tmB, &bars[0], g * kN + kb * 64, (int)tc0, b);
        }
    }
    __syncthreads();
    const uint32_t tmem = *slot;
    bool ok = wait_phase(&bars[0], 0);
    if (__syncthreads_or(!ok)) {
        if (tid == 0) record_timeout(40);
        scan_finish(tmem, warp);
        return;
    }
    msc::tc_fence_after();
    // G = C B^T (M = 128, N = Qi, K = 128), bf16 operands
    if (tid == 0) {
        const uint32_t idesc = msc::idesc_f16(true, 128, Qi);
        for (int k = 0; k < 8; ++k) {
            const uint32_t koff = (uint32_t)((k & 3) * 32);
            const uint64_t ad = msc::sdesc_sw128(msc::smem_u32(sC + (k >> 2) * 16384) + koff);
            const uint64_t bd = msc::sdesc_sw128(msc::smem_u32(sBM + (k >> 2) * Q * 128) + koff);
            msc::mma_f16(tmem + tG, ad, bd, idesc, k > 0 ? 1u : 0u);
        }
        msc::mma_commit(&bars[1]);
    }
    ok = wait_phase(&bars[1], 0);
    if (__syncthreads_or(!ok)) {
        if (tid == 0) record_timeout(41);
        scan_finish(tmem, warp);
        return;
    }
    msc::tc_fence_after();
    // C tile bf16 -> fp16 in place (the swizzle is a pure permutation of 2-byte slots)
    for (int u = tid; u < 128 * 128 / 8; u += 256) {
        uint4* q = reinterpret_cast<uint4*>(sC) + u;
        uint4 v = *q;
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = msc::pack_half2(msc::bf16lo(w[e]), msc::bf16hi(w[e]));
        *q = make_uint4(w[0], w[1], w[2], w[3]);
    }

    {
        const int hend = min(h0 + kHB, p.H);
        for (int h = h0, it = 0; h < hend; ++h, ++it) {
            const uint32_t par = (uint32_t)(it & 1);
            if (tid == 0) {
                msc::mbar_arrive_expect_tx(&bars[2], 32768u);
                const uint16_t* src = p.Hin + (((size_t)b * p.nc + c) * p.H + h) * (2 * kP * kN);
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                        msc::smem_u32(sH)),
                    "l"(src), "r"(32768), "r"(msc::smem_u32(&bars[2]))
                    : "memory");
            }
            const size_t dbase = ((size_t)b * p.H + h) * p.Lp + (size_t)tc0;
            for (int j = tid; j < Qi; j += 256) {
                const float dtj = p.dt[dbase + j];
                s_w[j] = (dtj > 0.f ? __log2f(dtj) : -INFINITY) - p.cs[dbase + j] * MSC_LOG2E;
            }
            const float cs_i = p.cs[dbase + (i_chk < Qi ? i_chk : 0)];
            // x of the chunk, transposed to [p][j] fp16 (exact): unit = (j, 8 consecutive p)
            for (int u = tid; u < Qi * 8; u += 256) {
                const int j = u >> 3, p0 = (u & 7) * 8;
                const int64_t t = tc0 + j;
                uint4 v = make_uint4(0, 0, 0, 0);
                if (t < p.L) v = __ldg(reinterpret_cast<const uint4*>(p.x + (((int64_t)b * p.L + t) * p.H + h) * kP + p0));
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    *reinterpret_cast<uint16_t*>(sXd + msc::sw128_offset(p0 + 2 * e, j, kP)) = f2h_bits(msc::bf16lo(w[e]));
                    *reinterpret_cast<uint16_t*>(sXd + msc::sw128_offset(p0 + 2 * e + 1, j, kP)) = f2h_bits(msc::bf16hi(w[e]));
                }
            }
            __syncthreads();  // s_w complete
            // M'[i][j] = G[i][j] exp(cs_i - cs_j) Delta_j for j <= i, else 0, as fp16 hi + lo;
            // this thread: row i_loc, columns [half * Qi / 2, (half + 1) * Qi / 2)
            {
                const float csi = cs_i * MSC_LOG2E;
                const int j0 = half * (Qi / 2), j1 = j0 + Qi / 2;
                for (int jc = j0; jc < j1; jc += 16) {
                    float gv[16];
                    msc::tmem_ld16(tmem + tG + ((uint32_t)(32 * quarter) << 16) + (uint32_t)jc, gv);
                    msc::tmem_ld_wait();
                    uint32_t ph[8], pl[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int ja = jc + 2 * e, jb = ja + 1;
                        const float va = (ja <= i_chk) ? gv[2 * e] * msc::ex2_approx(csi + s_w[ja]) : 0.f;
                        const float vb = (jb <= i_chk) ? gv[2 * e + 1] * msc::ex2_approx(csi + s_w[jb]) : 0.f;
                        ph[e] = msc::pack_half2(va, vb);
                        const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&ph[e]));
                        pl[e] = msc::pack_half2(va - hf.x, vb - hf.y);
                    }
                    const uint32_t o0 = msc::sw128_offset(i_loc, jc, 128), o1 = msc::sw128_offset(i_loc, jc + 8, 128);
                    *reinterpret_cast<uint4*>(sBM + o0) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
                    *reinterpret_cast<uint4*>(sBM + o1) = make_uint4(ph[4], ph[5], ph[6], ph[7]);
                    *reinterpret_cast<uint4*>(sML + o0) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
                    *reinterpret_cast<uint4*>(sML + o1) = make_uint4(pl[4], pl[5], pl[6], pl[7]);
                }
            }
            ok = wait_phase(&bars[2], par);
            if (__syncthreads_or(!ok)) {
                if (tid == 0) record_timeout(42);
                break;
            }
            msc::fence_proxy_async_smem();
            msc::tc_fence_before();
            __syncthreads();
            msc::tc_fence_after();
            if (tid == 0) {
                const uint32_t id64 = msc::idesc_f16(false, 128, kP);
                for (int k = 0; k < Qi / 16; ++k) {
                    const uint32_t koff = (uint32_t)((k & 3) * 32);
                    const uint64_t bd = msc::sdesc_sw128(msc::smem_u32(sXd + (k >> 2) * kP * 128) + koff);
                    const uint64_t adh = msc::sdesc_sw128(msc::smem_u32(sBM + (k >> 2) * 16384) + koff);
                    const uint64_t adl = msc::sdesc_sw128(msc::smem_u32(sML + (k >> 2) * 16384) + koff);
                    msc::mma_f16(tmem + tYd, adh, bd, id64, k > 0 ? 1u : 0u);
                    msc::mma_f16(tmem + tYd, adl, bd, id64, 1u);
                }
                for (int k = 0; k < kN / 16; ++k) {
                    const uint32_t koff = (uint32_t)((k & 3) * 32);
                    const uint64_t ad = msc::sdesc_sw128(msc::smem_u32(sC + (k >> 2) * 16384) + koff);
                    const uint64_t bh = msc::sdesc_sw128(msc::smem_u32(sH + (k >> 2) * kP * 128) + koff);
                    const uint64_t bl = msc::sdesc_sw128(msc::smem_u32(sH + 16384 + (k >> 2) * kP * 128) + koff);
                    msc::mma_f16(tmem + tYo, ad, bh, id64, k > 0 ? 1u : 0u);
                    msc::mma_f16(tmem + tYo, ad, bl, id64, 1u);
                }
                msc::mma_commit(&bars[3]);
            }
            ok = wait_phase(&bars[3], par);
            if (__syncthreads_or(!ok)) {
                if (tid == 0) record_timeout(43);
                break;
            }
            msc::tc_fence_after();
            // epilogue: row i_loc, columns p in [32 half, 32 half + 32)
            {
                const int64_t t = tc0 + i_chk;
                const bool store = (i_loc < rows_valid) && (t < p.L);
                const float e_i = msc::ex2_approx(cs_i * MSC_LOG2E);
                const float Dh = p.D ? p.D[h] : 0.f;
                float* yrow = p.y + (((int64_t)b * p.L + t) * p.H + h) * kP;
                const uint16_t* zrow = p.z ? p.z + (((int64_t)b * p.L + t) * p.H + h) * kP : nullptr;
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int pc = 32 * half + 16 * cc;
                    float yd[16], yo[16];
                    msc::tmem_ld16(tmem + tYd + ((uint32_t)(32 * quarter) << 16) + (uint32_t)pc, yd);
                    msc::tmem_ld16(tmem + tYo + ((uint32_t)(32 * quarter) << 16) + (uint32_t)pc, yo);
                    msc::tmem_ld_wait();
                    if (store) {
                        const uint16_t* xrow = p.x + (((int64_t)b * p.L + t) * p.H + h) * kP;
                        const uint4 xv0 = __ldg(reinterpret_cast<const uint4*>(xrow + pc));
                        const uint4 xv1 = __ldg(reinterpret_cast<const uint4*>(xrow + pc + 8));
                        const uint32_t xw[8] = {xv0.x, xv0.y, xv0.z, xv0.w, xv1.x, xv1.y, xv1.z, xv1.w};
                        float out[16];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            out[2 * e] = fmaf(e_i, yo[2 * e], yd[2 * e]) + Dh * msc::bf16lo(xw[e]);
                            out[2 * e + 1] = fmaf(e_i, yo[2 * e + 1], yd[2 * e + 1]) + Dh * msc::bf16hi(xw[e]);
                        }
                        if (zrow) {
                            const uint4 zv0 = __ldg(reinterpret_cast<const uint4*>(zrow + pc));
                            const uint4 zv1 = __ldg(reinterpret_cast<const uint4*>(zrow + pc + 8));
                            const uint32_t zw[8] = {zv0.x, zv0.y, zv0.z, zv0.w, zv1.x, zv1.y, zv1.z, zv1.w};
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                out[2 * e] *= msc::silu_f(msc::bf16lo(zw[e]));
                                out[2 * e + 1] *= msc::silu_f(msc::bf16hi(zw[e]));
                            }
                        }
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            __stcs(reinterpret_cast<float4*>(yrow + pc) + e,
                                   make_float4(out[4 * e], out[4 * e + 1], out[4 * e + 2], out[4 * e + 3]));
                    }
                }
            }
            msc::tc_fence_before();
            __syncthreads();
        }
    }
    scan_finish(tmem, warp);
}

size_t a256(size_t x) { return (x + 255) / 256 * 256; }

constexpr int kScanSmem = 1024 + 32768 + 65536 + 65536 + 32768 + 32768 + 1024 + 64;

int state_smem(int Q) { return 1024 + kN * Q * 2 + 2 * kP * Q * 2 + 64 + Q * 4; }

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
    p.L = a.L; p.H = (int)a.H; p.G = (int)a.G; p.hpg = (int)(a.H / a.G); p.Q = (int)a.Q;
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
    // (2) chunk states
    {
        const int smem = state_smem(p.Q);
        static int configured = 0;
        if (configured < smem) {
            cudaError_t e = cudaFuncSetAttribute(ssd_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, state_smem(256));
            if (e != cudaSuccess) return fail(MSC_ERR_CUDA, "ssd_state smem attribute: %s", cudaGetErrorString(e));
            configured = smem;
        }
        ssd_state_kernel<<<dim3(p.nc, (p.H + kHB - 1) / kHB, (unsigned)a.batch), 128, smem, st>>>(p);
        if ((s = check_launch("ssd_state")) != MSC_OK) return s;
    }
    // (3) inter-chunk state pass
    {
        const int64_t per_b = (int64_t)p.H * kP * kN;
        ssd_pass_kernel<<<dim3((unsigned)((per_b + 255) / 256), (unsigned)a.batch), 256, 0, st>>>(p);
        if ((s = check_launch("ssd_pass")) != MSC_OK) return s;
    }
    // (4) chunk scan
    {
        ScanMaps m;
        const uint64_t bcd[3] = {(uint64_t)(a.G * kN), (uint64_t)a.L, (uint64_t)a.batch};
        const uint64_t bcs[2] = {(uint64_t)(a.G * kN * 2), (uint64_t)(a.L * a.G * kN * 2)};
        const uint32_t cbox[3] = {64, 128, 1};
        const uint32_t bbox[3] = {64, (uint32_t)(p.Q < 256 ? p.Q : 256), 1};
        const int nib = (p.Q + 127) / 128;
        // the B box is the whole chunk (Q rows); a row block uses its first Qi
        if (!encode_tmap(&m.C, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.C, bcd, bcs, cbox, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_tmap(&m.B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.B, bcd, bcs, bbox, CU_TENSOR_MAP_SWIZZLE_128B))
            return MSC_ERR_CUDA;
        static bool configured = false;
        if (!configured) {
            cudaError_t e = cudaFuncSetAttribute(ssd_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kScanSmem);
            if (e != cudaSuccess) return fail(MSC_ERR_CUDA, "ssd_scan smem attribute: %s", cudaGetErrorString(e));
            configured = true;
        }
        ssd_scan_kernel<<<dim3(p.nc * nib, (p.H + kHB - 1) / kHB, (unsigned)a.batch), 256, kScanSmem, st>>>(m.C, m.B, p);
        if ((s = check_launch("ssd_scan")) != MSC_OK) return s;
    }
    return MSC_OK;
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
