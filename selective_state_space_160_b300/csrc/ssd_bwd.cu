// ssd_bwd.cu -- Mamba-2 SSD chunked backward on sm_103a (tcgen05 for the large products).
//
// The pages give the SSD forward (bqwf survey sec. 3.2: scalar A_t = alpha_t I;
// "Mamba 解密" sec. 6.2: Y = M (X . B^T) C, M_ij = a_{j+1} ... a_i); the backward is
// derived by hand from the chunk decomposition the forward uses.  Per batch b,
// head h (group g), chunk c of Q steps, local steps i, j, with E_ij =
// exp(cs_i - cs_j), G_ij = C_i . B_j, w_j = exp(cs_last - cs_j) Delta_j, Hin the state
// entering the chunk and g_i = dy_i * silu(z_i) (dy_i without a gate):
//   forward:  y_i = sum_{j<=i} E_ij G_ij Delta_j x_j + exp(cs_i) Hin C_i + D x_i
//             Hin' = exp(cs_last) Hin + S,   S = sum_j w_j x_j (x) B_j
//   dz_i   = dy_i y_pre_i silu'(z_i),  dD = sum g.x
//   U_c    = sum_i exp(cs_i) g_i (x) C_i;   dH_c = U_c + exp(cs_last) dH_{c+1};   dS_c = dH_{c+1}
//   dx_j   = Delta_j sum_{i>=j} E_ij G_ij g_i + w_j dS B_j + D g_j
//   dG_ij  = sum_h E_ij Delta_j (g_i . x_j)     (heads of the group; j <= i)
//   dC_i   = sum_{j<=i} dG_ij B_j + sum_h exp(cs_i) Hin^T g_i
//   dB_j   = sum_{i>=j} dG_ij C_i + sum_h w_j dS^T x_j
//   dDelta_j = sum_{i>=j} E_ij G_ij (g_i . x_j) + exp(cs_last - cs_j) (x_j . dS B_j)
//   dcs_i += sum_{j<=i} T_ij,  dcs_j -= sum_{i>=j} T_ij   with T_ij = E_ij G_ij Delta_j (g_i . x_j)
//   dcs_i += exp(cs_i) g_i . (Hin C_i);   dcs_last += w_j dw_j, dcs_j -= w_j dw_j (dw_j = x_j . dS B_j);
//   dcs_last += exp(cs_last) <Hin, dH_{c+1}>
//   cs_i = A sum_{r<=i} Delta_r:  dDelta_r += A sum_{i>=r} dcs_i,  dA += sum_i dcs_i sum_{r<=i} Delta_r
//   ddelta = dDelta sigmoid(delta + bias),  dbias = sum ddelta.
// The oracle checks the same gradients through the S6 backward (its pins include
// finite differences of the SSD forward).
//
// Kernels (cross-head sums are accumulated inside one CTA per group; U, dG, dx
// and the state parts of dB, dC run on tcgen05 with fp32 operands split into
// bf16 hi + lo; G = C B^T and dC, dB from dG are 64-row tiles of fp32 FMAs
// staged through shared memory):
//   ssd_gmat_kernel     G = C B^T per (chunk, group), lower block triangle
//   ssd_ugrad           U_c per (chunk, head): the forward's chunk-state kernel on dy, C
//   ssd_rpass_kernel    reverse state pass: dS_c (bf16 hi + lo images), dcs_last
//   ssd_dg_tc_kernel    dG per (chunk, group, 128 x 128 tile) over its heads; dDelta, dcs of Y_diag
//   ssd_dbc_kernel      dC, dB from dG
//   ssd_dx_tc_kernel    dx, dz, dD per (chunk, head, 128 steps); dDelta, dcs of the state and Y_off terms
//   ssd_dbcs_tc_kernel  state parts of dB, dC per (chunk, group, 128 steps, 16 heads)
//   ssd_dcs_kernel      cs -> Delta, A; ddelta, dbias
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>

#include "msc_common.cuh"
#include "msc_internal.h"
#include "msc_tc.cuh"
#include "msc_tma.cuh"

namespace {

constexpr uint32_t kSleepNs = 20000;  // suspend hint of the blocks' mbarrier waits

constexpr int kP = 64;
constexpr int kN = 128;
constexpr int kT = 64;       // tile rows / steps per block
constexpr int kKS = 32;      // K slab of a tile product
constexpr int kHBlk = 16;    // heads per CTA of the cross-head state kernel

__device__ unsigned int g_ssdb_status[2];

__device__ __forceinline__ void record_timeout(unsigned int site) {
    if (atomicCAS(&g_ssdb_status[0], 0u, (unsigned int)MSC_ERR_TIMEOUT) == 0u) g_ssdb_status[1] = site;
}

struct SsdBwdParams {
    const uint16_t *x, *delta, *B, *C, *z, *dy;  // bf16
    const float *A, *D, *bias;
    const float* ypre;                           // [b, L, H, P] pre-gate output (z given)
    const float *dt, *cs;                        // [b, H, Lp]
    const float* Hin;                            // [b, nc, H, P, N]
    const float* U;                              // [b, nc, H, P, N]: U_c
    uint16_t* dSimg;                             // [b, nc, H] (hi, lo) bf16 images of dS_c, K-major [64 p][128 n] SW128
    const uint16_t* Himg;                        // the same images of Hin
    float *Gm, *dG;                              // [b, nc, Gr, Q, Q]
    float *dcs, *dDelta;                         // [b, H, Lp] accumulators
    float *dx, *ddelta, *dA, *dB, *dC, *dD, *dz, *dbias;
    int64_t L, Lp;
    int batch, H, Gr, hpg, Q, nc;
    int dg_hpb;                                  // heads per CTA of the dG kernel
};

__device__ __forceinline__ float bfv(uint16_t v) { return __uint_as_float(((uint32_t)v) << 16); }

// B or C of step t, group g, states n0 .. n0 + 7 (n0 a multiple of 8): one 16-byte load
__device__ __forceinline__ void bval8(const uint16_t* M, const SsdBwdParams& p, int b, int64_t t, int g, int n0,
                                      float* v) {
    if (t >= p.L) {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = 0.f;
        return;
    }
    const uint4 w = *reinterpret_cast<const uint4*>(M + (((size_t)b * p.L + t) * p.Gr + g) * kN + n0);
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        v[2 * e] = msc::bf16lo(ww[e]);
        v[2 * e + 1] = msc::bf16hi(ww[e]);
    }
}

// vector reduction into global memory (16-byte aligned)
__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// acc[r][c] += sum_{k < K} As[(ty * 4 + r) * lda + k] * Bs[k * ldb + tx * TC + c]:
// 256 threads make a 64 x (16 TC) tile, thread (ty, tx) = (tid / 16, tid % 16).
template <int TC>
__device__ __forceinline__ void tile_fma(const float* As, int lda, const float* Bs, int ldb, int K,
                                         float (&acc)[4][TC], int tid) {
    const int ty = tid >> 4, tx = tid & 15;
#pragma unroll 4
    for (int k = 0; k < K; ++k) {
        float a[4], bb[TC];
#pragma unroll
        for (int r = 0; r < 4; ++r) a[r] = As[(ty * 4 + r) * lda + k];
#pragma unroll
        for (int c = 0; c < TC; ++c) bb[c] = Bs[k * ldb + tx * TC + c];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < TC; ++c) acc[r][c] = fmaf(a[r], bb[c], acc[r][c]);
    }
}

template <int TC>
__device__ __forceinline__ void zero_acc(float (&acc)[4][TC]) {
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < TC; ++c) acc[r][c] = 0.f;
}

// ------------------------------------------------------------------ G = C B^T
// CTA = (64 x 64 tile (ib, jb) with jb <= ib, chunk, batch * Gr); K = N in slabs.
__global__ void __launch_bounds__(256) ssd_gmat_kernel(const SsdBwdParams p) {
    __shared__ float As[kT][kKS + 1];
    __shared__ float Bs[kKS][kT + 4];
    int ib = 0, rem = blockIdx.x;
    while (rem > ib) { rem -= ib + 1; ++ib; }
    const int jb = rem;
    const int c = blockIdx.y, b = blockIdx.z / p.Gr, g = blockIdx.z % p.Gr;
    const int tid = threadIdx.x;
    const int64_t t0 = (int64_t)c * p.Q;
    float acc[4][4];
    zero_acc(acc);
    for (int k0 = 0; k0 < kN; k0 += kKS) {
        {
            // 64 rows x 4 chunks of 8 states: one chunk of C and one of B per thread
            const int r = tid >> 2, ch = tid & 3;
            float vc[8], vb[8];
            bval8(p.C, p, b, t0 + ib * kT + r, g, k0 + 8 * ch, vc);
            bval8(p.B, p, b, t0 + jb * kT + r, g, k0 + 8 * ch, vb);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                As[r][8 * ch + e] = vc[e];
                Bs[8 * ch + e][r] = vb[e];
            }
        }
        __syncthreads();
        tile_fma<4>(&As[0][0], kKS + 1, &Bs[0][0], kT + 4, kKS, acc, tid);
        __syncthreads();
    }
    const int ty = tid >> 4, tx = tid & 15;
    float* dst = p.Gm + (((size_t)b * p.nc + c) * p.Gr + g) * p.Q * p.Q;
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
            dst[(size_t)(ib * kT + ty * 4 + r) * p.Q + jb * kT + tx * 4 + cc] = acc[r][cc];
}

// ------------------------------------------------------------------ reverse state pass
// Thread = (b, h, p, 8 consecutive n).  Walking chunks last to first: dS_c =
// dH_{c+1} (written as bf16 hi + lo tile images for the tensor cores),
// dH_c = U_c + exp(cs_last) dH_{c+1}, and dcs_last(c) += exp(cs_last) <Hin_c, dH_{c+1}>
// (a warp sum, then one atomic per warp).  U and Hin of four chunks are loaded
// ahead of the dependent chain.
constexpr int kRpAhead = 4;

__global__ void __launch_bounds__(256) ssd_rpass_kernel(const SsdBwdParams p) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int b = blockIdx.y;
    const int lane = threadIdx.x & 31;
    constexpr int kN8 = kN / 8;
    const int n0 = (int)(idx % kN8) * 8;
    const int pp = (int)((idx / kN8) % kP);
    const int h = (int)(idx / (kN8 * kP));
    const size_t dbase = ((size_t)b * p.H + h) * p.Lp;
    const uint32_t off = msc::sw128_offset(pp, n0, kP);
    float dh[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) dh[e] = 0.f;
    for (int ctop = p.nc - 1; ctop >= 0; ctop -= kRpAhead) {
        float4 uv[kRpAhead][2], hv[kRpAhead][2];
        float av[kRpAhead];
#pragma unroll
        for (int k = 0; k < kRpAhead; ++k) {
            const int c = ctop - k;
            if (c >= 0) {
                const size_t o = ((((size_t)b * p.nc + c) * p.H + h) * kP + pp) * kN + n0;
                const float4* u4 = reinterpret_cast<const float4*>(p.U + o);
                const float4* h4 = reinterpret_cast<const float4*>(p.Hin + o);
                uv[k][0] = __ldcs(u4);
                uv[k][1] = __ldcs(u4 + 1);
                hv[k][0] = __ldcs(h4);
                hv[k][1] = __ldcs(h4 + 1);
                av[k] = p.cs[dbase + (size_t)c * p.Q + p.Q - 1];
            }
        }
#pragma unroll
        for (int k = 0; k < kRpAhead; ++k) {
            const int c = ctop - k;
            if (c < 0) break;
            {
                uint8_t* tile = reinterpret_cast<uint8_t*>(p.dSimg) + (((size_t)b * p.nc + c) * p.H + h) * 32768;
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) msc::split_bf16x2(dh[2 * e], dh[2 * e + 1], hi[e], lo[e]);
                *reinterpret_cast<uint4*>(tile + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4*>(tile + 16384 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            const float a = msc::ex2_approx(av[k] * MSC_LOG2E);
            const float h8[8] = {hv[k][0].x, hv[k][0].y, hv[k][0].z, hv[k][0].w,
                                 hv[k][1].x, hv[k][1].y, hv[k][1].z, hv[k][1].w};
            const float u8[8] = {uv[k][0].x, uv[k][0].y, uv[k][0].z, uv[k][0].w,
                                 uv[k][1].x, uv[k][1].y, uv[k][1].z, uv[k][1].w};
            float part = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                part = fmaf(h8[e], dh[e], part);
                dh[e] = fmaf(a, dh[e], u8[e]);
            }
#pragma unroll
            for (int o2 = 16; o2 > 0; o2 >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o2);
            if (lane == 0 && part != 0.f) atomicAdd(p.dcs + dbase + (size_t)c * p.Q + p.Q - 1, a * part);
        }
    }
}

// ------------------------------------------------------------------ dG on tcgen05
// CTA = (128 x 128 tile (ib, jb) with jb <= ib, and a block of the group's heads;
// chunk; batch * Gr).  Per head the tensor cores form R = g_I x_J^T (M = 128
// steps i, N = 128 steps j, K = P; g is dy, or dy silu(z) split hi + lo) into one
// of two tensor-memory buffers; the CUDA cores then take, per element with i >= j,
//   er = E_ij R_ij,  dG_ij += er Delta_j,  p1 = er G_ij,
//   dcs_i += sum_j Delta_j p1,  dDelta_j += sum_i p1,  dcs_j -= Delta_j sum_i p1,
// with the dG accumulators in registers (thread = row i, 32 columns j; 16
// warps) and G in shared memory, while the MMAs of the next head run.  Column sums: a butterfly
// over the 32 lanes of a warp, then the four row quarters through shared memory.
// The head blocks of a tile add their dG with vector reductions (dG starts at 0).
constexpr int kDgStages = 3;
constexpr uint32_t kDgStage = 49152;           // A hi [128][64] | A lo (z) | B = x [128][64]
constexpr int kDgOpWarps = 16;
constexpr int kDgWarpLoad = kDgOpWarps, kDgWarpMma = kDgOpWarps + 1;
constexpr int kDgThreads = (kDgOpWarps + 2) * 32;
constexpr int kDgGld = 132;                    // row stride (floats) of the G tile: 16-byte rows
constexpr size_t kDgSmem = 1024 + kDgStages * kDgStage + (3 * 128 * 3 + 2 * (4 * 4 * 32 + 4 * 128) + 128 * kDgGld) * 4 + 20 * 8 + 16;

// v[0..15] of every lane -> sum over the warp's 32 lanes of v[lane >> 1]
__device__ __forceinline__ float warp_colsum16(float (&v)[16], int lane) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const bool up = lane & 16;
        const float send = up ? v[c] : v[c + 8];
        const float keep = up ? v[c + 8] : v[c];
        v[c] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const bool up = lane & 8;
        const float send = up ? v[c] : v[c + 4];
        const float keep = up ? v[c + 4] : v[c];
        v[c] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const bool up = lane & 4;
        const float send = up ? v[c] : v[c + 2];
        const float keep = up ? v[c + 2] : v[c];
        v[c] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    {
        const bool up = lane & 2;
        const float send = up ? v[0] : v[1];
        const float keep = up ? v[1] : v[0];
        v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
    }
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

__global__ void __launch_bounds__(kDgThreads, 1) ssd_dg_tc_kernel(const __grid_constant__ CUtensorMap tmX,
                                                                  const __grid_constant__ CUtensorMap tmDy,
                                                                  const __grid_constant__ CUtensorMap tmZ,
                                                                  const SsdBwdParams p) {
    extern __shared__ uint8_t s_dyn[];
    uint8_t* stages = s_dyn + ((1024u - (msc::smem_u32(s_dyn) & 1023u)) & 1023u);
    // cs of the tile's rows i and columns j and Delta of its columns, per head, in
    // a ring of three (bulk copies with the head's tiles)
    float* s_ci = reinterpret_cast<float*>(stages + kDgStages * kDgStage);  // [3][128]
    float* s_cj = s_ci + 384;                                              // [3][128]
    float* s_dj = s_cj + 384;                                              // [3][128]
    // column and row sums exchanged between warps, by head parity (a buffer is
    // rewritten two heads later, after every warp has passed the barrier between)
    float* s_col = s_dj + 384;                                             // [2][4 col quarters][4 row quarters][32]
    float* s_row = s_col + 1024;                                           // [2][4 col quarters][128]
    float* s_G = s_row + 1024;                                             // [128 i][kDgGld] G of the tile
    uint64_t* bars = reinterpret_cast<uint64_t*>(s_G + 128 * kDgGld);
    // 0-2 stage loaded, 3-5 stage built, 6-8 stage free, 9-10 R ready, 11-12 R read, 13 drain,
    // 14-16 the head's cs / Delta rows read
    uint64_t *tfull = bars, *full = bars + 3, *empty = bars + 6, *rfull = bars + 9, *rfree = bars + 11,
             *drain = bars + 13, *cfree = bars + 14;
    uint32_t* slot = reinterpret_cast<uint32_t*>(bars + 17);
    volatile uint32_t* abort = slot + 1;

    const int Q = p.Q;
    const int nhb = (p.hpg + p.dg_hpb - 1) / p.dg_hpb;
    const int tile = blockIdx.x / nhb, hb = blockIdx.x % nhb;
    int ib = 0, rem = tile;
    while (rem > ib) { rem -= ib + 1; ++ib; }
    const int jb = rem;
    const int c = blockIdx.y, b = blockIdx.z / p.Gr, g = blockIdx.z % p.Gr;
    const int rv = min(128, Q);                  // valid rows / columns of a tile (Q = 64: half)
    const int hh0 = hb * p.dg_hpb;
    const int nh = min(p.dg_hpb, p.hpg - hh0);
    const int64_t tc0 = (int64_t)c * Q;
    const bool has_z = p.z != nullptr;
    const bool diag_tile = ib == jb;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (warp == 0) {
        msc::tmem_alloc(slot, 256);
        msc::tmem_relinquish();
    }
    if (tid == 32) {
        for (int k = 0; k < kDgStages; ++k) {
            msc::mbar_init(&tfull[k], 1);
            msc::mbar_init(&full[k], kDgOpWarps);
            msc::mbar_init(&empty[k], 1);
        }
        for (int k = 0; k < 2; ++k) {
            msc::mbar_init(&rfull[k], 1);
            msc::mbar_init(&rfree[k], kDgOpWarps);
        }
        for (int k = 0; k < 3; ++k) msc::mbar_init(&cfree[k], kDgOpWarps);
        msc::mbar_init(drain, 1);
        slot[1] = 0u;
        msc::fence_barrier_init();
    }
    for (int e = tid; e < 3 * 384; e += kDgThreads) s_ci[e] = 0.f;  // rows past a short chunk stay 0
    msc::tc_fence_before();
    __syncthreads();
    msc::tc_fence_after();
    const uint32_t tmem = *slot;

    if (warp == kDgWarpLoad) {
        if (lane == 0) {
            msc::prefetch_tmap(&tmX);
            msc::prefetch_tmap(&tmDy);
            if (has_z) msc::prefetch_tmap(&tmZ);
            int issued = 0;
            for (int hh = 0; hh < nh; ++hh) {
                const int st = hh % kDgStages, use = hh / kDgStages;
                if (use > 0 && !(msc::wait_bounded(&empty[st], (uint32_t)((use - 1) & 1), abort, kSleepNs) &&
                                 msc::wait_bounded(&cfree[st], (uint32_t)((use - 1) & 1), abort, kSleepNs))) {
                    record_timeout(121);
                    *abort = 1u;
                    break;
                }
                const int h = g * p.hpg + hh0 + hh;
                const size_t dbase = ((size_t)b * p.H + h) * p.Lp + (size_t)tc0;
                uint8_t* sg = stages + st * kDgStage;
                const uint32_t rb4 = 4u * (uint32_t)rv;
                msc::mbar_arrive_expect_tx(&tfull[st], (has_z ? 49152u : 32768u) + 3u * rb4);
                msc::bulk_g2s(s_ci + 128 * st, p.cs + dbase + 128 * ib, rb4, &tfull[st]);
                msc::bulk_g2s(s_cj + 128 * st, p.cs + dbase + 128 * jb, rb4, &tfull[st]);
                msc::bulk_g2s(s_dj + 128 * st, p.dt + dbase + 128 * jb, rb4, &tfull[st]);
                msc::tma_load_3d(sg, &tmDy, &tfull[st], h * kP, (int)(tc0 + 128 * ib), b);
                if (has_z) msc::tma_load_3d(sg + 16384, &tmZ, &tfull[st], h * kP, (int)(tc0 + 128 * ib), b);
                msc::tma_load_3d(sg + 32768, &tmX, &tfull[st], h * kP, (int)(tc0 + 128 * jb), b);
                ++issued;
            }
            for (int st = 0; st < kDgStages && st < issued; ++st)
                if (!msc::wait_bounded(&tfull[st], (uint32_t)(((issued - 1 - st) / kDgStages) & 1), nullptr, kSleepNs)) record_timeout(122);
        }
        __syncwarp();
    } else if (warp == kDgWarpMma) {
        if (lane == 0) {
            const uint32_t idK = msc::idesc_f16(true, 128, 128);
            bool ok = true;
            for (int hh = 0; hh < nh && ok; ++hh) {
                const int st = hh % kDgStages, use = hh / kDgStages, rb = hh & 1;
                ok = msc::wait_bounded(&tfull[st], (uint32_t)(use & 1), abort, kSleepNs) &&
                     msc::wait_bounded(&full[st], (uint32_t)(use & 1), abort, kSleepNs);
                if (ok && hh >= 2) ok = msc::wait_bounded(&rfree[rb], (uint32_t)(((hh - 2) >> 1) & 1), abort, kSleepNs);
                if (!ok) break;
                msc::tc_fence_after();
                const uint32_t a = msc::smem_u32(stages + st * kDgStage);
                const uint32_t acc = tmem + 128u * (uint32_t)rb;
                for (int k = 0; k < 4; ++k) {
                    const uint64_t bd = msc::sdesc_sw128(a + 32768 + 32 * k);
                    msc::mma_f16(acc, msc::sdesc_sw128(a + 32 * k), bd, idK, k ? 1u : 0u);
                    if (has_z) msc::mma_f16(acc, msc::sdesc_sw128(a + 16384 + 32 * k), bd, idK, 1u);
                }
                msc::mma_commit(&empty[st]);
                msc::mma_commit(&rfull[rb]);
            }
            if (!ok) {
                record_timeout(123);
                *abort = 1u;
            }
            msc::mma_commit(drain);
            if (!msc::wait_bounded(drain, 0, nullptr, kSleepNs)) record_timeout(124);
        }
        __syncwarp();
    } else {
        const int lq = warp & 3, cq = warp >> 2;     // row quarter (TMEM lanes), column quarter
        const int row = 32 * lq + lane;              // i within the tile
        const int il = 128 * ib + row;               // i within the chunk
        const bool row_ok = row < rv;
        const float* Gt = p.Gm + (((size_t)b * p.nc + c) * p.Gr + g) * (size_t)Q * Q;
        float dgacc[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) dgacc[k] = 0.f;
        // G of the tile (entries above the diagonal are never used: set to 0)
#pragma unroll 4
        for (int e = tid; e < 128 * 128; e += 32 * kDgOpWarps) {
            const int r = e >> 7, jj = e & 127;
            const int ir = 128 * ib + r;
            s_G[r * kDgGld + jj] = (r < rv && jj < rv && ir >= 128 * jb + jj) ? Gt[(size_t)ir * Q + 128 * jb + jj] : 0.f;
        }
        asm volatile("bar.sync 1, 512;" ::: "memory");
        bool ok = true;
        auto produce = [&](int hh) {
            const int st = hh % kDgStages, use = hh / kDgStages;
            if (has_z) {
                ok = ok && __all_sync(0xffffffffu, msc::wait_bounded(&tfull[st], (uint32_t)(use & 1), abort, kSleepNs));
                if (ok) {
                    uint8_t* sg = stages + st * kDgStage;
#pragma unroll 1
                    for (int u = tid; u < 1024; u += 32 * kDgOpWarps) {
                        uint4* ph = reinterpret_cast<uint4*>(sg + 16 * u);
                        uint4* pl = reinterpret_cast<uint4*>(sg + 16384 + 16 * u);
                        const uint4 dv = *ph, zv = *pl;
                        const uint32_t dw[4] = {dv.x, dv.y, dv.z, dv.w}, zw[4] = {zv.x, zv.y, zv.z, zv.w};
                        uint32_t hi[4], lo[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            msc::split_bf16x2(msc::bf16lo(dw[q]) * msc::silu_f(msc::bf16lo(zw[q])),
                                              msc::bf16hi(dw[q]) * msc::silu_f(msc::bf16hi(zw[q])), hi[q], lo[q]);
                        *ph = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                        *pl = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    }
                    msc::fence_proxy_async_smem();
                }
            }
            __syncwarp();
            if (lane == 0) msc::mbar_arrive(&full[st]);
        };
        auto epilogue = [&](int hh) {
            const int buf = hh & 1, cb = hh % 3;
            const int h = g * p.hpg + hh0 + hh;
            const size_t dbase = ((size_t)b * p.H + h) * p.Lp + (size_t)tc0;
            float* s_colh = s_col + 512 * buf;
            float* s_rowh = s_row + 512 * buf;
            ok = ok && __all_sync(0xffffffffu, msc::wait_bounded(&rfull[buf], (uint32_t)((hh >> 1) & 1), abort, kSleepNs) &&
                                                   msc::wait_bounded(&tfull[cb], (uint32_t)((hh / 3) & 1), abort, kSleepNs));
            msc::tc_fence_after();
            // the diagonal T_ii would enter dcs_i once as +T and once as -T: it is
            // left out of both sums (exactly zero), which keeps the large diagonal
            // terms of a fast-decaying chunk from cancelling in fp32; its dDelta
            // share goes in separately
            float rowt = 0.f, pdiag = 0.f;
            const float csi = s_ci[128 * cb + row];
            const float* cjp = s_cj + 128 * cb;
            const float* djp = s_dj + 128 * cb;
            const float* gp = s_G + row * kDgGld;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int c0 = 32 * cq + 16 * q;
                // warp-uniform: every element of the chunk lies above the diagonal or
                // outside a short chunk
                const bool skip = (diag_tile && c0 > 32 * lq + 31) || c0 >= rv || 32 * lq >= rv;
                float cs_ = 0.f;
                if (!skip) {
                    float r[16], col[16];
                    if (ok) {
                        msc::tmem_ld16(tmem + 128u * (uint32_t)buf + ((uint32_t)(32 * lq) << 16) + (uint32_t)c0, r);
                        msc::tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) r[e] = 0.f;
                    }
                    // warp-uniform: every row of the warp lies below every column of the
                    // chunk (no mask, no diagonal element): two columns per packed op
                    const bool dense = (!diag_tile || c0 + 15 < 32 * lq) && rv == 128;
                    if (dense) {
                        const uint64_t csi2 = msc::pk2(csi, csi);
                        uint64_t rowt2 = 0ull;
#pragma unroll
                        for (int e4 = 0; e4 < 4; ++e4) {
                            const ulonglong2 cj4 = *reinterpret_cast<const ulonglong2*>(cjp + c0 + 4 * e4);
                            const ulonglong2 dj4 = *reinterpret_cast<const ulonglong2*>(djp + c0 + 4 * e4);
                            const ulonglong2 g4 = *reinterpret_cast<const ulonglong2*>(gp + c0 + 4 * e4);
#pragma unroll
                            for (int tp = 0; tp < 2; ++tp) {
                                const int e = 4 * e4 + 2 * tp, k = 16 * q + e;
                                const uint64_t cj2 = tp ? cj4.y : cj4.x, dj2 = tp ? dj4.y : dj4.x;
                                const uint64_t g2 = tp ? g4.y : g4.x;
                                // the difference first (exact), then the scale
                                const uint64_t diff2 = msc::fma2(cj2, msc::pk2(-1.f, -1.f), csi2);
                                const uint64_t e2 = msc::ex2_2(msc::mul2(diff2, msc::pk2(MSC_LOG2E, MSC_LOG2E)));
                                const uint64_t er2 = msc::mul2(e2, msc::pk2(r[e], r[e + 1]));
                                uint64_t dg2 = msc::fma2(er2, dj2, msc::pk2(dgacc[k], dgacc[k + 1]));
                                msc::upk2(dg2, dgacc[k], dgacc[k + 1]);
                                const uint64_t p12 = msc::mul2(er2, g2);
                                rowt2 = msc::fma2(p12, dj2, rowt2);
                                msc::upk2(p12, col[e], col[e + 1]);
                            }
                        }
                        float ra, rb;
                        msc::upk2(rowt2, ra, rb);
                        rowt += ra + rb;
                    } else {
#pragma unroll
                    for (int e4 = 0; e4 < 4; ++e4) {
                        const float4 cj4 = *reinterpret_cast<const float4*>(cjp + c0 + 4 * e4);
                        const float4 dj4 = *reinterpret_cast<const float4*>(djp + c0 + 4 * e4);
                        const float4 g4 = *reinterpret_cast<const float4*>(gp + c0 + 4 * e4);
                        const float cj[4] = {cj4.x, cj4.y, cj4.z, cj4.w};
                        const float dj[4] = {dj4.x, dj4.y, dj4.z, dj4.w};
                        const float gv[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const int e = 4 * e4 + t, jj = c0 + e;
                            const bool m = row_ok && jj < rv && (!diag_tile || row >= jj);
                            // the difference first: |cs| reaches thousands in a fast-decaying chunk
                            const float er = m ? msc::ex2_approx((csi - cj[t]) * MSC_LOG2E) * r[e] : 0.f;
                            dgacc[16 * q + e] = fmaf(er, dj[t], dgacc[16 * q + e]);
                            const float p1 = er * gv[t];
                            const bool dg_ = diag_tile && row == jj;
                            rowt = dg_ ? rowt : fmaf(p1, dj[t], rowt);
                            col[e] = dg_ ? 0.f : p1;
                            pdiag = dg_ ? p1 : pdiag;
                        }
                    }
                    }
                    cs_ = warp_colsum16(col, lane);
                }
                if ((lane & 1) == 0) s_colh[128 * cq + 32 * lq + 16 * q + (lane >> 1)] = cs_;
            }
            msc::tc_fence_before();
            __syncwarp();
            if (lane == 0) msc::mbar_arrive(&rfree[buf]);
            if (pdiag != 0.f) atomicAdd(p.dDelta + dbase + il, pdiag);
            s_rowh[128 * cq + row] = rowt;
            asm volatile("bar.sync 1, 512;" ::: "memory");
            if (tid < 128) {
                const int jj = tid, cf = jj >> 5, k = jj & 31;
                const float cd = s_colh[128 * cf + k] + s_colh[128 * cf + 32 + k] + s_colh[128 * cf + 64 + k] +
                                 s_colh[128 * cf + 96 + k];
                if (jj < rv && cd != 0.f) {
                    atomicAdd(p.dDelta + dbase + 128 * jb + jj, cd);
                    atomicAdd(p.dcs + dbase + 128 * jb + jj, -djp[jj] * cd);
                }
            } else if (tid < 256) {
                const int r2 = tid - 128;
                const float rt = s_rowh[r2] + s_rowh[128 + r2] + s_rowh[256 + r2] + s_rowh[384 + r2];
                if (r2 < rv && rt != 0.f) atomicAdd(p.dcs + dbase + 128 * ib + r2, rt);
            }
            __syncwarp();
            if (lane == 0) msc::mbar_arrive(&cfree[cb]);
        };
        for (int hh = 0; hh <= nh; ++hh) {
            if (hh < nh) produce(hh);
            if (hh >= 1) epilogue(hh - 1);
        }
        if (!ok) {
            if (lane == 0) record_timeout(125);
            *abort = 1u;
        }
        if (row_ok && 32 * cq < rv) {
            float* dst = p.dG + (((size_t)b * p.nc + c) * p.Gr + g) * (size_t)Q * Q + (size_t)il * Q + 128 * jb + 32 * cq;
#pragma unroll
            for (int k = 0; k < 32; k += 4) red_add_v4(dst + k, dgacc[k], dgacc[k + 1], dgacc[k + 2], dgacc[k + 3]);
        }
        msc::tc_fence_before();
    }
    __syncthreads();
    if (warp == 0) {
        msc::tc_fence_after();
        msc::tmem_dealloc(tmem, 256);
    }
}

// ------------------------------------------------------------------ dC, dB from dG
// CTA = (row block kb and side, chunk, batch * Gr); side 0: dC_I = sum_{J <= I} dG_IJ B_J,
// side 1: dB_J = sum_{I >= J} dG_IJ^T C_I; 64 x 128 tile, K = 64 per partner block.
// Stores (later kernels add the state parts with atomics).
__global__ void __launch_bounds__(256) ssd_dbc_kernel(const SsdBwdParams p) {
    __shared__ float As[kT][kT + 1];
    __shared__ float Bs[kKS][kN + 4];
    const int nb = p.Q / kT;
    const int kb = blockIdx.x % nb, side = blockIdx.x / nb;
    const int c = blockIdx.y, b = blockIdx.z / p.Gr, g = blockIdx.z % p.Gr;
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    const int64_t t0 = (int64_t)c * p.Q;
    const float* dGt = p.dG + (((size_t)b * p.nc + c) * p.Gr + g) * p.Q * p.Q;
    float acc[4][8];
    zero_acc(acc);
    const int lo = side ? kb : 0, hi = side ? nb - 1 : kb;
    for (int ob = lo; ob <= hi; ++ob) {
        // As[r][k]: side 0 dG[kb*64 + r][ob*64 + k]; side 1 dG[ob*64 + k][kb*64 + r]
        for (int e = tid; e < kT * kT; e += 256) {
            const int r = e / kT, k = e % kT;
            if (side == 0)
                As[r][k] = dGt[(size_t)(kb * kT + r) * p.Q + ob * kT + k];
            else
                As[k][r] = dGt[(size_t)(ob * kT + r) * p.Q + kb * kT + k];
        }
        for (int k0 = 0; k0 < kT; k0 += kKS) {
#pragma unroll
            for (int e = tid; e < kKS * kN / 8; e += 256) {  // 32 rows x 16 chunks of 8 states
                const int k = e >> 4, ch = e & 15;
                float v[8];
                bval8(side ? p.C : p.B, p, b, t0 + ob * kT + k0 + k, g, 8 * ch, v);
                *reinterpret_cast<float4*>(&Bs[k][8 * ch]) = make_float4(v[0], v[1], v[2], v[3]);
                *reinterpret_cast<float4*>(&Bs[k][8 * ch + 4]) = make_float4(v[4], v[5], v[6], v[7]);
            }
            __syncthreads();
            tile_fma<8>(&As[0][k0], kT + 1, &Bs[0][0], kN + 4, kKS, acc, tid);
            __syncthreads();
        }
    }
    float* dst = side ? p.dB : p.dC;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int64_t t = t0 + kb * kT + ty * 4 + r;
        if (t >= p.L) continue;
        float4* q = reinterpret_cast<float4*>(dst + (((size_t)b * p.L + t) * p.Gr + g) * kN + tx * 8);
        q[0] = make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
        q[1] = make_float4(acc[r][4], acc[r][5], acc[r][6], acc[r][7]);
    }
}

// ------------------------------------------------------------------ dx on tcgen05
// CTA = (chunk * nmb + row block mb of 128 steps j, block of kDxHB heads, batch),
// persistent over its heads: 16 operand / epilogue warps, one load warp, one MMA
// warp (the chunk length is a template parameter, so that the strided shared
// memory reads take immediate offsets).  Per head three accumulators in tensor
// memory (two buffers, so that the epilogue of one head runs while the MMAs of
// the next do), M = 128 rows j, N = 64 channels p, all fp32:
//   acc1 = sum_{i >= j} (E_ij G_ij) g_i[p]  A: E o G formed by CUDA cores, split hi + lo;
//                                          B: g tile [64 i][64 p], MN-major (dy itself, or
//                                          dy silu(z) split hi + lo)
//   acc2 = B_j . dS[p, :]                  A: B tile by TMA (exact bf16); B: dS hi, lo images
//   acc3 = C_j . Hin[p, :]                 A: C tile by TMA; B: Hin hi, lo images
// The operands stream through a ring of two 80 KB stages, one K slab of 64
// each: A hi [128][64] | A lo | B hi [64][64] | B lo (bf16, 128-byte swizzle) |
// G [64 i][128 j] (fp32, by TMA, read by the CUDA cores forming A).  Per head the
// first na slabs feed acc1, one per 64 steps i >= j0, then four by TMA: acc2
// (n blocks 0, 1), acc3 (n blocks 0, 1).  The head's cs and Delta rows come by
// bulk copy into a ring of three.
// Epilogue (thread = row j, a quarter of the p columns):
//   dx_j = Delta_j acc1 + w_j acc2 + D g_j;  dw_j = x_j . acc2;  v_j = exp(cs_j) g_j . acc3
// and, since it reads dy, x and z of the row anyway, the gate's dz and dD.
constexpr int kDxStages = 2;
constexpr uint32_t kDxStage = 81920;           // A hi | A lo | B hi | B lo | G [64 i][128 j] fp32
constexpr int kDxOpWarps = 16;
constexpr int kDxWarpLoad = kDxOpWarps, kDxWarpMma = kDxOpWarps + 1;
constexpr int kDxThreads = (kDxOpWarps + 2) * 32;
constexpr int kDxHB = 8;                       // heads per CTA
constexpr uint32_t kDxEpi = 32768;             // the epilogue's dy and x tiles [128 j][64 p] (no gate)
constexpr size_t kDxSmem = 1024 + kDxStages * kDxStage + kDxEpi + (3 * 512 + 1024) * 4 + 24 * 8 + 16;

template <int kQ, bool kZ>
__global__ void __launch_bounds__(kDxThreads, 1) ssd_dx_tc_kernel(const __grid_constant__ CUtensorMap tmB,
                                                                  const __grid_constant__ CUtensorMap tmC,
                                                                  const __grid_constant__ CUtensorMap tmDy,
                                                                  const __grid_constant__ CUtensorMap tmZ,
                                                                  const __grid_constant__ CUtensorMap tmG,
                                                                  const __grid_constant__ CUtensorMap tmDyE,
                                                                  const __grid_constant__ CUtensorMap tmXE,
                                                                  const SsdBwdParams p) {
    extern __shared__ uint8_t s_dyn[];
    uint8_t* stages = s_dyn + ((1024u - (msc::smem_u32(s_dyn) & 1023u)) & 1023u);
    uint8_t* s_epi = stages + kDxStages * kDxStage;                            // dy | x tiles of the head
    float* s_rows = reinterpret_cast<float*>(s_epi + kDxEpi);                  // [3][cs 256 | Delta 256]
    float* s_part = s_rows + 3 * 512;                                          // [dw, v][4 quarters][128 rows]
    uint64_t* bars = reinterpret_cast<uint64_t*>(s_part + 1024);
    // 0-1 stage loaded (TMA), 2-3 stage built (16 warps), 4-5 stage free (MMA), 6-8 rows loaded,
    // 9-11 rows free (16 warps), 12-13 accumulators ready, 14-15 accumulators free (16 warps), 16 drain,
    // 17 epilogue tiles loaded, 18 epilogue tiles read (16 warps)
    uint64_t *tfull = bars, *full = bars + 2, *empty = bars + 4, *rfull = bars + 6, *rfree = bars + 9,
             *afull = bars + 12, *afree = bars + 14, *drain = bars + 16, *efull = bars + 17, *efree = bars + 18;
    uint32_t* slot = reinterpret_cast<uint32_t*>(bars + 19);
    volatile uint32_t* abort = slot + 1;

    constexpr int Q = kQ;
    constexpr int nmb = (Q + 127) / 128;
    constexpr int kGW = Q < 128 ? Q : 128;       // columns j of a G slab
    const int c = blockIdx.x / nmb, mb = blockIdx.x % nmb;
    const int hb = blockIdx.y, b = blockIdx.z;
    const int j0 = 128 * mb;
    const int rows_valid = min(128, Q - j0);
    const int na = (Q - j0) / 64;                // acc1 slabs per head
    const int ns = na + 4;                       // slabs per head
    const int nh = min(kDxHB, p.H - hb * kDxHB);
    const int64_t tc0 = (int64_t)c * Q;
    constexpr bool has_z = kZ;  // a gate: g = dy silu(z), dz
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (warp == 0) {
        msc::tmem_alloc(slot, 512);
        msc::tmem_relinquish();
    }
    if (tid == 32) {
        for (int k = 0; k < kDxStages; ++k) {
            msc::mbar_init(&tfull[k], 1);
            msc::mbar_init(&full[k], kDxOpWarps);
            msc::mbar_init(&empty[k], 1);
        }
        for (int k = 0; k < 3; ++k) {
            msc::mbar_init(&rfull[k], 1);
            msc::mbar_init(&rfree[k], kDxOpWarps);
        }
        for (int k = 0; k < 2; ++k) {
            msc::mbar_init(&afull[k], 1);
            msc::mbar_init(&afree[k], kDxOpWarps);
        }
        msc::mbar_init(drain, 1);
        msc::mbar_init(efull, 1);
        msc::mbar_init(efree, kDxOpWarps);
        slot[1] = 0u;
        msc::fence_barrier_init();
    }
    msc::tc_fence_before();
    __syncthreads();
    msc::tc_fence_after();
    const uint32_t tmem = *slot;

    if (warp == kDxWarpLoad) {
        // ------------------------------------------------------------ loads
        if (lane == 0) {
            msc::prefetch_tmap(&tmB);
            msc::prefetch_tmap(&tmC);
            msc::prefetch_tmap(&tmDy);
            msc::prefetch_tmap(&tmG);
            if (has_z) msc::prefetch_tmap(&tmZ);
            else {
                msc::prefetch_tmap(&tmDyE);
                msc::prefetch_tmap(&tmXE);
            }
            int issued = 0, rissued = 0, eissued = 0;
            bool ok = true;
            for (int hh = 0; hh < nh && ok; ++hh) {
                const int h = hb * kDxHB + hh, g = h / p.hpg;
                const size_t dbase = ((size_t)b * p.H + h) * p.Lp + (size_t)tc0;
                const size_t img = (((size_t)b * p.nc + c) * p.H + h) * 32768;
                const int grow = ((b * p.nc + c) * p.Gr + g) * Q;  // first row of the chunk's G (2-D view)
                const int rb = hh % 3;
                if (hh >= 3 && !msc::wait_bounded(&rfree[rb], (uint32_t)(((hh - 3) / 3) & 1), abort, kSleepNs)) {
                    ok = false;
                    break;
                }
                msc::mbar_arrive_expect_tx(&rfull[rb], 8u * (uint32_t)Q);
                msc::bulk_g2s(s_rows + 512 * rb, p.cs + dbase, 4u * (uint32_t)Q, &rfull[rb]);
                msc::bulk_g2s(s_rows + 512 * rb + 256, p.dt + dbase, 4u * (uint32_t)Q, &rfull[rb]);
                ++rissued;
                for (int s = 0; s < ns; ++s) {
                    const int u = hh * ns + s, st = u % kDxStages, use = u / kDxStages;
                    if (use > 0 && !msc::wait_bounded(&empty[st], (uint32_t)((use - 1) & 1), abort, kSleepNs)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sg = stages + st * kDxStage;
                    if (s >= na) {
                        const int which = (s - na) >> 1, kb = (s - na) & 1;
                        const uint8_t* im = reinterpret_cast<const uint8_t*>(which ? p.Himg : p.dSimg) + img;
                        msc::mbar_arrive_expect_tx(&tfull[st], 32768u);
                        msc::tma_load_3d(sg, which ? &tmC : &tmB, &tfull[st], g * kN + 64 * kb, (int)(tc0 + j0), b);
                        msc::bulk_g2s(sg + 32768, im + 8192 * kb, 8192u, &tfull[st]);
                        msc::bulk_g2s(sg + 40960, im + 16384 + 8192 * kb, 8192u, &tfull[st]);
                    } else {
                        const int i0 = j0 + 64 * s;
                        msc::mbar_arrive_expect_tx(&tfull[st], (has_z ? 16384u : 8192u) + 256u * kGW);
                        msc::tma_load_2d(sg + 49152, &tmG, &tfull[st], j0, grow + i0);
                        msc::tma_load_3d(sg + 32768, &tmDy, &tfull[st], h * kP, (int)(tc0 + i0), b);
                        if (has_z) msc::tma_load_3d(sg + 40960, &tmZ, &tfull[st], h * kP, (int)(tc0 + i0), b);
                    }
                    ++issued;
                }
                if (!ok) break;
                // the epilogue's dy and x rows of this head (one buffer: after the
                // previous head's epilogue has read it)
                if (!has_z) {
                    if (hh >= 1 && !msc::wait_bounded(efree, (uint32_t)((hh - 1) & 1), abort, kSleepNs)) {
                        ok = false;
                        break;
                    }
                    msc::mbar_arrive_expect_tx(efull, kDxEpi);
                    msc::tma_load_3d(s_epi, &tmDyE, efull, h * kP, (int)(tc0 + j0), b);
                    msc::tma_load_3d(s_epi + 16384, &tmXE, efull, h * kP, (int)(tc0 + j0), b);
                    ++eissued;
                }
            }
            if (!ok) {
                record_timeout(101);
                *abort = 1u;
            }
            // no copy may still be landing when the block exits
            for (int st = 0; st < kDxStages && st < issued; ++st)
                if (!msc::wait_bounded(&tfull[st], (uint32_t)(((issued - 1 - st) / kDxStages) & 1), nullptr, kSleepNs))
                    record_timeout(102);
            for (int rb = 0; rb < 3 && rb < rissued; ++rb)
                if (!msc::wait_bounded(&rfull[rb], (uint32_t)(((rissued - 1 - rb) / 3) & 1), nullptr, kSleepNs))
                    record_timeout(102);
            if (eissued > 0 && !msc::wait_bounded(efull, (uint32_t)((eissued - 1) & 1), nullptr, kSleepNs))
                record_timeout(102);
        }
        __syncwarp();
    } else if (warp == kDxWarpMma) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            const uint32_t idK = msc::idesc_f16(true, 128, kP);
            const uint32_t idX = msc::idesc_f16(true, 128, kP, false, true);
            bool ok = true;
            for (int hh = 0; hh < nh && ok; ++hh) {
                const int ab = hh & 1;
                const uint32_t acc1 = tmem + 256u * (uint32_t)ab;
                if (hh >= 2) ok = msc::wait_bounded(&afree[ab], (uint32_t)(((hh - 2) >> 1) & 1), abort, kSleepNs);
                for (int s = 0; s < ns && ok; ++s) {
                    const int u = hh * ns + s, st = u % kDxStages, use = u / kDxStages;
                    ok = msc::wait_bounded(&tfull[st], (uint32_t)(use & 1), abort, kSleepNs) &&
                         msc::wait_bounded(&full[st], (uint32_t)(use & 1), abort, kSleepNs);
                    if (!ok) break;
                    msc::tc_fence_after();
                    const uint32_t a = msc::smem_u32(stages + st * kDxStage);
                    if (s >= na) {
                        const int si = s - na;
                        const uint32_t acc = acc1 + (si < 2 ? 64u : 128u);
                        for (int k = 0; k < 4; ++k) {
                            const uint64_t ad = msc::sdesc_sw128(a + 32 * k);
                            msc::mma_f16(acc, ad, msc::sdesc_sw128(a + 32768 + 32 * k), idK, ((si & 1) || k) ? 1u : 0u);
                            msc::mma_f16(acc, ad, msc::sdesc_sw128(a + 40960 + 32 * k), idK, 1u);
                        }
                    } else {
                        for (int k = 0; k < 4; ++k) {
                            const uint64_t bh = msc::sdesc_sw128_mn(a + 32768 + 2048 * k, 8192u);
                            const uint64_t ah = msc::sdesc_sw128(a + 32 * k);
                            msc::mma_f16(acc1, ah, bh, idX, (s > 0 || k) ? 1u : 0u);
                            msc::mma_f16(acc1, msc::sdesc_sw128(a + 16384 + 32 * k), bh, idX, 1u);
                            if (has_z) msc::mma_f16(acc1, ah, msc::sdesc_sw128_mn(a + 40960 + 2048 * k, 8192u), idX, 1u);
                        }
                    }
                    msc::mma_commit(&empty[st]);
                }
                if (ok) msc::mma_commit(&afull[ab]);
            }
            if (!ok) {
                record_timeout(103);
                *abort = 1u;
            }
            // every MMA issued completes before the tensor memory is released
            msc::mma_commit(drain);
            if (!msc::wait_bounded(drain, 0, nullptr, kSleepNs)) record_timeout(104);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ operands, then epilogue
        bool ok = true;
        auto fail_here = [&]() {
            if (lane == 0) record_timeout(105);
            *abort = 1u;
        };
        auto produce_head = [&](int hh) {
            const int rb = hh % 3;
            ok = ok && __all_sync(0xffffffffu, msc::wait_bounded(&rfull[rb], (uint32_t)((hh / 3) & 1), abort, kSleepNs));
            const float* s_cs = s_rows + 512 * rb;
            for (int s = 0; s < ns && ok; ++s) {
                const int u = hh * ns + s, st = u % kDxStages, use = u / kDxStages;
                uint8_t* sg = stages + st * kDxStage;
                // every slab: the stage's previous MMAs are done before this use is
                // announced (a full barrier may not run a phase ahead of its consumer)
                if (use > 0) ok = __all_sync(0xffffffffu, msc::wait_bounded(&empty[st], (uint32_t)((use - 1) & 1), abort, kSleepNs));
                if (!ok) break;
                if (s < na) {
                    // A = (E o G)^T of this slab: rows j (128), K = 64 steps i from i0; G and
                    // the g tile arrive by TMA
                    ok = __all_sync(0xffffffffu, msc::wait_bounded(&tfull[st], (uint32_t)(use & 1), abort, kSleepNs));
                    if (!ok) break;
                    const int i0 = j0 + 64 * s;
                    const float* sG = reinterpret_cast<const float*>(sg + 49152);
                    // thread: row (tid & 127), chunks kc = tid / 128 + 4 r of 8 steps
                    const int row = tid & 127, j = j0 + row;
                    const bool row_on = row < rows_valid;
                    const float csj = s_cs[row_on ? j : 0];
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const int kc = (tid >> 7) + 4 * r, ib = i0 + 8 * kc;
                        uint32_t hi[4] = {0u, 0u, 0u, 0u}, lo[4] = {0u, 0u, 0u, 0u};
                        if (row_on && ib + 7 >= j) {  // else the whole chunk lies above the diagonal
                            float v[8];
                            const float* gcol = sG + (ib - i0) * kGW + row;
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                const int i = ib + q;
                                v[q] = i >= j ? gcol[q * kGW] * msc::ex2_approx((s_cs[i] - csj) * MSC_LOG2E) : 0.f;
                            }
#pragma unroll
                            for (int q = 0; q < 4; ++q) msc::split_bf16x2(v[2 * q], v[2 * q + 1], hi[q], lo[q]);
                        }
                        const uint32_t off = msc::sw128_offset(row, 8 * kc, 128);
                        *reinterpret_cast<uint4*>(sg + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                        *reinterpret_cast<uint4*>(sg + 16384 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    }
                    if (has_z) {
                        // g = dy silu(z) in place: hi over dy, lo over z (one 16-byte chunk per thread)
                        uint4* ph = reinterpret_cast<uint4*>(sg + 32768 + 16 * tid);
                        uint4* pl = reinterpret_cast<uint4*>(sg + 40960 + 16 * tid);
                        const uint4 dv = *ph, zv = *pl;
                        const uint32_t dw[4] = {dv.x, dv.y, dv.z, dv.w}, zw[4] = {zv.x, zv.y, zv.z, zv.w};
                        uint32_t hi[4], lo[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            msc::split_bf16x2(msc::bf16lo(dw[q]) * msc::silu_f(msc::bf16lo(zw[q])),
                                              msc::bf16hi(dw[q]) * msc::silu_f(msc::bf16hi(zw[q])), hi[q], lo[q]);
                        *ph = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                        *pl = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    }
                }
                msc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) msc::mbar_arrive(&full[st]);
            }
            if (!ok) fail_here();
        };
        // warp w: TMEM lanes 32 (w % 4) .. (rows j), columns 16 (w / 4) .. of each accumulator
        const int lq = warp & 3, cq = warp >> 2;
        const int row = 32 * lq + lane, j = j0 + row;
        const int64_t t = tc0 + j;
        auto epilogue_head = [&](int hh) {
            const int ab = hh & 1, rb = hh % 3;
            const int h = hb * kDxHB + hh;
            const size_t dbase = ((size_t)b * p.H + h) * p.Lp + (size_t)tc0;
            const float* s_cs = s_rows + 512 * rb;
            const float* s_dt = s_cs + 256;
            const float Dh = p.D ? __ldg(p.D + h) : 0.f;  // issued before the waits
            ok = ok && __all_sync(0xffffffffu, msc::wait_bounded(&afull[ab], (uint32_t)((hh >> 1) & 1), abort, kSleepNs));
            msc::tc_fence_after();
            const bool valid = ok && row < rows_valid && t < p.L;
            float dw = 0.f, v = 0.f, ej = 0.f, wj = 0.f, ecs = 0.f, dd = 0.f;
            float a1[16], a2[16], a3[16];
            if (ok) {
                const uint32_t ta = tmem + 256u * (uint32_t)ab + ((uint32_t)(32 * lq) << 16) + (uint32_t)(16 * cq);
                msc::tmem_ld16(ta, a1);
                msc::tmem_ld16(ta + 64, a2);
                msc::tmem_ld16(ta + 128, a3);
                msc::tmem_ld_wait();
            }
            msc::tc_fence_before();
            __syncwarp();
            if (lane == 0) msc::mbar_arrive(&afree[ab]);  // the next head but one may write this buffer
            if (!has_z) ok = ok && __all_sync(0xffffffffu, msc::wait_bounded(efull, (uint32_t)(hh & 1), abort, kSleepNs));
            if (valid) {
                const size_t o = (((size_t)b * p.L + t) * p.H + h) * kP + 16 * cq;
                const float dtj = s_dt[j];
                ej = msc::ex2_approx((s_cs[Q - 1] - s_cs[j]) * MSC_LOG2E);
                wj = ej * dtj;
                ecs = msc::ex2_approx(s_cs[j] * MSC_LOG2E);
#pragma unroll
                for (int q8 = 0; q8 < 2; ++q8) {
                    uint4 dv, xv;
                    if (has_z) {
                        dv = *reinterpret_cast<const uint4*>(p.dy + o + 8 * q8);
                        xv = *reinterpret_cast<const uint4*>(p.x + o + 8 * q8);
                    } else {
                        const uint32_t eo = msc::sw128_offset(row, 16 * cq + 8 * q8, 128);
                        dv = *reinterpret_cast<const uint4*>(s_epi + eo);
                        xv = *reinterpret_cast<const uint4*>(s_epi + 16384 + eo);
                    }
                    uint4 zv = make_uint4(0u, 0u, 0u, 0u);
                    if (has_z) zv = *reinterpret_cast<const uint4*>(p.z + o + 8 * q8);
                    const uint32_t dwd[4] = {dv.x, dv.y, dv.z, dv.w}, xw[4] = {xv.x, xv.y, xv.z, xv.w};
                    const uint32_t zw[4] = {zv.x, zv.y, zv.z, zv.w};
                    float yp[8];
                    if (has_z) {
                        const float4 y0 = *reinterpret_cast<const float4*>(p.ypre + o + 8 * q8);
                        const float4 y1 = *reinterpret_cast<const float4*>(p.ypre + o + 8 * q8 + 4);
                        yp[0] = y0.x; yp[1] = y0.y; yp[2] = y0.z; yp[3] = y0.w;
                        yp[4] = y1.x; yp[5] = y1.y; yp[6] = y1.z; yp[7] = y1.w;
                    }
                    float out[8], dzo[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int q = 8 * q8 + e;
                        const float dyv = (e & 1) ? msc::bf16hi(dwd[e >> 1]) : msc::bf16lo(dwd[e >> 1]);
                        const float xvv = (e & 1) ? msc::bf16hi(xw[e >> 1]) : msc::bf16lo(xw[e >> 1]);
                        float gv = dyv;
                        if (has_z) {
                            // gate: g = dy silu(z), dz = dy y_pre silu'(z)
                            const float zz = (e & 1) ? msc::bf16hi(zw[e >> 1]) : msc::bf16lo(zw[e >> 1]);
                            const float sg = msc::sigmoid_f(zz);
                            gv = dyv * zz * sg;
                            dzo[e] = dyv * yp[e] * sg * (1.f + zz * (1.f - sg));
                        }
                        out[e] = dtj * a1[q] + wj * a2[q] + Dh * gv;
                        dw = fmaf(xvv, a2[q], dw);
                        v = fmaf(gv, a3[q], v);
                        dd = fmaf(gv, xvv, dd);
                    }
                    msc::st_cs_v8(p.dx + o + 8 * q8, out);
                    if (has_z) msc::st_cs_v8(p.dz + o + 8 * q8, dzo);
                }
            }
            if (!has_z) {
                __syncwarp();
                if (lane == 0) msc::mbar_arrive(efree);   // the next head's tiles may land
            }
            s_part[128 * cq + row] = dw;
            s_part[512 + 128 * cq + row] = v;
            // dD = sum g . x over steps and channels of the head
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) dd += __shfl_xor_sync(0xffffffffu, dd, off);
            if (lane == 0 && p.dD && dd != 0.f) atomicAdd(p.dD + h, dd);
            asm volatile("bar.sync 1, 512;" ::: "memory");
            if (cq == 0) {
                float lastp = 0.f;
                if (valid) {
                    const float dwt = dw + s_part[128 + row] + s_part[256 + row] + s_part[384 + row];
                    const float vt = v + s_part[640 + row] + s_part[768 + row] + s_part[896 + row];
                    atomicAdd(p.dDelta + dbase + j, ej * dwt);
                    // w_j dw_j goes to dcs_last and out of dcs_j: for j = last the two
                    // cancel exactly and are left out
                    const bool last = j == Q - 1;
                    atomicAdd(p.dcs + dbase + j, ecs * vt - (last ? 0.f : wj * dwt));
                    lastp = last ? 0.f : wj * dwt;
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) lastp += __shfl_xor_sync(0xffffffffu, lastp, off);
                if (lane == 0 && lastp != 0.f) atomicAdd(p.dcs + dbase + Q - 1, lastp);
            }
            asm volatile("bar.sync 1, 512;" ::: "memory");  // s_part is rewritten by the next head
            __syncwarp();
            if (lane == 0) msc::mbar_arrive(&rfree[rb]);
        };
        for (int hh = 0; hh <= nh; ++hh) {
            if (hh < nh) produce_head(hh);
            if (hh >= 1) epilogue_head(hh - 1);
        }
        if (!ok) fail_here();
        msc::tc_fence_before();
    }
    __syncthreads();
    if (warp == 0) {
        msc::tc_fence_after();
        msc::tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ state parts of dB, dC on tcgen05
// CTA = (chunk * nmb + row block mb of 128 steps, group * nhb + block of up to
// kHBlk heads, batch).  Two accumulators in tensor memory, M = 128 steps,
// N = 128 states, summed over the block's heads (K = heads x P):
//   accB[j, n] += sum_p (w_j x_j[p]) dS_h[p, n]        (dB_j += sum_h w_j x_j . dS_h)
//   accC[i, n] += sum_p (exp(cs_i) g_i[p]) Hin_h[p, n]  (dC_i += sum_h exp(cs_i) g_i . Hin_h)
// Per head two slabs through a ring of three 64 KB stages: A hi [128][64 p] |
// A lo | B hi [64 p][128 n] | B lo.  A is the TMA tile of x (or dy, with z
// landing in the A lo slot), scaled per row (and gated) and split in place; B
// is the head's dS or Hin image used MN-major (N = n, K = p), which is the same
// bytes as the K-major [64 p][128 n] image.  The sums are added to dB, dC
// (which already hold the dG terms) with vector reductions.
constexpr int kSbStages = 3;
constexpr uint32_t kSbStage = 65536;
constexpr int kSbOpWarps = 8;
constexpr int kSbWarpLoad = kSbOpWarps, kSbWarpMma = kSbOpWarps + 1;
constexpr int kSbThreads = (kSbOpWarps + 2) * 32;
constexpr size_t kSbSmem = 1024 + kSbStages * kSbStage + kSbStages * 384 * 4 + 16 * 8 + 16;

__global__ void __launch_bounds__(kSbThreads, 1) ssd_dbcs_tc_kernel(const __grid_constant__ CUtensorMap tmX,
                                                                    const __grid_constant__ CUtensorMap tmDy,
                                                                    const __grid_constant__ CUtensorMap tmZ,
                                                                    const SsdBwdParams p) {
    extern __shared__ uint8_t s_dyn[];
    uint8_t* stages = s_dyn + ((1024u - (msc::smem_u32(s_dyn) & 1023u)) & 1023u);
    float* s_cw = reinterpret_cast<float*>(stages + kSbStages * kSbStage);  // per stage: cs [256], Delta [128]
    uint64_t* bars = reinterpret_cast<uint64_t*>(s_cw + kSbStages * 384);
    // 0-2 stage loaded (TMA), 3-5 stage built (8 warps), 6-8 free (MMA), 9 done, 10 drain
    uint64_t *tfull = bars, *full = bars + 3, *empty = bars + 6, *done = bars + 9, *drain = bars + 10;
    uint32_t* slot = reinterpret_cast<uint32_t*>(bars + 11);
    volatile uint32_t* abort = slot + 1;

    const int Q = p.Q;
    const int nmb = (Q + 127) / 128;
    const int nhb = (p.hpg + kHBlk - 1) / kHBlk;
    const int c = blockIdx.x / nmb, mb = blockIdx.x % nmb;
    const int g = blockIdx.y / nhb, hb = blockIdx.y % nhb;
    const int b = blockIdx.z;
    const int j0 = 128 * mb;
    const int rows_valid = min(128, Q - j0);
    const int hh0 = hb * kHBlk;
    const int nh = min(kHBlk, p.hpg - hh0);
    const int ns = 2 * nh;                       // slab 2 k: dB term of head k, 2 k + 1: dC term
    const int64_t tc0 = (int64_t)c * Q;
    const bool has_z = p.z != nullptr;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (warp == 0) {
        msc::tmem_alloc(slot, 256);
        msc::tmem_relinquish();
    }
    if (tid == 32) {
        for (int k = 0; k < kSbStages; ++k) {
            msc::mbar_init(&tfull[k], 1);
            msc::mbar_init(&full[k], kSbOpWarps);
            msc::mbar_init(&empty[k], 1);
        }
        msc::mbar_init(done, 1);
        msc::mbar_init(drain, 1);
        slot[1] = 0u;
        msc::fence_barrier_init();
    }
    msc::tc_fence_before();
    __syncthreads();
    msc::tc_fence_after();
    const uint32_t tmem = *slot;

    if (warp == kSbWarpLoad) {
        if (lane == 0) {
            msc::prefetch_tmap(&tmX);
            msc::prefetch_tmap(&tmDy);
            if (has_z) msc::prefetch_tmap(&tmZ);
            int issued = 0;
            for (int s = 0; s < ns; ++s) {
                const int st = s % kSbStages, use = s / kSbStages;
                if (use > 0 && !msc::wait_bounded(&empty[st], (uint32_t)((use - 1) & 1), abort, kSleepNs)) {
                    record_timeout(111);
                    *abort = 1u;
                    break;
                }
                const int h = g * p.hpg + hh0 + (s >> 1);
                const bool cterm = s & 1;
                uint8_t* sg = stages + st * kSbStage;
                const uint8_t* im = reinterpret_cast<const uint8_t*>(cterm ? p.Himg : p.dSimg) +
                                    (((size_t)b * p.nc + c) * p.H + h) * 32768;
                const size_t dbase = ((size_t)b * p.H + h) * p.Lp + (size_t)tc0;
                msc::mbar_arrive_expect_tx(&tfull[st], ((cterm && has_z) ? 65536u : 49152u) + 4u * (uint32_t)(Q + rows_valid));
                msc::bulk_g2s(s_cw + 384 * st, p.cs + dbase, 4u * (uint32_t)Q, &tfull[st]);
                msc::bulk_g2s(s_cw + 384 * st + 256, p.dt + dbase + j0, 4u * (uint32_t)rows_valid, &tfull[st]);
                msc::tma_load_3d(sg, cterm ? &tmDy : &tmX, &tfull[st], h * kP, (int)(tc0 + j0), b);
                if (cterm && has_z) msc::tma_load_3d(sg + 16384, &tmZ, &tfull[st], h * kP, (int)(tc0 + j0), b);
                msc::bulk_g2s(sg + 32768, im, 32768u, &tfull[st]);
                ++issued;
            }
            for (int st = 0; st < kSbStages && st < issued; ++st)
                if (!msc::wait_bounded(&tfull[st], (uint32_t)(((issued - 1 - st) / kSbStages) & 1), nullptr, kSleepNs)) record_timeout(112);
        }
        __syncwarp();
    } else if (warp == kSbWarpMma) {
        if (lane == 0) {
            const uint32_t idX = msc::idesc_f16(true, 128, kN, false, true);
            bool ok = true;
            for (int s = 0; s < ns && ok; ++s) {
                const int st = s % kSbStages, use = s / kSbStages;
                ok = msc::wait_bounded(&tfull[st], (uint32_t)(use & 1), abort, kSleepNs) &&
                     msc::wait_bounded(&full[st], (uint32_t)(use & 1), abort, kSleepNs);
                if (!ok) break;
                msc::tc_fence_after();
                const uint32_t a = msc::smem_u32(stages + st * kSbStage);
                const uint32_t acc = tmem + ((s & 1) ? 128u : 0u);
                for (int k = 0; k < 4; ++k) {
                    const uint64_t ah = msc::sdesc_sw128(a + 32 * k), al = msc::sdesc_sw128(a + 16384 + 32 * k);
                    const uint64_t bh = msc::sdesc_sw128_mn(a + 32768 + 2048 * k, 8192u);
                    const uint64_t bl = msc::sdesc_sw128_mn(a + 49152 + 2048 * k, 8192u);
                    msc::mma_f16(acc, ah, bh, idX, (s > 1 || k) ? 1u : 0u);
                    msc::mma_f16(acc, ah, bl, idX, 1u);
                    msc::mma_f16(acc, al, bh, idX, 1u);
                }
                msc::mma_commit(&empty[st]);
            }
            if (ok) {
                msc::mma_commit(done);
            } else {
                record_timeout(113);
                *abort = 1u;
            }
            msc::mma_commit(drain);
            if (!msc::wait_bounded(drain, 0, nullptr, kSleepNs)) record_timeout(114);
        }
        __syncwarp();
    } else {
        bool ok = true;
        for (int s = 0; s < ns; ++s) {
            const int st = s % kSbStages, use = s / kSbStages;
            const bool cterm = s & 1;
            uint8_t* sg = stages + st * kSbStage;
            ok = ok && __all_sync(0xffffffffu, msc::wait_bounded(&tfull[st], (uint32_t)(use & 1), abort, kSleepNs));
            if (!ok) break;
            const float* scs = s_cw + 384 * st;
            const float cs_last = scs[Q - 1];
            // 1024 chunks of 16 bytes (8 p of one row) per tile, 4 per thread
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int u = tid + 256 * r;
                const int row = u >> 3;
                float wr = 0.f;
                if (row < rows_valid) {
                    const float csr = scs[j0 + row];
                    wr = cterm ? msc::ex2_approx(csr * MSC_LOG2E) : msc::ex2_approx((cs_last - csr) * MSC_LOG2E) * scs[256 + row];
                }
                uint4* ph = reinterpret_cast<uint4*>(sg + 16 * u);
                uint4* pl = reinterpret_cast<uint4*>(sg + 16384 + 16 * u);
                const uint4 xv = *ph;
                const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
                uint32_t zw[4] = {0u, 0u, 0u, 0u};
                if (cterm && has_z) {
                    const uint4 zv = *pl;
                    zw[0] = zv.x; zw[1] = zv.y; zw[2] = zv.z; zw[3] = zv.w;
                }
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float a0 = msc::bf16lo(xw[q]) * wr, a1 = msc::bf16hi(xw[q]) * wr;
                    if (cterm && has_z) {
                        a0 *= msc::silu_f(msc::bf16lo(zw[q]));
                        a1 *= msc::silu_f(msc::bf16hi(zw[q]));
                    }
                    msc::split_bf16x2(a0, a1, hi[q], lo[q]);
                }
                *ph = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *pl = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            msc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) msc::mbar_arrive(&full[st]);
            // the next use of this stage is loaded only after these MMAs (empty), so no wait here
        }
        if (!ok) {
            if (lane == 0) record_timeout(115);
            *abort = 1u;
        }
        ok = ok && __all_sync(0xffffffffu, msc::wait_bounded(done, 0, abort, kSleepNs));
        msc::tc_fence_after();
        if (ok) {
            const int lq = warp & 3, half = warp >> 2;
            const int row = 32 * lq + lane;
            const int64_t t = tc0 + j0 + row;
            const bool valid = row < rows_valid && t < p.L;
            const size_t o = (((size_t)b * p.L + t) * p.Gr + g) * kN + 64 * half;
#pragma unroll 1
            for (int term = 0; term < 2; ++term) {
                float* dst = (term ? p.dC : p.dB) + o;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float v[16];
                    msc::tmem_ld16(tmem + ((uint32_t)(32 * lq) << 16) + (uint32_t)(128 * term + 64 * half + 16 * q), v);
                    msc::tmem_ld_wait();
                    if (valid) {
#pragma unroll
                        for (int e = 0; e < 16; e += 4) red_add_v4(dst + 16 * q + e, v[e], v[e + 1], v[e + 2], v[e + 3]);
                    }
                }
            }
        }
        msc::tc_fence_before();
    }
    __syncthreads();
    if (warp == 0) {
        msc::tc_fence_after();
        msc::tmem_dealloc(tmem, 256);
    }
}

// ------------------------------------------------------------------ cs -> Delta, A; softplus
// CTA = (chunk, head, batch), thread = step.  With R_r = sum_{i >= r} dcs_i (within the
// chunk): dDelta_r += A R_r, dA += Delta_r R_r; ddelta = dDelta sigmoid(delta + bias).
__global__ void __launch_bounds__(256) ssd_dcs_kernel(const SsdBwdParams p) {
    __shared__ float s_w[8];
    __shared__ float s_red[2][8];
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const size_t dbase = ((size_t)b * p.H + h) * p.Lp + (size_t)c * p.Q;
    const int r = p.Q - 1 - tid;  // thread tid walks the chunk backwards
    float v = (r >= 0) ? p.dcs[dbase + r] : 0.f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) s_w[warp] = v;
    __syncthreads();
    for (int w = 0; w < warp; ++w) v += s_w[w];
    float da = 0.f, dbias = 0.f;
    if (r >= 0) {
        const int64_t t = (int64_t)c * p.Q + r;
        const float A = p.A[h];
        da = p.dt[dbase + r] * v;
        if (t < p.L) {
            const float dD = p.dDelta[dbase + r] + A * v;
            const float xv = bfv(p.delta[((size_t)b * p.L + t) * p.H + h]) + (p.bias ? p.bias[h] : 0.f);
            const float dd = dD * msc::sigmoid_f(xv);
            p.ddelta[((size_t)b * p.L + t) * p.H + h] = dd;
            dbias = dd;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        da += __shfl_xor_sync(0xffffffffu, da, o);
        dbias += __shfl_xor_sync(0xffffffffu, dbias, o);
    }
    if (lane == 0) {
        s_red[0][warp] = da;
        s_red[1][warp] = dbias;
    }
    __syncthreads();
    if (tid == 0) {
        float sa = 0.f, sb = 0.f;
        for (int w = 0; w < 8; ++w) {
            sa += s_red[0][w];
            sb += s_red[1][w];
        }
        atomicAdd(p.dA + h, sa);
        if (p.dbias) atomicAdd(p.dbias + h, sb);
    }
}

size_t a256(size_t v) { return (v + 255) & ~size_t(255); }

}  // namespace

namespace msc_host {

size_t ssd_bwd_workspace(int64_t batch, int64_t L, int64_t H, int64_t G, int64_t Q, bool has_z) {
    const int64_t nc = (L + Q - 1) / Q, Lp = nc * Q;
    size_t s = 1024;
    s += 4 * a256((size_t)batch * H * Lp * 4);            // dt, cs, dcs, dDelta
    s += 5 * a256((size_t)batch * nc * H * kP * kN * 4);  // S, Hin, U / dS, and the Hin, dS bf16 hi + lo images
    s += 2 * a256((size_t)batch * nc * G * Q * Q * 4);    // G, dG
    if (has_z) s += a256((size_t)batch * L * H * kP * 4);  // pre-gate output
    return s;
}

msc_status ssd_bwd_launch(const SsdBwdArgs& a, cudaStream_t st) {
    const SsdArgs& f = a.f;
    SsdBwdParams p{};
    p.x = static_cast<const uint16_t*>(f.x);
    p.delta = static_cast<const uint16_t*>(f.delta);
    p.B = static_cast<const uint16_t*>(f.B);
    p.C = static_cast<const uint16_t*>(f.C);
    p.z = static_cast<const uint16_t*>(f.z);
    p.dy = static_cast<const uint16_t*>(a.dy);
    p.A = f.A; p.D = f.D; p.bias = f.delta_bias;
    p.dx = a.dx; p.ddelta = a.ddelta; p.dA = a.dA; p.dB = a.dB; p.dC = a.dC;
    p.dD = a.dD; p.dz = a.dz; p.dbias = a.ddelta_bias;
    p.L = f.L; p.batch = (int)f.batch; p.H = (int)f.H; p.Gr = (int)f.G; p.hpg = (int)(f.H / f.G); p.Q = (int)f.Q;
    p.nc = (int)((f.L + f.Q - 1) / f.Q);
    p.Lp = (int64_t)p.nc * f.Q;
    const size_t nrow = (size_t)f.batch * f.H * p.Lp * 4;
    const size_t nst = (size_t)f.batch * p.nc * f.H * kP * kN * 4;
    const size_t ngm = (size_t)f.batch * p.nc * f.G * f.Q * f.Q * 4;
    // the first four buffers are laid out as the forward's workspace (Delta, cs,
    // chunk states, state images), so that with a gate the forward run that
    // gives y_pre also leaves the states the backward needs
    char* base = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(a.workspace) + 1023) & ~uintptr_t(1023));
    char* ws = base;
    float* dt = reinterpret_cast<float*>(ws); ws += a256(nrow);
    float* cs = reinterpret_cast<float*>(ws); ws += a256(nrow);
    float* S = reinterpret_cast<float*>(ws); ws += a256(nst);
    uint16_t* Himg = reinterpret_cast<uint16_t*>(ws); ws += a256(nst);
    p.dcs = reinterpret_cast<float*>(ws); ws += a256(nrow);
    p.dDelta = reinterpret_cast<float*>(ws); ws += a256(nrow);
    float* Hin = reinterpret_cast<float*>(ws); ws += a256(nst);
    float* U = reinterpret_cast<float*>(ws); ws += a256(nst);
    p.U = U;
    p.dSimg = reinterpret_cast<uint16_t*>(ws); ws += a256(nst);
    p.Himg = Himg;
    p.Gm = reinterpret_cast<float*>(ws); ws += a256(ngm);
    p.dG = reinterpret_cast<float*>(ws); ws += a256(ngm);
    p.dt = dt; p.cs = cs; p.Hin = Hin;
    msc_status s;
    if (f.z) {
        // the forward without the gate: y_pre, and Delta, cs, S, Hin in this workspace
        float* ypre = reinterpret_cast<float*>(ws); ws += a256((size_t)f.batch * f.L * f.H * kP * 4);
        SsdArgs fa = f;
        fa.z = nullptr; fa.y = ypre; fa.final_state = nullptr; fa.workspace = base; fa.Hin32 = Hin;
        if ((s = ssd_launch(fa, st)) != MSC_OK) return s;
        p.ypre = ypre;
    } else if ((s = ssd_states(f, dt, cs, S, Hin, Himg, st)) != MSC_OK) {
        return s;
    }
    cudaError_t e = cudaMemsetAsync(p.dcs, 0, 2 * a256(nrow), st);  // dcs and dDelta are adjacent
    if (e == cudaSuccess) e = cudaMemsetAsync(p.dA, 0, (size_t)f.H * 4, st);
    if (e == cudaSuccess && p.dD) e = cudaMemsetAsync(p.dD, 0, (size_t)f.H * 4, st);
    if (e == cudaSuccess && p.dbias) e = cudaMemsetAsync(p.dbias, 0, (size_t)f.H * 4, st);
    if (e != cudaSuccess) return fail(MSC_ERR_CUDA, "ssd bwd memset: %s", cudaGetErrorString(e));
    const unsigned nb = (unsigned)(f.Q / kT), ntri = nb * (nb + 1) / 2;
    const unsigned B = (unsigned)f.batch, H = (unsigned)f.H, nc = (unsigned)p.nc, BG = (unsigned)(f.batch * f.G);
    // B, C as [128 steps][64 n] boxes; x, dy, z as [64 steps][64 p] and [128 steps][64 p] boxes
    // (bf16, 128-byte swizzle)
    CUtensorMap mB, mC, mDy, mZ, mX128, mDy128, mZ128, mG;
    {
        const uint64_t bcd[3] = {(uint64_t)(f.G * kN), (uint64_t)f.L, (uint64_t)f.batch};
        const uint64_t bcs[2] = {(uint64_t)(f.G * kN * 2), (uint64_t)(f.L * f.G * kN * 2)};
        const uint64_t xd[3] = {(uint64_t)(f.H * kP), (uint64_t)f.L, (uint64_t)f.batch};
        const uint64_t xs[2] = {(uint64_t)(f.H * kP * 2), (uint64_t)(f.L * f.H * kP * 2)};
        const uint32_t box128[3] = {64, 128, 1}, box64[3] = {64, 64, 1};
        const void* zsrc = f.z ? f.z : a.dy;  // unused without a gate
        if (!encode_tmap(&mB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, f.B, bcd, bcs, box128, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_tmap(&mC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, f.C, bcd, bcs, box128, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_tmap(&mDy, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.dy, xd, xs, box64, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_tmap(&mZ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, zsrc, xd, xs, box64, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_tmap(&mX128, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, f.x, xd, xs, box128, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_tmap(&mDy128, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.dy, xd, xs, box128, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_tmap(&mZ128, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, zsrc, xd, xs, box128, CU_TENSOR_MAP_SWIZZLE_128B))
            return MSC_ERR_CUDA;
        // G as rows of Q fp32, [64 i][min(Q, 128) j] boxes
        const uint64_t gd[2] = {(uint64_t)f.Q, (uint64_t)(f.batch * p.nc * f.G * f.Q)};
        const uint64_t gs[1] = {(uint64_t)(f.Q * 4)};
        const uint32_t gbox[2] = {(uint32_t)std::min<int64_t>(f.Q, 128), 64};
        if (!encode_tmap(&mG, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, p.Gm, gd, gs, gbox, CU_TENSOR_MAP_SWIZZLE_NONE))
            return MSC_ERR_CUDA;
        static std::atomic<uint64_t> configured{0};  // one bit per device on which the attribute is set
        if (!(configured & msc_host::device_bit())) {
            cudaError_t e2 = cudaSuccess;
            for (const void* k : {(const void*)ssd_dx_tc_kernel<64, false>, (const void*)ssd_dx_tc_kernel<64, true>,
                                  (const void*)ssd_dx_tc_kernel<128, false>, (const void*)ssd_dx_tc_kernel<128, true>,
                                  (const void*)ssd_dx_tc_kernel<256, false>, (const void*)ssd_dx_tc_kernel<256, true>})
                if (e2 == cudaSuccess) e2 = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDxSmem);
            if (e2 == cudaSuccess)
                e2 = cudaFuncSetAttribute(ssd_dbcs_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSbSmem);
            if (e2 == cudaSuccess)
                e2 = cudaFuncSetAttribute(ssd_dg_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDgSmem);
            if (e2 != cudaSuccess) return fail(MSC_ERR_CUDA, "ssd bwd smem attribute: %s", cudaGetErrorString(e2));
            configured |= msc_host::device_bit();
        }
    }
    const unsigned nmb = (unsigned)((f.Q + 127) / 128), ntri128 = nmb * (nmb + 1) / 2;
    ssd_gmat_kernel<<<dim3(ntri, nc, BG), 256, 0, st>>>(p);
    if ((s = check_launch("ssd_gmat")) != MSC_OK) return s;
    if ((s = ssd_ugrad(f, a.dy, cs, U, st)) != MSC_OK) return s;
    ssd_rpass_kernel<<<dim3(H * (kP * kN / 8) / 256, B), 256, 0, st>>>(p);
    if ((s = check_launch("ssd_rpass")) != MSC_OK) return s;
    {
        // enough head blocks per tile to give every SM about two CTAs
        const int tiles = (int)(ntri128 * nc * BG);
        const int want = std::max(1, std::min(p.hpg, (2 * 148 + tiles - 1) / tiles));
        p.dg_hpb = (p.hpg + want - 1) / want;
        const unsigned nhb = (unsigned)((p.hpg + p.dg_hpb - 1) / p.dg_hpb);
        e = cudaMemsetAsync(p.dG, 0, ngm, st);
        if (e != cudaSuccess) return fail(MSC_ERR_CUDA, "ssd bwd memset: %s", cudaGetErrorString(e));
        ssd_dg_tc_kernel<<<dim3(ntri128 * nhb, nc, BG), kDgThreads, kDgSmem, st>>>(mX128, mDy128, mZ128, p);
    }
    if ((s = check_launch("ssd_dg_tc")) != MSC_OK) return s;
    ssd_dbc_kernel<<<dim3(2 * nb, nc, BG), 256, 0, st>>>(p);
    if ((s = check_launch("ssd_dbc")) != MSC_OK) return s;
    {
        const dim3 gdx(nc * nmb, (H + kDxHB - 1) / kDxHB, B);
        auto dx = [&](auto kern) { kern<<<gdx, kDxThreads, kDxSmem, st>>>(mB, mC, mDy, mZ, mG, mDy128, mX128, p); };
        const bool z = f.z != nullptr;
        if (f.Q == 64)
            z ? dx(ssd_dx_tc_kernel<64, true>) : dx(ssd_dx_tc_kernel<64, false>);
        else if (f.Q == 128)
            z ? dx(ssd_dx_tc_kernel<128, true>) : dx(ssd_dx_tc_kernel<128, false>);
        else
            z ? dx(ssd_dx_tc_kernel<256, true>) : dx(ssd_dx_tc_kernel<256, false>);
        if ((s = check_launch("ssd_dx_tc")) != MSC_OK) return s;
        const unsigned nhb = (unsigned)((p.hpg + kHBlk - 1) / kHBlk);
        ssd_dbcs_tc_kernel<<<dim3(nc * nmb, (unsigned)f.G * nhb, B), kSbThreads, kSbSmem, st>>>(mX128, mDy128, mZ128, p);
        if ((s = check_launch("ssd_dbcs_tc")) != MSC_OK) return s;
    }
    ssd_dcs_kernel<<<dim3(nc, H, B), 256, 0, st>>>(p);
    return check_launch("ssd_dcs");
}

msc_status ssd_bwd_take_status(unsigned int* code, unsigned int* site) {
    unsigned int w[2] = {0, 0};
    cudaError_t e = cudaMemcpyFromSymbol(w, g_ssdb_status, sizeof(w));
    if (e != cudaSuccess) return fail(MSC_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
    if (w[0] != 0) {
        const unsigned int zz[2] = {0, 0};
        e = cudaMemcpyToSymbol(g_ssdb_status, zz, sizeof(zz));
        if (e != cudaSuccess) return fail(MSC_ERR_CUDA, "status clear: %s", cudaGetErrorString(e));
    }
    *code = w[0];
    *site = w[1];
    return MSC_OK;
}

}  // namespace msc_host
