// s6_bwd.cu -- S6 selective-scan backward on sm_103a, by recomputation.
//
// Gradients of y_t = (sum_n C_tn h_tn + D u_t) silu(z_t) with
// h_tn = exp(Delta_t A_n) h_{t-1,n} + Delta_t B_tn u_t, Delta_t = softplus(delta_t + bias)
// (zero initial state).  The pages only say that the backward recomputes the
// states instead of storing them (bqwf survey sec. 2.2); the adjoint is derived
// by hand:
//   g'_t = dy_t silu(z_t),  dz_t = dy_t y'_t sig(z_t) (1 + z_t (1 - sig(z_t)))
//   lambda_tn = g'_t C_tn + abar_{t+1,n} lambda_{t+1,n}
//   du_t = g'_t D + Delta_t sum_n lambda_tn B_tn
//   dDelta_t = u_t sum_n lambda_tn B_tn + sum_n lambda_tn A_n abar_tn h_{t-1,n}
//   ddelta_t = dDelta_t sig(delta_t + bias),   dbias = sum ddelta,  dD = sum g' u
//   dA_n = sum_t lambda_tn Delta_t abar_tn h_{t-1,n}
//   dB_tn = sum_d lambda_tn Delta_t u_t,        dC_tn = sum_d g'_t h_tn
//
// Two launches.  (1) The forward kernel in checkpoint mode writes the state
// entering every 8-step group (1/8 of the states, fp32) to the workspace.
// (2) This kernel walks each row backwards: TMA streams the tiles of u, delta,
// z, dy, B, C in reverse order into a two-stage ring; for each 8-step group it
// takes the checkpoint (loaded one group ahead), recomputes the 8 steps forward keeping abar,
// h_{t-1} and B in registers, then runs the adjoint backwards through them,
// loading only C; the readout C h_t (for dz) and dC = g' h_t are formed there
// too, where h_t is the next step's h_{t-1}.  Each B and C value is read from
// shared memory once per group.  Four
// lanes share a row (4 states each) so the two 8-step histories fit in
// registers.  dB and dC, sums over all channels of a batch entry, are first
// summed over row pairs in registers (one shuffle exchange: each row of a pair
// keeps half of its states), then over the CTA's 16 row pairs in shared memory
// (conflict-free layout), and added to global memory with one 4-wide vector
// reduction per 4 steps.
// dA, dD and dbias are per-lane sums added once per row at the end.
#include <cstdio>
#include <cstdlib>

#include "msc_common.cuh"
#include "msc_internal.h"
#include "msc_tma.cuh"

namespace {

constexpr int kRows = 32;       // channel rows per CTA
constexpr int kNG = 4;          // lanes per row
constexpr int kThreads = kRows * kNG;
constexpr int kStages = 2;
constexpr int kRowTile = 2048;  // 32 rows x 64 bytes
constexpr int kBCTile = 1024;   // 16 slots x 64 bytes
constexpr int kStageBytes = 4 * kRowTile + 2 * kBCTile;
// dB / dC reduction buffer s_red[x][k][row][n]: 16 floats per row, rows 16.. shifted by
// 16 floats so that the two row halves summed side by side use different banks
constexpr int kRedBlock = 32 * 16 + 32;  // floats per (x, k) block
__host__ __device__ constexpr int red_row(int r) { return r * 16 + (r >= 16 ? 16 : 0); }
// row pair p = r / 2 after the pairs are summed in registers; pairs 8.. shifted
// by 16 floats so that the two halves read side by side use different banks
__host__ __device__ constexpr int red_pair(int p) { return p * 16 + (p >= 8 ? 16 : 0); }
constexpr int kSumPitch = 12;  // floats per (x, n) row of the per-group sums

__device__ unsigned int g_s6_bwd_status[2];

struct BwdParams {
    const float* A;
    const float* D;
    const float* delta_bias;
    const float* ckpt;  // [rows, ckpt_groups, 16]
    float* du;
    float* ddelta;
    float* dz;
    float* dA;
    float* dB;
    float* dC;
    float* dD;
    float* dbias;
    int64_t dim, L, ckpt_groups;
    int N;
    int has_z;
};

// More than 16 states run as slices of up to 16 (every gradient is a sum over
// states of per-state terms, or per state): A, dA and ckpt hold the slice
// only, dB and dC point at its first state row, bc_rows state rows apart per
// batch entry.  The first slice adds the terms without states (D u in the
// readout, g' D in du, dD); later slices add du, ddelta and dz to what is
// there.  A parameter of its own, which the whole-state instance never reads.
struct BwdSlice {
    int64_t bc_rows;
    int first, accumulate;
};

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// Lanes j of a row's group exchange halves: after the two levels lane j holds
// the full sums of steps 2j, 2j+1 in v[0], v[1].
__device__ __forceinline__ void reduce_scatter8(float* v, int j) {
    {
        const bool side = (j & 2) != 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float send = side ? v[k] : v[k + 4];
            const float keep = side ? v[k + 4] : v[k];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
        }
    }
    {
        const bool side = (j & 1) != 0;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const float send = side ? v[k] : v[k + 2];
            const float keep = side ? v[k + 2] : v[k];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
        }
    }
}

__device__ __forceinline__ float sigmoid_acc(float x) { return msc::rcp_approx(1.f + msc::ex2_approx(-x * MSC_LOG2E)); }

template <bool kBF16>
__device__ __forceinline__ void load2(const uint8_t* tile, int r, uint32_t boff, float& a, float& b) {
    const uint8_t* q = tile + msc::sw64(r, boff >> 4) + (boff & 15);
    if constexpr (kBF16) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(q);
        a = msc::bf16lo(w);
        b = msc::bf16hi(w);
    } else {
        const float2 v = *reinterpret_cast<const float2*>(q);
        a = v.x;
        b = v.y;
    }
}

// Two CTAs per SM (248-254 registers: the group's B pairs stay in registers
// from the recompute to the adjoint, so the adjoint loads only C).  At 16 x
// 2048 x 2048 bf16: 1.64 ms, against 1.72 with B loaded twice at three CTAs per
// SM and 2.4 with B kept but squeezed into three CTAs per SM (spills); the
// row-pair exchange of the dB/dC sums then 1.61.
// kSlice: one 16-state slice of a wider state (the flags and dB / dC stride of
// BwdParams apply); otherwise the whole state, 16 or fewer.
template <bool kBF16, bool kSlice>
__global__ void __launch_bounds__(kThreads, 2) s6_bwd_kernel(const __grid_constant__ CUtensorMap tm_u,
                                                         const __grid_constant__ CUtensorMap tm_d,
                                                         const __grid_constant__ CUtensorMap tm_z,
                                                         const __grid_constant__ CUtensorMap tm_dy,
                                                         const __grid_constant__ CUtensorMap tm_B,
                                                         const __grid_constant__ CUtensorMap tm_C,
                                                         const BwdParams p, const BwdSlice sl) {
    constexpr int kTT = kBF16 ? 32 : 16;  // steps per 64-byte tile row
    constexpr int kGroups = kTT / 8;
    constexpr int kPitch = 2 * kTT + 4;
    constexpr int kES = kBF16 ? 2 : 4;
    // dynamic shared memory, carved at a 1024-byte aligned base (TMA swizzle atoms)
    extern __shared__ uint8_t s_dyn[];
    // (offset from s_dyn itself, so the compiler keeps shared-memory accesses)
    uint8_t* base = s_dyn + ((1024u - (msc::smem_u32(s_dyn) & 1023u)) & 1023u);
    uint8_t (*s_raw)[kStageBytes] = reinterpret_cast<uint8_t (*)[kStageBytes]>(base);
    float (*s_bc)[8][kPitch] = reinterpret_cast<float (*)[8][kPitch]>(base + kStages * kStageBytes);
    float* s_red = reinterpret_cast<float*>(base + kStages * kStageBytes + 2 * 8 * kPitch * 4);
    // [x][n][k] row sums of one group, rows of kSumPitch floats (8 steps and a
    // pad: the four n of a warp's stores fall on two bank groups, not one)
    float* s_sum = s_red + 2 * 8 * kRedBlock;
    uint64_t* s_full = reinterpret_cast<uint64_t*>(s_sum + 2 * 16 * kSumPitch);

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int r = tid >> 2;  // row within the CTA
    const int j = tid & 3;   // states 4j..4j+3, steps 2j, 2j+1 of each group
    const int glane0 = lane & ~3;
    const int64_t b = blockIdx.y;
    const int64_t d0 = (int64_t)blockIdx.x * kRows;
    const int nrows = (int)((p.dim - d0) < kRows ? (p.dim - d0) : kRows);
    const bool row_ok = r < nrows;
    const int64_t d = row_ok ? d0 + r : d0;
    const int64_t row = b * p.dim + d;
    const int N = p.N;
    const bool has_z = p.has_z != 0;

    uint64_t A2p[2], Ap[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        float a[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int n = 4 * j + 2 * q + e;
            a[e] = (row_ok && n < N) ? __ldg(p.A + d * N + n) : 0.f;
        }
        Ap[q] = msc::pk2(a[0], a[1]);
        A2p[q] = msc::pk2(a[0] * MSC_LOG2E, a[1] * MSC_LOG2E);
    }
    const bool first = !kSlice || sl.first != 0;
    const bool accumulate = kSlice && sl.accumulate != 0;
    const int64_t bc_rows = kSlice ? sl.bc_rows : (int64_t)p.N;
    const float Dd = (p.D && row_ok && first) ? __ldg(p.D + d) : 0.f;
    const float bias = (p.delta_bias && row_ok) ? __ldg(p.delta_bias + d) : 0.f;

    uint64_t lam[2] = {0ull, 0ull};      // lambda of the step after the current one
    uint64_t a_carry[2] = {0ull, 0ull};  // abar of the step after the current group
    uint64_t dA2[2] = {0ull, 0ull};
    float dD_acc = 0.f, dbias_acc = 0.f;

    const int ntiles = (int)((p.L + kTT - 1) / kTT);
    const uint32_t tx_bytes = kRowTile * (has_z ? 4 : 3) + 2 * kBCTile;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) msc::mbar_init(&s_full[s], 1);
        msc::fence_barrier_init();
        msc::prefetch_tmap(&tm_u);
        msc::prefetch_tmap(&tm_d);
        msc::prefetch_tmap(&tm_dy);
        msc::prefetch_tmap(&tm_B);
        msc::prefetch_tmap(&tm_C);
        if (has_z) msc::prefetch_tmap(&tm_z);
    }
    __syncthreads();

    // tiles are consumed last to first; the c-th consumed tile uses stage c % 2
    auto issue = [&](int c) {
        const int s = c % kStages;
        const int ti = ntiles - 1 - c;
        const int tj = ti * kTT;
        uint8_t* st = s_raw[s];
        msc::mbar_arrive_expect_tx(&s_full[s], tx_bytes);
        msc::tma_load_3d(st, &tm_u, &s_full[s], tj, (int)d0, (int)b);
        msc::tma_load_3d(st + kRowTile, &tm_d, &s_full[s], tj, (int)d0, (int)b);
        msc::tma_load_3d(st + 2 * kRowTile, &tm_dy, &s_full[s], tj, (int)d0, (int)b);
        if (has_z) msc::tma_load_3d(st + 3 * kRowTile, &tm_z, &s_full[s], tj, (int)d0, (int)b);
        msc::tma_load_3d(st + 4 * kRowTile, &tm_B, &s_full[s], tj, 0, (int)b);
        msc::tma_load_3d(st + 4 * kRowTile + kBCTile, &tm_C, &s_full[s], tj, 0, (int)b);
    };
    if (tid == 0)
        for (int c = 0; c < kStages && c < ntiles; ++c) issue(c);
    int issued = ntiles < kStages ? ntiles : kStages;

    // groups are walked last to first (p.L is a multiple of 8): the checkpoint of
    // the next group is loaded one group ahead of its use
    const float* ck = p.ckpt + (size_t)row * p.ckpt_groups * 16 + 4 * j;
    float4 hv_next = row_ok ? __ldg(reinterpret_cast<const float4*>(ck + (size_t)((p.L - 8) >> 3) * 16))
                            : make_float4(0.f, 0.f, 0.f, 0.f);

    bool failed = false;
    int c = 0;
    for (; c < ntiles; ++c) {
        const int st = c % kStages;
        const bool ok = msc::wait_bounded(&s_full[st], (uint32_t)((c / kStages) & 1));
        if (__syncthreads_or(!ok)) {
            if (tid == 0 && atomicCAS(&g_s6_bwd_status[0], 0u, (unsigned int)MSC_ERR_TIMEOUT) == 0u)
                g_s6_bwd_status[1] = 2;
            failed = true;
            break;
        }
        const uint8_t* raw = s_raw[st];
        const int ti = ntiles - 1 - c;
        const int64_t t0 = (int64_t)ti * kTT;
        const int nt = (int)((p.L - t0) < kTT ? (p.L - t0) : kTT);  // a multiple of 8

        // B and C of this tile -> fp32 pairs s_bc[x][q][2t + e] = X[n = 2q + e][t]
        if (tid < 64) {
            const int x = tid >> 5, q = lane & 7, cc = lane >> 3;
            const uint8_t* src = raw + 4 * kRowTile + x * kBCTile;
            const uint4 v0 = *reinterpret_cast<const uint4*>(src + msc::sw64(2 * q, cc));
            const uint4 v1 = *reinterpret_cast<const uint4*>(src + msc::sw64(2 * q + 1, cc));
            float* dst = &s_bc[x][q][0];
            if constexpr (kBF16) {
                const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w}, w1[4] = {v1.x, v1.y, v1.z, v1.w};
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    *reinterpret_cast<float4*>(dst + 2 * (8 * cc + 2 * k)) =
                        make_float4(msc::bf16lo(w0[k]), msc::bf16lo(w1[k]), msc::bf16hi(w0[k]), msc::bf16hi(w1[k]));
            } else {
                *reinterpret_cast<float4*>(dst + 2 * (4 * cc)) =
                    make_float4(__uint_as_float(v0.x), __uint_as_float(v1.x), __uint_as_float(v0.y), __uint_as_float(v1.y));
                *reinterpret_cast<float4*>(dst + 2 * (4 * cc + 2)) =
                    make_float4(__uint_as_float(v0.z), __uint_as_float(v1.z), __uint_as_float(v0.w), __uint_as_float(v1.w));
            }
        }
        __syncthreads();

#pragma unroll 1
        for (int g = kGroups - 1; g >= 0; --g) {
            if (8 * g >= nt) continue;
            const int64_t tg = t0 + 8 * g;  // first step of the group
            // ---- this lane's two steps (8g + 2j, +1)
            const uint32_t boff = (uint32_t)((8 * g + 2 * j) * kES);
            float uu[2], dl[2], dyv[2], zv[2] = {0.f, 0.f};
            load2<kBF16>(raw, r, boff, uu[0], uu[1]);
            load2<kBF16>(raw + kRowTile, r, boff, dl[0], dl[1]);
            load2<kBF16>(raw + 2 * kRowTile, r, boff, dyv[0], dyv[1]);
            if (has_z) load2<kBF16>(raw + 3 * kRowTile, r, boff, zv[0], zv[1]);
            float mdt[2], mdtu[2], mgp[2], msx[2], msz[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float x = dl[e] + bias;
                mdt[e] = msc::softplus_f(x);
                msx[e] = sigmoid_acc(x);
                mdtu[e] = mdt[e] * uu[e];
                if (has_z) {
                    msz[e] = sigmoid_acc(zv[e]);
                    mgp[e] = dyv[e] * zv[e] * msz[e];
                } else {
                    msz[e] = 0.f;
                    mgp[e] = dyv[e];
                }
            }
            // ---- per-step scalars of all 8 steps from their owner lanes
            float dts[8], dtus[8], gps[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int src = glane0 | (k >> 1);
                dts[k] = __shfl_sync(0xffffffffu, mdt[k & 1], src);
                dtus[k] = __shfl_sync(0xffffffffu, mdtu[k & 1], src);
                gps[k] = __shfl_sync(0xffffffffu, mgp[k & 1], src);
            }
            // ---- recompute the group forward from its checkpoint
            uint64_t h[2];
            {
                const float4 hv = hv_next;
                if (row_ok && tg >= 8) hv_next = __ldg(reinterpret_cast<const float4*>(ck + (size_t)((tg - 8) >> 3) * 16));
                h[0] = msc::pk2(hv.x, hv.y);
                h[1] = msc::pk2(hv.z, hv.w);
            }
            uint64_t ah[8][2], hp[8][2];
            float yp[8];
            const float* bsrc = &s_bc[0][2 * j][16 * g];
            const float* csrc = &s_bc[1][2 * j][16 * g];
            // B pairs of all 8 steps, kept for the adjoint; C pairs of steps (k, k + 1)
            uint64_t Bs[8][2], Ck[2][2];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                if ((k & 1) == 0) {
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const ulonglong2 vb = *reinterpret_cast<const ulonglong2*>(bsrc + q * kPitch + 2 * k);
                        Bs[k][q] = vb.x; Bs[k + 1][q] = vb.y;
                    }
                }
                const uint64_t dt2 = msc::pk2(dts[k], dts[k]);
                const uint64_t dtu2 = msc::pk2(dtus[k], dtus[k]);
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const uint64_t a = msc::ex2_2(msc::mul2(dt2, A2p[q]));
                    ah[k][q] = a;
                    hp[k][q] = h[q];
                    h[q] = msc::fma2(a, h[q], msc::mul2(dtu2, Bs[k][q]));
                }
            }
            // ---- the adjoint, backwards through the group
            float s1[8], s2[8];
#pragma unroll
            for (int k = 7; k >= 0; --k) {
                if (k & 1) {
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const ulonglong2 vc = *reinterpret_cast<const ulonglong2*>(csrc + q * kPitch + 2 * (k - 1));
                        Ck[0][q] = vc.x; Ck[1][q] = vc.y;
                    }
                }
                const uint64_t dt2 = msc::pk2(dts[k], dts[k]);
                const uint64_t dtu2 = msc::pk2(dtus[k], dtus[k]);
                const uint64_t gp2 = msc::pk2(gps[k], gps[k]);
                uint64_t t1 = 0ull, t2 = 0ull, ysum = 0ull;
                uint64_t db[2], dc[2];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const uint64_t Bq = Bs[k][q];
                    const uint64_t Cq = Ck[k & 1][q];
                    // h_t of this step: the state entering the next step (h after the
                    // group for its last step); readout C h for dz, and dC_{t,n} = g'_t h_{t,n}
                    const uint64_t ht = (k < 7) ? hp[k + 1][q] : h[q];
                    ysum = q == 0 ? msc::mul2(Cq, ht) : msc::fma2(Cq, ht, ysum);
                    dc[q] = msc::mul2(gp2, ht);
                    const uint64_t anext = (k < 7) ? ah[k + 1][q] : a_carry[q];
                    lam[q] = msc::fma2(anext, lam[q], msc::mul2(gp2, Cq));
                    const uint64_t qh = msc::mul2(ah[k][q], hp[k][q]);  // abar_t h_{t-1}
                    t1 = q == 0 ? msc::mul2(lam[q], Bq) : msc::fma2(lam[q], Bq, t1);
                    const uint64_t lq = msc::mul2(lam[q], qh);
                    t2 = q == 0 ? msc::mul2(lq, Ap[q]) : msc::fma2(lq, Ap[q], t2);
                    dA2[q] = msc::fma2(lq, dt2, dA2[q]);
                    // dB_{t,n} contribution of this row: lambda_{t,n} Delta_t u_t
                    db[q] = msc::mul2(lam[q], dtu2);
                }
                {
                    // rows r and r ^ 1 (lanes 4 apart) add their halves here: the even
                    // row keeps states 4j, 4j + 1, the odd row 4j + 2, 4j + 3
                    const bool odd = (r & 1) != 0;
                    auto xch = [](uint64_t v) {
                        float a, c;
                        msc::upk2(v, a, c);
                        return msc::pk2(__shfl_xor_sync(0xffffffffu, a, 4), __shfl_xor_sync(0xffffffffu, c, 4));
                    };
                    const uint64_t rb = xch(odd ? db[0] : db[1]);
                    const uint64_t rc = xch(odd ? dc[0] : dc[1]);
                    const int o = red_pair(r >> 1) + 4 * j + 2 * (r & 1);
                    *reinterpret_cast<uint64_t*>(s_red + k * kRedBlock + o) = msc::add2(odd ? db[1] : db[0], rb);
                    *reinterpret_cast<uint64_t*>(s_red + (8 + k) * kRedBlock + o) = msc::add2(odd ? dc[1] : dc[0], rc);
                }
                float lo, hi;
                msc::upk2(ysum, lo, hi);
                yp[k] = lo + hi;
                msc::upk2(t1, lo, hi);
                s1[k] = lo + hi;
                msc::upk2(t2, lo, hi);
                s2[k] = lo + hi;
            }
            a_carry[0] = ah[0][0];
            a_carry[1] = ah[0][1];
            // ---- finish this lane's two steps: sums over the row's 16 states
            reduce_scatter8(yp, j);
            reduce_scatter8(s1, j);
            reduce_scatter8(s2, j);
            float o_du[2], o_dd[2], o_dz[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float ypv = yp[e] + Dd * uu[e];
                o_du[e] = mgp[e] * Dd + mdt[e] * s1[e];
                o_dd[e] = (uu[e] * s1[e] + s2[e]) * msx[e];
                o_dz[e] = has_z ? dyv[e] * ypv * msz[e] * (1.f + zv[e] * (1.f - msz[e])) : 0.f;
                dD_acc += mgp[e] * uu[e];
                dbias_acc += o_dd[e];
            }
            if (row_ok) {
                const size_t off = (size_t)row * p.L + tg + 2 * j;
                if (accumulate) {
                    const float2 a = *reinterpret_cast<const float2*>(p.du + off);
                    const float2 c = *reinterpret_cast<const float2*>(p.ddelta + off);
                    o_du[0] += a.x; o_du[1] += a.y;
                    o_dd[0] += c.x; o_dd[1] += c.y;
                    if (has_z) {
                        const float2 e = *reinterpret_cast<const float2*>(p.dz + off);
                        o_dz[0] += e.x; o_dz[1] += e.y;
                    }
                }
                *reinterpret_cast<float2*>(p.du + off) = make_float2(o_du[0], o_du[1]);
                *reinterpret_cast<float2*>(p.ddelta + off) = make_float2(o_dd[0], o_dd[1]);
                if (has_z) *reinterpret_cast<float2*>(p.dz + off) = make_float2(o_dz[0], o_dz[1]);
            }
            __syncthreads();
            // ---- dB, dC of this group: sum the CTA's 16 row pairs (thread = (x, k, 4 states, half of the pairs)),
            // transpose through s_sum, one vector add per 4 steps
            {
                const int half = tid & 1, n4 = (tid >> 1) & 3, k = (tid >> 3) & 7, x = tid >> 6;
                const float* src = s_red + (8 * x + k) * kRedBlock + red_pair(8 * half) + 4 * n4;
                uint64_t a01 = 0ull, a23 = 0ull;
#pragma unroll
                for (int rr = 0; rr < 8; ++rr) {
                    const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(src + 16 * rr);
                    a01 = msc::add2(a01, v.x);
                    a23 = msc::add2(a23, v.y);
                }
                float s4[4];
                msc::upk2(a01, s4[0], s4[1]);
                msc::upk2(a23, s4[2], s4[3]);
#pragma unroll
                for (int e = 0; e < 4; ++e) s4[e] += __shfl_xor_sync(0xffffffffu, s4[e], 1);
                if (half == 0) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) s_sum[(16 * x + 4 * n4 + e) * kSumPitch + k] = s4[e];
                }
            }
            __syncthreads();
            if (tid < 64) {
                const int x = tid >> 5, n = (tid >> 1) & 15, kq = tid & 1;
                const float4 v = *reinterpret_cast<const float4*>(s_sum + (16 * x + n) * kSumPitch + 4 * kq);
                if (n < N) {
                    float* dst = (x == 0 ? p.dB : p.dC) + ((size_t)b * bc_rows + n) * p.L + tg + 4 * kq;
                    red_add_v4(dst, v.x, v.y, v.z, v.w);
                }
            }
            __syncthreads();
        }
        if (tid == 0 && issued < ntiles) issue(issued);
        ++issued;
    }

    if (failed) {
        if (tid == 0)
            for (int cc = c; cc < issued && cc < ntiles; ++cc)
                (void)msc::wait_bounded(&s_full[cc % kStages], (uint32_t)((cc / kStages) & 1));
        return;
    }
    // per-channel sums: dA over this row's states, dD and dbias over its steps
    dD_acc += __shfl_xor_sync(0xffffffffu, dD_acc, 1);
    dD_acc += __shfl_xor_sync(0xffffffffu, dD_acc, 2);
    dbias_acc += __shfl_xor_sync(0xffffffffu, dbias_acc, 1);
    dbias_acc += __shfl_xor_sync(0xffffffffu, dbias_acc, 2);
    if (!row_ok) return;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        float v0, v1;
        msc::upk2(dA2[q], v0, v1);
        const int n = 4 * j + 2 * q;
        if (n < N) atomicAdd(p.dA + d * N + n, v0);
        if (n + 1 < N) atomicAdd(p.dA + d * N + n + 1, v1);
    }
    if (j == 0) {
        if (p.dD && first) atomicAdd(p.dD + d, dD_acc);
        if (p.dbias) atomicAdd(p.dbias + d, dbias_acc);
    }
}

template <bool kBF16>
constexpr int bwd_smem_bytes() {
    return 1024 + kStages * kStageBytes + 2 * 8 * (2 * (kBF16 ? 32 : 16) + 4) * 4 + 2 * 8 * kRedBlock * 4 +
           2 * 16 * kSumPitch * 4 + kStages * 8;
}

template <bool kBF16, bool kSlice>
msc_status launch_bwd(const CUtensorMap* maps, const BwdParams& p, const BwdSlice& sl, int64_t batch,
                      cudaStream_t st) {
    constexpr int smem = bwd_smem_bytes<kBF16>();
    static std::atomic<uint64_t> configured{0};  // the attribute, set once per device (per instantiation)
    if (!(configured & msc_host::device_bit())) {
        cudaError_t e = cudaFuncSetAttribute(s6_bwd_kernel<kBF16, kSlice>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return msc_host::fail(MSC_ERR_CUDA, "s6_bwd smem attribute: %s", cudaGetErrorString(e));
        configured |= msc_host::device_bit();
    }
    dim3 grid((unsigned)((p.dim + kRows - 1) / kRows), (unsigned)batch, 1);
    s6_bwd_kernel<kBF16, kSlice><<<grid, kThreads, smem, st>>>(maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], p,
                                                                sl);
    return msc_host::check_launch("s6_bwd");
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

namespace msc_host {

// Rows whose byte stride is not a multiple of 16 are copied into a padded
// layout (zero tail) inside the workspace; the kernels then run on the copy.
static int64_t padded_len(int64_t L, bool bf16) {
    const int64_t m = 8;  // a multiple of 8 steps keeps both dtypes 16-byte aligned
    (void)bf16;
    return (L + m - 1) / m * m;
}

size_t s6_bwd_workspace(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate) {
    const int64_t rows = batch * dim;
    const int64_t Lp = padded_len(seqlen, true);
    size_t ws = align256((size_t)rows * (size_t)((Lp + 7) / 8) * 16 * sizeof(float));  // checkpoints (one slice)
    if (dstate > 16) ws += 2 * align256((size_t)dim * 16 * sizeof(float));             // A and dA of a slice
    if (Lp != seqlen) {
        // padded copies: u, delta, z, dy (4 bytes is the larger element) and
        // du, ddelta, dz; B, C, dB, dC
        ws += 7 * align256((size_t)rows * Lp * 4) + 4 * align256((size_t)batch * dstate * Lp * 4);
    }
    return ws;
}

// rows_per_b rows of L steps per batch entry, stride_rows rows apart (0: rows_per_b)
static msc_status make_row_map(CUtensorMap* m, const void* base, bool bf16, int64_t L, int64_t rows_per_b,
                               int64_t batch, uint32_t box_rows, int64_t stride_rows = 0) {
    const uint64_t es = bf16 ? 2 : 4;
    const uint64_t dims[3] = {(uint64_t)L, (uint64_t)rows_per_b, (uint64_t)batch};
    const uint64_t str[2] = {(uint64_t)L * es, (uint64_t)(stride_rows ? stride_rows : rows_per_b) * L * es};
    const uint32_t box[3] = {bf16 ? 32u : 16u, box_rows, 1};
    return encode_tmap(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims,
                       str, box, CU_TENSOR_MAP_SWIZZLE_64B)
               ? MSC_OK
               : MSC_ERR_CUDA;
}

static msc_status pad_copy(void* dst, const void* src, size_t es, int64_t rows, int64_t L, int64_t Lp,
                           cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(dst, 0, (size_t)rows * Lp * es, st);
    if (e == cudaSuccess)
        e = cudaMemcpy2DAsync(dst, Lp * es, src, L * es, L * es, rows, cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) return fail(MSC_ERR_CUDA, "padding copy: %s", cudaGetErrorString(e));
    return MSC_OK;
}

static msc_status unpad_copy(void* dst, const void* src, size_t es, int64_t rows, int64_t L, int64_t Lp,
                             cudaStream_t st) {
    cudaError_t e = cudaMemcpy2DAsync(dst, L * es, src, Lp * es, L * es, rows, cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) return fail(MSC_ERR_CUDA, "unpadding copy: %s", cudaGetErrorString(e));
    return MSC_OK;
}

msc_status s6_bwd_launch(const S6BwdArgs& a0, cudaStream_t st) {
    S6BwdArgs a = a0;
    const int64_t rows = a.batch * a.dim;
    const int64_t L = a.L;
    const int64_t Lp = padded_len(L, a.bf16);
    // the tiles' TMA coordinates (step, row) are signed 32-bit: refuse before any device work
    constexpr int64_t kMaxCoord = ((int64_t)1 << 31) - 64;
    if (Lp > kMaxCoord || a.dim > kMaxCoord)
        return fail(MSC_ERR_UNSUPPORTED, "the backward needs seqlen and dim below 2^31");
    const size_t es = a.bf16 ? 2 : 4;
    if (a.ckpt_in && Lp != L) return fail(MSC_ERR_UNSUPPORTED, "checkpoints need seqlen a multiple of 8");
    char* ws = static_cast<char*>(a.workspace);
    const float* ckpt = a.ckpt_in;
    if (!ckpt) {
        ckpt = reinterpret_cast<float*>(ws);
        ws += align256((size_t)rows * (size_t)((Lp + 7) / 8) * 16 * sizeof(float));
    }

    // outputs that are sums start at zero
    cudaError_t e = cudaSuccess;
    if (Lp == L) {
        e = cudaMemsetAsync(a.dB, 0, (size_t)a.batch * a.N * L * sizeof(float), st);
        if (e == cudaSuccess) e = cudaMemsetAsync(a.dC, 0, (size_t)a.batch * a.N * L * sizeof(float), st);
    }
    if (e == cudaSuccess) e = cudaMemsetAsync(a.dA, 0, (size_t)a.dim * a.N * sizeof(float), st);
    if (e == cudaSuccess && a.dD) e = cudaMemsetAsync(a.dD, 0, (size_t)a.dim * sizeof(float), st);
    if (e == cudaSuccess && a.ddelta_bias) e = cudaMemsetAsync(a.ddelta_bias, 0, (size_t)a.dim * sizeof(float), st);
    if (e != cudaSuccess) return fail(MSC_ERR_CUDA, "zeroing gradients: %s", cudaGetErrorString(e));

    // padded copies for rows whose stride TMA cannot describe
    const void *u = a.u, *dl = a.delta, *z = a.z, *dy = a.dy, *B = a.B, *C = a.C;
    float *du = a.du, *ddl = a.ddelta, *dz = a.dz, *dB = a.dB, *dC = a.dC;
    // A and dA of one slice of 16 states (more than 16 states)
    const int nslices = (a.N + 15) / 16;
    float* A_s = nullptr;
    float* dA_s = nullptr;
    if (nslices > 1) {
        if (a.ckpt_in) return fail(MSC_ERR_UNSUPPORTED, "kept checkpoints are for up to 16 states");
        A_s = reinterpret_cast<float*>(ws); ws += align256((size_t)a.dim * 16 * sizeof(float));
        dA_s = reinterpret_cast<float*>(ws); ws += align256((size_t)a.dim * 16 * sizeof(float));
    }
    if (Lp != L) {
        const size_t rbytes = align256((size_t)rows * Lp * 4), bbytes = align256((size_t)a.batch * a.N * Lp * 4);
        void* pu = ws; ws += rbytes;
        void* pd = ws; ws += rbytes;
        void* pz = ws; ws += rbytes;
        void* pdy = ws; ws += rbytes;
        float* pdu = reinterpret_cast<float*>(ws); ws += rbytes;
        float* pdd = reinterpret_cast<float*>(ws); ws += rbytes;
        float* pdz = reinterpret_cast<float*>(ws); ws += rbytes;
        void* pB = ws; ws += bbytes;
        void* pC = ws; ws += bbytes;
        float* pdB = reinterpret_cast<float*>(ws); ws += bbytes;
        float* pdC = reinterpret_cast<float*>(ws); ws += bbytes;
        msc_status s;
        if ((s = pad_copy(pu, u, es, rows, L, Lp, st)) != MSC_OK) return s;
        if ((s = pad_copy(pd, dl, es, rows, L, Lp, st)) != MSC_OK) return s;
        if ((s = pad_copy(pdy, dy, es, rows, L, Lp, st)) != MSC_OK) return s;
        if (z && (s = pad_copy(pz, z, es, rows, L, Lp, st)) != MSC_OK) return s;
        if ((s = pad_copy(pB, B, es, a.batch * a.N, L, Lp, st)) != MSC_OK) return s;
        if ((s = pad_copy(pC, C, es, a.batch * a.N, L, Lp, st)) != MSC_OK) return s;
        e = cudaMemsetAsync(pdB, 0, (size_t)a.batch * a.N * Lp * sizeof(float), st);
        if (e == cudaSuccess) e = cudaMemsetAsync(pdC, 0, (size_t)a.batch * a.N * Lp * sizeof(float), st);
        if (e != cudaSuccess) return fail(MSC_ERR_CUDA, "zeroing gradients: %s", cudaGetErrorString(e));
        u = pu; dl = pd; dy = pdy; z = z ? pz : nullptr; B = pB; C = pC;
        du = pdu; ddl = pdd; dz = a.dz ? pdz : nullptr; dB = pdB; dC = pdC;
    }

    // Per slice of up to 16 states: (1) the states entering every 8-step group
    // (unless the training forward kept them), (2) the reverse pass.
    msc_status s = MSC_OK;
    for (int sl = 0; sl < nslices; ++sl) {
        const int n0 = 16 * sl, ns = a.N - n0 < 16 ? a.N - n0 : 16;
        const float* A = a.A;
        float* dA = a.dA;
        const void* Bs = static_cast<const char*>(B) + (size_t)n0 * Lp * es;
        const void* Cs = static_cast<const char*>(C) + (size_t)n0 * Lp * es;
        if (nslices > 1) {
            e = cudaMemcpy2DAsync(A_s, ns * sizeof(float), a.A + n0, a.N * sizeof(float), ns * sizeof(float),
                                  a.dim, cudaMemcpyDeviceToDevice, st);
            if (e == cudaSuccess) e = cudaMemsetAsync(dA_s, 0, (size_t)a.dim * ns * sizeof(float), st);
            if (e != cudaSuccess) return fail(MSC_ERR_CUDA, "state slice: %s", cudaGetErrorString(e));
            A = A_s;
            dA = dA_s;
        }
        if (!a.ckpt_in) {
            S6FwdArgs f{};
            f.batch = a.batch; f.dim = a.dim; f.L = Lp; f.N = ns; f.bf16 = a.bf16;
            f.u = u; f.delta = dl; f.B = Bs; f.C = Cs; f.A = A; f.delta_bias = a.delta_bias;
            f.bc_rows = a.N;
            s = s6_fwd_checkpoints(f, const_cast<float*>(ckpt), st);
            if (s != MSC_OK) return s;
        }
        CUtensorMap maps[6];
        if ((s = make_row_map(&maps[0], u, a.bf16, Lp, a.dim, a.batch, kRows)) != MSC_OK) return s;
        if ((s = make_row_map(&maps[1], dl, a.bf16, Lp, a.dim, a.batch, kRows)) != MSC_OK) return s;
        if ((s = make_row_map(&maps[2], z ? z : u, a.bf16, Lp, a.dim, a.batch, kRows)) != MSC_OK) return s;
        if ((s = make_row_map(&maps[3], dy, a.bf16, Lp, a.dim, a.batch, kRows)) != MSC_OK) return s;
        if ((s = make_row_map(&maps[4], Bs, a.bf16, Lp, ns, a.batch, 16, a.N)) != MSC_OK) return s;
        if ((s = make_row_map(&maps[5], Cs, a.bf16, Lp, ns, a.batch, 16, a.N)) != MSC_OK) return s;
        BwdParams p{};
        p.A = A; p.D = a.D; p.delta_bias = a.delta_bias; p.ckpt = ckpt;
        p.du = du; p.ddelta = ddl; p.dz = dz; p.dA = dA; p.dB = dB + (size_t)n0 * Lp; p.dC = dC + (size_t)n0 * Lp;
        p.dD = a.dD; p.dbias = a.ddelta_bias;
        p.dim = a.dim; p.L = Lp; p.ckpt_groups = (Lp + 7) / 8; p.N = ns; p.has_z = z != nullptr;
        BwdSlice sp{};
        sp.bc_rows = a.N; sp.first = sl == 0; sp.accumulate = sl > 0;
        if (nslices > 1)
            s = a.bf16 ? launch_bwd<true, true>(maps, p, sp, a.batch, st) : launch_bwd<false, true>(maps, p, sp, a.batch, st);
        else
            s = a.bf16 ? launch_bwd<true, false>(maps, p, sp, a.batch, st)
                       : launch_bwd<false, false>(maps, p, sp, a.batch, st);
        if (s != MSC_OK) return s;
        if (nslices > 1) {
            e = cudaMemcpy2DAsync(a.dA + n0, a.N * sizeof(float), dA_s, ns * sizeof(float), ns * sizeof(float),
                                  a.dim, cudaMemcpyDeviceToDevice, st);
            if (e != cudaSuccess) return fail(MSC_ERR_CUDA, "state slice: %s", cudaGetErrorString(e));
        }
    }
    if (Lp != L) {
        if ((s = unpad_copy(a.du, du, 4, rows, L, Lp, st)) != MSC_OK) return s;
        if ((s = unpad_copy(a.ddelta, ddl, 4, rows, L, Lp, st)) != MSC_OK) return s;
        if (a.dz && (s = unpad_copy(a.dz, dz, 4, rows, L, Lp, st)) != MSC_OK) return s;
        if ((s = unpad_copy(a.dB, dB, 4, a.batch * a.N, L, Lp, st)) != MSC_OK) return s;
        if ((s = unpad_copy(a.dC, dC, 4, a.batch * a.N, L, Lp, st)) != MSC_OK) return s;
    }
    return MSC_OK;
}

msc_status s6_bwd_take_status(unsigned int* code, unsigned int* site) {
    unsigned int w[2] = {0, 0};
    cudaError_t e = cudaMemcpyFromSymbol(w, g_s6_bwd_status, sizeof(w));
    if (e != cudaSuccess) return fail(MSC_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
    if (w[0] != 0) {
        const unsigned int zz[2] = {0, 0};
        e = cudaMemcpyToSymbol(g_s6_bwd_status, zz, sizeof(zz));
        if (e != cudaSuccess) return fail(MSC_ERR_CUDA, "status clear: %s", cudaGetErrorString(e));
    }
    *code = w[0];
    *site = w[1];
    return MSC_OK;
}

}  // namespace msc_host
