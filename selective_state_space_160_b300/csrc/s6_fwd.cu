// s6_fwd.cu -- S6 selective-scan forward on sm_103a.
//
// What it computes (per channel row (b, d), t = 0..L-1, n < N):
//   Delta_t = softplus(delta_t + Delta_bias[d])          selection, bqwf survey sec. 2.2
//   abar    = exp(Delta_t A[d,n]);  h_n = abar h_n + Delta_t B[b,n,t] u_t
//                                                         exponential-Euler, Mamba 解密 sec. 6.3
//   y_t     = (sum_n C[b,n,t] h_n + D[d] u_t) * silu(z_t)  readout + gate, Mamba 解密 sec. 3
//
// Design ("row-resident" scan).  The recurrence is sequential in t and the
// selection makes it time-varying, so it is run as a sequential loop in which
// one lane owns one channel row and keeps all N (<= 16) fp32 states in
// registers.  Per (t, n) this costs one MUFU ex2 (exp(Delta A) as
// ex2(Delta * A log2 e)) and four FP32 ops -- no scan overhead at all.  Rows
// give the parallelism (b * dim rows); a CTA is 32 rows of one batch entry
// (two lanes per row: 64 threads), stepping through time in tiles of 64-byte
// rows (32 bf16 or 16 fp32 steps).
//
// Main kernel (s6_fwd_tma_kernel): one thread issues 3-D TMA tile loads of
// u / delta / z (32 rows x one tile) and B / C (16 slots x one tile, shared by
// the warp's rows) into a two-stage shared-memory ring completed on mbarriers,
// so the next tile streams in while the current one is computed.  Out-of-range
// rows, slots and steps arrive zero-filled.  Two lanes share a row (8 states
// each); each computes Delta, Delta*u and D*u for half of an 8-step group
// (softplus on packed pairs) and gathers the other half with shuffles, then
// runs the n loop on packed fp32 pairs (fma.rn.f32x2: two states per issue
// slot) with B / C converted once per tile into an n-pair-interleaved fp32
// layout (each pair is one 64-bit broadcast operand).  The readout partial sums
// are reduce-scattered between the pair and y is stored from registers; rows of
// 2^19 steps or more stage y in shared memory instead and write each row's
// 32-step window as one 128-byte run (kLongRows).  A tile takes two CTA
// barriers with 16 state slots (the wait's vote with the end of the B/C
// conversion, and the tile's end before its stage is refilled) and one with
// more slots (the next tile issued at the first).
// Rows whose byte stride is not a multiple of 16 cannot be described to TMA;
// they take the plain-load kernel (s6_fwd_rows_kernel), which stages each tile
// with coalesced loads and computes the same way in scalar fp32.
//
// Enough rows to fill the GPU: the 32-row blocks run on persistent CTAs (at
// most one per row block) that take (row block, chunk) items in chunk-major
// order from a ticket counter.  Chunk c of a block starts from the state chunk
// c - 1 left in the workspace, once that chunk's flag (release / acquire, a
// bounded wait) says it is there; the predecessor was taken a full round of
// tickets earlier, so it is normally finished.  A block's chunks thus run on
// different SMs, which evens out the load that a fixed grid leaves uneven
// (1280 blocks on 148 SMs: some schedulers hold five warps, the average 4.3).
//
// Few rows and a long sequence (b * dim too small to fill 148 SMs) split each
// row into G segments: an aggregate pass computes, from a zero state, each
// segment's end state and sum of Delta (segment decay exp(A sum Delta)); a tiny
// carry pass chains them (h_in(g+1) = exp(A sum Delta_g) h_in(g) + H_g); the
// full pass then runs every segment from its carry.  The chained operator is
// the scan composition (a, b) o (a', b') = (a a', a' b + b') of the
// associative parallel scan (study note: Blelloch's work-efficient scan).
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>

#include "msc_common.cuh"
#include "msc_internal.h"
#include "msc_tma.cuh"

namespace {

constexpr int kRows = 32;  // channel rows per CTA (one per lane)
constexpr int kT = 32;     // timesteps per staged tile
constexpr int kNS = 16;    // state slots of the plain-load kernel, the checkpoints and the fused conv
constexpr int kStride = kT + 4;

// State slots of a row in the TMA forward: 16, 32 or 64 (dstate <= 64).
inline int state_slots(int64_t N) { return N <= 16 ? 16 : N <= 32 ? 32 : 64; }

// Full: y (and h_last); Agg: segment end states and Delta sums; Ckpt: the
// state entering every 8-step group only; FullCkpt: y and those states.
enum { kModeFull = 0, kModeAgg = 1, kModeCkpt = 2, kModeFullCkpt = 3 };
// input-term discretisation (values of msc_discretization)
enum { kDiscEuler = 0, kDiscZoh = 1, kDiscTrap = 2 };

__device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }

struct FwdParams {
    const void* u;
    const void* delta;
    const void* z;
    const void* B;
    const void* C;
    const float* A;
    const float* D;
    const float* delta_bias;
    const float* h0;
    float* y;
    float* h_last;
    float* seg_state;  // [rows, G, N]: aggregates, then carries
    float* seg_dsum;   // [rows, G]
    float* ckpt;       // [rows, ckpt_groups, 16]: state at every 8-step group start
    int64_t ckpt_groups;
    const float* conv_w;  // fused front end: [dim, conv_k] causal conv taps (u then holds its input x)
    const float* conv_b;  // [dim] or null
    int conv_k;
    int64_t dim, L, seg_len;
    int N, G;
    // chained schedule (full pass only): persistent CTAs take (row block, chunk)
    // items from a ticket counter; chunk q > 0 starts from the state chunk q - 1
    // left in chain_state once flags[block] says q chunks are done
    unsigned long long* ctr;  // ticket counter (null: one item per CTA from blockIdx)
    unsigned* flags;          // [chains] finished chunks per row block
    float* chain_state;       // [batch * dim, 16]
    unsigned* abort_word;     // set by a CTA whose wait ran out, so that the others stop waiting
    int64_t chunk, nblk, chains, total_items;
    int chained;
};

// Stage a [kRows x kT] tile of a [rows, L] tensor (rows d0.. of batch entry b),
// timesteps t0 .. t0 + nt - 1, as fp32 into dst[row][t] (zeros outside).
template <bool kBF16, bool kVec>
__device__ __forceinline__ void stage_rows(float (*dst)[kStride], const void* src, int64_t row0,
                                           int nrows, int64_t L, int64_t t0, int nt, int lane) {
    if constexpr (kVec) {
        // 32 rows x 4 segments of 8 steps; 4 segments per lane.
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            int s = lane + 32 * i;
            int r = s >> 2, tt = (s & 3) * 8;
            float v[8];
            if (r < nrows && tt + 8 <= nt) {
                msc::ld8<kBF16>(src, (row0 + r) * L + t0 + tt, v);
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    v[k] = (r < nrows && tt + k < nt) ? msc::ld_elem<kBF16>(src, (row0 + r) * L + t0 + tt + k) : 0.f;
            }
            *reinterpret_cast<float4*>(&dst[r][tt]) = make_float4(v[0], v[1], v[2], v[3]);
            *reinterpret_cast<float4*>(&dst[r][tt + 4]) = make_float4(v[4], v[5], v[6], v[7]);
        }
    } else {
        for (int e = lane; e < kRows * kT; e += 32) {
            int r = e / kT, tt = e % kT;
            dst[r][tt] = (r < nrows && tt < nt) ? msc::ld_elem<kBF16>(src, (row0 + r) * L + t0 + tt) : 0.f;
        }
    }
}

// Stage B or C of batch entry b ([N, L] slice) transposed into dst[t][n].
template <bool kBF16, bool kVec>
__device__ __forceinline__ void stage_bc(float (*dst)[kNS], const void* src, int64_t b, int N,
                                         int64_t L, int64_t t0, int nt, int lane) {
    const int64_t base = b * (int64_t)N * L;
    if constexpr (kVec) {
        // 16 slots x 4 segments of 8 steps; 2 segments per lane.
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            int s = lane + 32 * i;
            int n = s >> 2, tt = (s & 3) * 8;
            float v[8];
            if (n < N && tt + 8 <= nt) {
                msc::ld8<kBF16>(src, base + n * L + t0 + tt, v);
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    v[k] = (n < N && tt + k < nt) ? msc::ld_elem<kBF16>(src, base + n * L + t0 + tt + k) : 0.f;
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) dst[tt + k][n] = v[k];
        }
    } else {
        for (int e = lane; e < kNS * kT; e += 32) {
            int n = e / kT, tt = e % kT;
            dst[tt][n] = (n < N && tt < nt) ? msc::ld_elem<kBF16>(src, base + n * L + t0 + tt) : 0.f;
        }
    }
}

template <bool kVec>
__device__ __forceinline__ void store_rows(float* dst, float (*src)[kStride], int64_t row0, int nrows,
                                           int64_t L, int64_t t0, int nt, int lane) {
    if constexpr (kVec) {
        // 32 rows x 8 segments of 4 steps; 8 segments per lane.
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            int s = lane + 32 * i;
            int r = s >> 3, tt = (s & 7) * 4;
            if (r >= nrows) continue;
            float4 v = *reinterpret_cast<const float4*>(&src[r][tt]);
            float* q = dst + (row0 + r) * L + t0 + tt;
            if (tt + 4 <= nt) {
                __stcs(reinterpret_cast<float4*>(q), v);
            } else {
                if (tt + 0 < nt) q[0] = v.x;
                if (tt + 1 < nt) q[1] = v.y;
                if (tt + 2 < nt) q[2] = v.z;
            }
        }
    } else {
        for (int e = lane; e < kRows * kT; e += 32) {
            int r = e / kT, tt = e % kT;
            if (r < nrows && tt < nt) dst[(row0 + r) * L + t0 + tt] = src[r][tt];
        }
    }
}

template <bool kBF16, bool kVec, int kMode, int kDisc = kDiscEuler, bool kConv = false>
__global__ void __launch_bounds__(32) s6_fwd_rows_kernel(const FwdParams p) {
    __shared__ __align__(16) float s_u[kRows][kStride];
    __shared__ __align__(16) float s_d[kRows][kStride];  // delta in, y out
    __shared__ __align__(16) float s_z[kRows][kStride];
    __shared__ __align__(16) float s_B[kT][kNS];
    __shared__ __align__(16) float s_C[kT][kNS];

    constexpr bool kFull = (kMode == kModeFull);
    const int lane = threadIdx.x;
    const int64_t b = blockIdx.y;
    const int64_t d0 = (int64_t)blockIdx.x * kRows;
    const int nrows = (int)imin64(kRows, p.dim - d0);
    const int64_t d = d0 + lane;
    const bool row_ok = lane < nrows;
    const int64_t row = b * p.dim + (row_ok ? d : d0);
    const int seg = blockIdx.z;
    const int N = p.N;
    const bool has_z = kFull && p.z != nullptr;

    float A2[kNS], h[kNS];
#pragma unroll
    for (int n = 0; n < kNS; ++n) {
        A2[n] = (row_ok && n < N) ? __ldg(p.A + d * N + n) * MSC_LOG2E : 0.f;
        float h_init = 0.f;
        if (kFull && row_ok && n < N) {
            if (p.G > 1)
                h_init = p.seg_state[((size_t)row * p.G + seg) * N + n];
            else if (p.h0)
                h_init = __ldg(p.h0 + row * N + n);
        }
        h[n] = h_init;
    }
    const float Dd = (kFull && p.D && row_ok) ? __ldg(p.D + d) : 0.f;
    const float bias = (p.delta_bias && row_ok) ? __ldg(p.delta_bias + d) : 0.f;
    float dsum = 0.f;

    const int64_t t_begin = (int64_t)seg * p.seg_len;
    const int64_t t_end = imin64(p.L, t_begin + p.seg_len);
    const int64_t row0 = b * p.dim + d0;

    // fused conv front end: taps right-aligned in a 4-tap window (cw[m] multiplies
    // x_{t-3+m}) and the three inputs before the current step (0 before t = 0);
    // the staged u tile then holds x, and u = silu(conv) is formed step by step
    float cw[4] = {0.f, 0.f, 0.f, 0.f}, cbias = 0.f, xw[3] = {0.f, 0.f, 0.f};
    if constexpr (kConv) {
        const int K = p.conv_k;
#pragma unroll
        for (int m = 0; m < 4; ++m) cw[m] = (row_ok && m + K >= 4) ? __ldg(p.conv_w + d * K + (m + K - 4)) : 0.f;
        cbias = (row_ok && p.conv_b) ? __ldg(p.conv_b + d) : 0.f;
#pragma unroll
        for (int m = 0; m < 3; ++m) {
            const int64_t tp = t_begin - 3 + m;
            xw[m] = (row_ok && tp >= 0) ? msc::ld_elem<kBF16>(p.u, row * p.L + tp) : 0.f;
        }
    }
    // zero-order hold: 1/A per state (0 where A = 0: the series branch covers it);
    // trapezoid: the half input term of the previous step, per state (from the
    // step before the segment, none before t = 0)
    float invA[kDisc == kDiscZoh ? kNS : 1];
    float ep[kDisc == kDiscTrap ? kNS : 1];
    if constexpr (kDisc == kDiscZoh) {
#pragma unroll
        for (int n = 0; n < kNS; ++n) {
            const float a = A2[n] * MSC_LN2;
            invA[n] = a != 0.f ? 1.f / a : 0.f;
        }
    }
    if constexpr (kDisc == kDiscTrap) {
        float eu = 0.f;
        if (row_ok && t_begin > 0) {
            const int64_t tp = t_begin - 1;
            eu = 0.5f * msc::softplus_f(msc::ld_elem<kBF16>(p.delta, row * p.L + tp) + bias) *
                 msc::ld_elem<kBF16>(p.u, row * p.L + tp);
        }
#pragma unroll
        for (int n = 0; n < kNS; ++n)
            ep[n] = (eu != 0.f && n < N) ? eu * msc::ld_elem<kBF16>(p.B, (b * N + n) * p.L + t_begin - 1) : 0.f;
    }

    for (int64_t t0 = t_begin; t0 < t_end; t0 += kT) {
        const int nt = (int)imin64(kT, t_end - t0);
        __syncwarp();
        stage_rows<kBF16, kVec>(s_u, p.u, row0, nrows, p.L, t0, nt, lane);
        stage_rows<kBF16, kVec>(s_d, p.delta, row0, nrows, p.L, t0, nt, lane);
        if (has_z) stage_rows<kBF16, kVec>(s_z, p.z, row0, nrows, p.L, t0, nt, lane);
        stage_bc<kBF16, kVec>(s_B, p.B, b, N, p.L, t0, nt, lane);
        if (kFull) stage_bc<kBF16, kVec>(s_C, p.C, b, N, p.L, t0, nt, lane);
        __syncwarp();

        for (int tq = 0; tq < nt; tq += 4) {
            const float4 u4 = *reinterpret_cast<const float4*>(&s_u[lane][tq]);
            const float4 d4 = *reinterpret_cast<const float4*>(&s_d[lane][tq]);
            float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
            if (has_z) z4 = *reinterpret_cast<const float4*>(&s_z[lane][tq]);
            float uu[4] = {u4.x, u4.y, u4.z, u4.w};
            const float dd[4] = {d4.x, d4.y, d4.z, d4.w};
            if constexpr (kConv) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if (tq + k < nt) {
                        const float x = uu[k];
                        float acc = cbias;
                        acc = fmaf(cw[0], xw[0], acc);
                        acc = fmaf(cw[1], xw[1], acc);
                        acc = fmaf(cw[2], xw[2], acc);
                        acc = fmaf(cw[3], x, acc);
                        uu[k] = msc::silu_f(acc);
                        xw[0] = xw[1];
                        xw[1] = xw[2];
                        xw[2] = x;
                    }
                }
            }
            const float zz[4] = {z4.x, z4.y, z4.z, z4.w};
            float yy[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                yy[k] = 0.f;
                if (tq + k < nt) {
                    const int t = tq + k;
                    const float dt = msc::softplus_f(dd[k] + bias);
                    const float dtu = kDisc == kDiscTrap ? 0.5f * dt * uu[k] : dt * uu[k];
                    const float rdt = kDisc == kDiscZoh ? (dt > 0.f ? msc::rcp_approx(dt) : 0.f) : 0.f;
                    if (!kFull) dsum += dt;
                    float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
#pragma unroll
                    for (int q = 0; q < kNS / 4; ++q) {
                        const float4 bq = *reinterpret_cast<const float4*>(&s_B[t][4 * q]);
                        const float bv[4] = {bq.x, bq.y, bq.z, bq.w};
                        float cv[4] = {0.f, 0.f, 0.f, 0.f};
                        if (kFull) {
                            const float4 cq = *reinterpret_cast<const float4*>(&s_C[t][4 * q]);
                            cv[0] = cq.x; cv[1] = cq.y; cv[2] = cq.z; cv[3] = cq.w;
                        }
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int n = 4 * q + j;
                            const float arg = dt * A2[n];
                            const float a = msc::ex2_approx(arg);
                            if constexpr (kDisc == kDiscEuler) {
                                h[n] = fmaf(a, h[n], dtu * bv[j]);
                            } else if constexpr (kDisc == kDiscZoh) {
                                // phi = (e^x - 1) / x with x = Delta A: a series near 0
                                const float x = arg * MSC_LN2;
                                float ps = fmaf(x, 1.f / 24.f, 1.f / 6.f);
                                ps = fmaf(x, ps, 0.5f);
                                ps = fmaf(x, ps, 1.f);
                                const float phi = fabsf(x) < 0.03f ? ps : (a - 1.f) * invA[n] * rdt;
                                h[n] = fmaf(a, h[n], phi * (dtu * bv[j]));
                            } else {
                                const float e2 = dtu * bv[j];  // half the Euler term
                                h[n] = fmaf(a, h[n] + ep[n], e2);
                                ep[n] = e2;
                            }
                            if (kFull) {
                                if (j == 0) acc0 = fmaf(cv[j], h[n], acc0);
                                if (j == 1) acc1 = fmaf(cv[j], h[n], acc1);
                                if (j == 2) acc2 = fmaf(cv[j], h[n], acc2);
                                if (j == 3) acc3 = fmaf(cv[j], h[n], acc3);
                            }
                        }
                    }
                    if (kFull) {
                        float yv = (acc0 + acc1) + (acc2 + acc3) + Dd * uu[k];
                        if (has_z) yv *= msc::silu_f(zz[k]);
                        yy[k] = yv;
                    }
                }
            }
            if (kFull) *reinterpret_cast<float4*>(&s_d[lane][tq]) = make_float4(yy[0], yy[1], yy[2], yy[3]);
        }
        if (kFull) {
            __syncwarp();
            store_rows<kVec>(p.y, s_d, row0, nrows, p.L, t0, nt, lane);
        }
    }

    if (!row_ok) return;
    if (kFull) {
        if (p.h_last && seg == p.G - 1) {
#pragma unroll
            for (int n = 0; n < kNS; ++n)
                if (n < N) p.h_last[row * N + n] = h[n];
        }
    } else {
#pragma unroll
        for (int n = 0; n < kNS; ++n)
            if (n < N) p.seg_state[((size_t)row * p.G + seg) * N + n] = h[n];
        p.seg_dsum[(size_t)row * p.G + seg] = dsum;
    }
}


// --------------------------------------------------------------------------
// Device status word of this module: (code, site) of the first bounded wait
// that ran out.  Read and cleared by msc_check_device_status().
__device__ unsigned int g_s6_fwd_status[2];

__device__ __forceinline__ void record_timeout(unsigned int site) {
    if (atomicCAS(&g_s6_fwd_status[0], 0u, (unsigned int)MSC_ERR_TIMEOUT) == 0u)
        g_s6_fwd_status[1] = site;
}

// Wait until *flag >= target (acquire), about one second at most by the global
// timer; gives up early once another CTA of the launch has given up.
__device__ __forceinline__ bool wait_flag_geq(const unsigned* flag, unsigned target, const volatile unsigned* abort) {
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        unsigned v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
        if (v >= target) return true;
        if (i >= 16) {
            uint64_t t1;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
            if (i == 16) t0 = t1;
            else if (t1 - t0 > 1000000000ull) return false;
            if (abort && *abort != 0u) return false;
            __nanosleep(128);
        }
    }
}

constexpr int kStages = 2;
constexpr int kRowTile = 2048;               // bytes of one 32-row x 64-byte tile
// Issues the TMA loads of one tile (u, delta, [z], B, [C]) into `st`.
__device__ __forceinline__ void issue_tile(int, int64_t tj64, uint8_t* st, uint64_t* bar, uint32_t tx_bytes,
                                           uint32_t bc_tile,
                                           const CUtensorMap* tu, const CUtensorMap* td, const CUtensorMap* tz,
                                           const CUtensorMap* tb, const CUtensorMap* tc, int64_t d0, int64_t b,
                                           bool has_z, bool with_c) {
    const int tj = (int)tj64;
    msc::mbar_arrive_expect_tx(bar, tx_bytes);
    msc::tma_load_3d(st, tu, bar, tj, (int)d0, (int)b);
    msc::tma_load_3d(st + kRowTile, td, bar, tj, (int)d0, (int)b);
    if (has_z) msc::tma_load_3d(st + 2 * kRowTile, tz, bar, tj, (int)d0, (int)b);
    msc::tma_load_3d(st + 3 * kRowTile, tb, bar, tj, 0, (int)b);
    if (with_c) msc::tma_load_3d(st + 3 * kRowTile + bc_tile, tc, bar, tj, 0, (int)b);
}

// One level of the readout reduce-scatter: lanes that differ in bit `kSL` of
// their group position exchange halves of v[0..kSpan) and keep the half of
// their side, summed, in v[0..kSpan/2).
// kJShift: the lane bit at which the position j within the group starts.
template <int kSL, int kSpan, int kJShift = 0>
__device__ __forceinline__ void reduce_scatter_level(float* v, int j) {
    const bool side = (j & kSL) != 0;
#pragma unroll
    for (int k = 0; k < kSpan / 2; ++k) {
        const float send = side ? v[k] : v[k + kSpan / 2];
        const float keep = side ? v[k + kSpan / 2] : v[k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, kSL << kJShift);
    }
}

// kNG lanes share a channel row: lane j of the group owns states
// n in [j * 16 / kNG, (j + 1) * 16 / kNG) and the per-step work (softplus, gate,
// store) of steps j * 8 / kNG .. of every 8-step group.  Per-step scalars are
// gathered from their owner lane with shuffles; the readout partial sums are
// reduce-scattered back with a shuffle butterfly.
//
// kDisc selects the input term b_t of h_t = abar_t h_{t-1} + b_t:
//  - exponential Euler: b = Delta B u;
//  - zero-order hold ("Mamba 解密" sec. 3 / sec. 5): b = phi(Delta A) Delta B u with
//    phi(x) = expm1(x) / x, taken from its series 1 + x/2 + x^2/6 + x^3/24 when
//    |x| < 0.03 (truncation < 1e-8) and from (abar - 1) (1/A) (1/Delta) otherwise
//    (the rounding of abar then costs < 1e-5 relative); 1/A per state is set up
//    once and 1/Delta is one reciprocal per step shared by the row's states;
//  - exponential-trapezoidal ("Mamba 解密" sec. 6.3): b_t = e_t + abar_t e_{t-1}
//    with e_t = Delta_t B_t u_t / 2, carried per state in registers; a segment's
//    first step rebuilds e_{t0-1} from the inputs at t0 - 1 (none before t = 0).
// kConv: the u tiles hold the input x of the causal conv1d + SiLU front end, and
// every lane forms u_t = silu(b + sum_k w_k x_{t-K+1+k}) for its own four steps
// of each 8-step group: it loads its x as packed pairs and takes the three steps
// before from its partner lane (the partner's steps of this group, or of the
// previous group, which the second lane keeps in registers across groups and
// tiles; at a segment start they are read from memory), so u never goes
// through HBM.
// Resident CTAs asked of the compiler (0: its own choice), as timed best at
// 8 x 5120 x 2048: 16 slots: its choice (126-128 registers, 8 per SM); 32 slots:
// its choice with bf16 (126 registers, 4 per SM; held to 5 it spills and runs
// 3-4% slower), 4 with fp32; 64 slots: 3.
template <bool kBF16, int kSN>
constexpr int fwd_min_ctas() { return kSN == 16 ? 0 : kSN == 32 ? (kBF16 ? 0 : 4) : 3; }

template <bool kBF16, int kMode, int kNG, int kDisc = kDiscEuler, bool kConv = false, int kSN = kNS,
          bool kLongRows = false>
__global__ void __launch_bounds__(32 * kNG, (fwd_min_ctas<kBF16, kSN>())) s6_fwd_tma_kernel(const __grid_constant__ CUtensorMap tm_u,
                                                              const __grid_constant__ CUtensorMap tm_d,
                                                              const __grid_constant__ CUtensorMap tm_z,
                                                              const __grid_constant__ CUtensorMap tm_B,
                                                              const __grid_constant__ CUtensorMap tm_C,
                                                              const FwdParams p) {
    constexpr bool kFull = (kMode == kModeFull || kMode == kModeFullCkpt);
    constexpr bool kWriteCk = (kMode == kModeCkpt || kMode == kModeFullCkpt);
    constexpr int kTT = kBF16 ? 32 : 16;  // steps per 64-byte tile row
    constexpr int kGroups = kTT / 8;
    constexpr int kPitch = 2 * kTT + 4;   // floats per n-pair row of s_bc (padded: conflict-free stores)
    constexpr int kES = kBF16 ? 2 : 4;    // bytes per element
    constexpr int kPPL = kSN / (2 * kNG); // state pairs per lane
    constexpr int kSPG = 8 / kNG;         // steps per lane per 8-step group
    constexpr int kBCT = kSN * 64;        // bytes of one B or C tile (kSN slots x 64 bytes)
    constexpr int kSB = 3 * kRowTile + 2 * kBCT;
    static_assert(kSN == kNS || !kWriteCk, "checkpoints are kept for 16 states");
    static_assert(!kConv || kSN == kNS, "the fused conv front end runs with up to 16 states");
    __shared__ __align__(1024) uint8_t s_raw[kStages][kSB];
    // Refill point of the two-stage ring.  Early (more than 16 slots, four warps
    // per CTA): tile i + 1 is issued at the one barrier of tile i, once every
    // thread is past tile i - 1, whose stage it takes.  Late (16 slots): tile
    // i + 2 is issued after a second barrier at the end of tile i, which gives the
    // load a whole tile of lead.  Timed at 8 x 5120 x 2048: the early refill is
    // 4% faster with 32 slots and 2% slower with 16.
    constexpr bool kEarly = kSN != kNS;
    // [tile parity][B|C][lane j of a row][n pair q - kPPL j][t * 2 + n parity]: each
    // lane's kPPL rows, then kSkew floats, so that the four lanes of a row read
    // distinct banks (without the skew their rows are 0 mod 32 banks apart).  With
    // the early refill there are two buffers: tile i is converted while slower
    // warps may still read tile i - 1.
    constexpr int kSkew = kSN == kNS ? 0 : 8;
    __shared__ __align__(16) float s_bc[kEarly ? 2 : 1][2][kNG][kPPL * kPitch + kSkew];
    // kLongRows (rows of y a megabyte or more apart): y of a 32-step window of
    // every row (one tile with bf16 inputs, two with fp32) is staged here and
    // written out after the tile-end barrier as whole 128-byte row runs.
    // Stored 16 bytes a lane straight from the groups, each row's line is
    // assembled from four to eight separate stores, which at 1 x 1536 x 2^20
    // (rows 4 MB apart) cost a sixth of the time; with short rows the staging
    // costs more than it saves (3% at 8 x 5120 x 2048).  Row pitch 40 floats:
    // the eight lanes of a store phase (four rows, two chunks) hit distinct banks.
    constexpr bool kStageY = kLongRows && kFull && !kEarly;
    static_assert(!kLongRows || kStageY, "long-row staging is for the 16-slot full pass");
    __shared__ __align__(16) float s_y[kStageY ? kRows : 1][kStageY ? 40 : 4];
    __shared__ __align__(8) uint64_t s_full[kStages];

    // Lanes of a row: with two lanes, adjacent lanes (j = lane bit 0).  With
    // four, lanes 8 apart (j = lane >> 3; a warp holds 8 rows): a 16-byte shared
    // load costs two wavefronts when each quarter-warp reads one address (all
    // its lanes the same state quarter), about four when the quarter-warp's
    // lanes read four (measured: the B/C loads of the adjacent layout cost 3.9
    // wavefronts each with the shared-memory pipe 94% busy).
    constexpr int kJShift = kNG == 4 ? 3 : 0;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int r = kNG == 4 ? (tid >> 5) * 8 + (lane & 7) : tid / kNG;  // row within the CTA
    const int j = (lane >> kJShift) & (kNG - 1);                       // position within the row's lane group
    const int glane0 = lane & ~((kNG - 1) << kJShift);
    const int N = p.N;
    const bool has_z = kFull && p.z != nullptr;
    __shared__ long long s_ticket;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) msc::mbar_init(&s_full[s], 1);
        msc::fence_barrier_init();
        msc::prefetch_tmap(&tm_u);
        msc::prefetch_tmap(&tm_d);
        msc::prefetch_tmap(&tm_B);
        if (has_z) msc::prefetch_tmap(&tm_z);
        if (kFull) msc::prefetch_tmap(&tm_C);
    }
    __syncthreads();

    // Items: one per CTA from blockIdx (row block, batch entry, segment), or,
    // with a ticket counter, (row block, chunk) items taken in order until none
    // are left.  tbase counts the tiles earlier items took through the stage ring.
    uint32_t tbase = 0;
    for (;;) {
    int64_t b, d0, chain = 0, t_begin, t_end;
    int seg;
    if (p.ctr) {
        if (tid == 0) s_ticket = (long long)atomicAdd(p.ctr, 1ull);
        __syncthreads();
        const long long item = s_ticket;
        if (item >= p.total_items) break;
        chain = item % p.chains;
        seg = (int)(item / p.chains);
        b = chain / p.nblk;
        d0 = (chain % p.nblk) * kRows;
        t_begin = (int64_t)seg * p.chunk;
        t_end = imin64(p.L, t_begin + p.chunk);
    } else {
        b = blockIdx.y;
        d0 = (int64_t)blockIdx.x * kRows;
        seg = blockIdx.z;
        t_begin = (int64_t)seg * p.seg_len;
        t_end = imin64(p.L, t_begin + p.seg_len);
    }
    const bool chained_in = p.ctr && p.chained && seg > 0;  // starts from the previous chunk's state
    if (chained_in) {
        bool ok = true;
        if (tid == 0) ok = wait_flag_geq(&p.flags[chain], (unsigned)seg, p.abort_word);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                record_timeout(3);
                atomicExch(p.abort_word, 1u);
            }
            return;
        }
    }
    const int nrows = (int)imin64(kRows, p.dim - d0);
    const bool row_ok = r < nrows;
    const int64_t d = row_ok ? d0 + r : d0;
    const int64_t row = b * p.dim + d;

    uint64_t A2p[kPPL], h2[kPPL];
#pragma unroll
    for (int q = 0; q < kPPL; ++q) {
        float a[2], h[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int n = 2 * (kPPL * j + q) + e;
            a[e] = (row_ok && n < N) ? __ldg(p.A + d * N + n) * MSC_LOG2E : 0.f;
            h[e] = 0.f;
            if (kFull && row_ok && n < N) {
                if (chained_in)
                    h[e] = __ldcg(p.chain_state + row * kSN + n);
                else if (p.G > 1)
                    h[e] = p.seg_state[((size_t)row * p.G + seg) * N + n];
                else if (p.h0 && seg == 0)
                    h[e] = __ldg(p.h0 + row * N + n);
            }
        }
        A2p[q] = msc::pk2(a[0], a[1]);
        h2[q] = msc::pk2(h[0], h[1]);
    }
    const float Dd = (kFull && p.D && row_ok) ? __ldg(p.D + d) : 0.f;
    const float bias = (p.delta_bias && row_ok) ? __ldg(p.delta_bias + d) : 0.f;
    float dsum = 0.f;

    // fused conv: taps right-aligned in a 4-tap window (cw[m] multiplies x_{t-3+m}),
    // as packed pairs; xprev = x of the three steps before this lane's group (kept by
    // the second lane of the row: its last three steps)
    static_assert(!kConv || kNG == 2, "the fused conv front end runs with two lanes per row");
    uint64_t cw2[4];
    uint64_t cb2 = 0ull;
    float xprev[3] = {0.f, 0.f, 0.f};
    if constexpr (kConv) {
        const int K = p.conv_k;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float w = (row_ok && m + K >= 4) ? __ldg(p.conv_w + d * K + (m + K - 4)) : 0.f;
            cw2[m] = msc::pk2(w, w);
        }
        const float cb = (row_ok && p.conv_b) ? __ldg(p.conv_b + d) : 0.f;
        cb2 = msc::pk2(cb, cb);
#pragma unroll
        for (int m = 0; m < 3; ++m) {
            const int64_t tp = t_begin - 3 + m;
            xprev[m] = (j == 1 && row_ok && tp >= 0) ? msc::ld_elem<kBF16>(p.u, row * p.L + tp) : 0.f;
        }
    }
    // zero-order hold: 1/A per state (0 where A = 0: the series branch covers it)
    uint64_t invA2[kDisc == kDiscZoh ? kPPL : 1];
    // trapezoid: half input term of the previous step, per state
    uint64_t ep2[kDisc == kDiscTrap ? kPPL : 1];
    if constexpr (kDisc == kDiscZoh) {
#pragma unroll
        for (int q = 0; q < kPPL; ++q) {
            float a0, a1;
            msc::upk2(A2p[q], a0, a1);
            a0 *= MSC_LN2;
            a1 *= MSC_LN2;
            invA2[q] = msc::pk2(a0 != 0.f ? 1.f / a0 : 0.f, a1 != 0.f ? 1.f / a1 : 0.f);
        }
    }
    if constexpr (kDisc == kDiscTrap) {
        float eu = 0.f;
        if (row_ok && t_begin > 0) {
            const int64_t tp = t_begin - 1;
            const float dtp = msc::softplus_f(msc::ld_elem<kBF16>(p.delta, row * p.L + tp) + bias);
            eu = 0.5f * dtp * msc::ld_elem<kBF16>(p.u, row * p.L + tp);
        }
#pragma unroll
        for (int q = 0; q < kPPL; ++q) {
            float e[2] = {0.f, 0.f};
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int n = 2 * (kPPL * j + q) + k;
                if (eu != 0.f && n < N) e[k] = eu * msc::ld_elem<kBF16>(p.B, (b * N + n) * p.L + t_begin - 1);
            }
            ep2[q] = msc::pk2(e[0], e[1]);
        }
    }
    const int ntiles = (int)((t_end - t_begin + kTT - 1) / kTT);
    const uint32_t tx_bytes = kRowTile * (has_z ? 3 : 2) + kBCT * (kFull ? 2 : 1);

    static_assert(kStages == 2, "the early refill puts tile i + 1 in the stage of tile i - 1");
    const int ahead = kEarly ? 1 : kStages;  // tiles issued before the first is computed
    if (tid == 0)
        for (int jt = 0; jt < ahead && jt < ntiles; ++jt)
            issue_tile(jt, t_begin + (int64_t)jt * kTT, s_raw[(tbase + jt) % kStages], &s_full[(tbase + jt) % kStages],
                       tx_bytes, kBCT, &tm_u, &tm_d, &tm_z, &tm_B, &tm_C, d0, b, has_z, kFull);
    int issued = ntiles < ahead ? ntiles : ahead;

    bool failed = false;
    int i = 0;
    for (; i < ntiles; ++i) {
        const int st = (tbase + i) % kStages;
        const int buf = kEarly ? (int)((tbase + i) & 1u) : 0;
        const bool ok = msc::wait_bounded(&s_full[st], (uint32_t)(((tbase + i) / kStages) & 1), p.abort_word);
        const uint8_t* raw = s_raw[st];
        const int64_t t0 = t_begin + (int64_t)i * kTT;
        const int nt = (int)imin64(kTT, t_end - t0);

        // B (and C) of this tile -> fp32 pairs s_bc[x][q][2t + e] = X[n = 2q + e][t];
        // one task per (B|C, n pair q, 16-byte chunk c)
        constexpr int kTasks = (kFull ? 2 : 1) * 2 * kSN;
#pragma unroll
        for (int it = 0; it < (kTasks + 32 * kNG - 1) / (32 * kNG); ++it) {
            const int task = tid + it * 32 * kNG;
            const int x = task / (2 * kSN), q = task % (kSN / 2), c = (task % (2 * kSN)) / (kSN / 2);
            if (task < kTasks) {
                const uint8_t* src = raw + 3 * kRowTile + x * kBCT;
                const uint4 v0 = *reinterpret_cast<const uint4*>(src + msc::sw64(2 * q, c));
                const uint4 v1 = *reinterpret_cast<const uint4*>(src + msc::sw64(2 * q + 1, c));
                float* dst = &s_bc[buf][x][q / kPPL][(q % kPPL) * kPitch];
                if constexpr (kBF16) {
                    const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w}, w1[4] = {v1.x, v1.y, v1.z, v1.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        *reinterpret_cast<float4*>(dst + 2 * (8 * c + 2 * k)) =
                            make_float4(msc::bf16lo(w0[k]), msc::bf16lo(w1[k]), msc::bf16hi(w0[k]), msc::bf16hi(w1[k]));
                    }
                } else {
                    *reinterpret_cast<float4*>(dst + 2 * (4 * c)) =
                        make_float4(__uint_as_float(v0.x), __uint_as_float(v1.x), __uint_as_float(v0.y), __uint_as_float(v1.y));
                    *reinterpret_cast<float4*>(dst + 2 * (4 * c + 2)) =
                        make_float4(__uint_as_float(v0.z), __uint_as_float(v1.z), __uint_as_float(v0.w), __uint_as_float(v1.w));
                }
            }
        }
        // One barrier: the vote on the wait (every thread takes the same branch, so
        // none is left at a barrier; after a timeout the converted values are
        // discarded) and the conversion complete -- and, for the early refill,
        // every thread past tile i - 1.
        if (__syncthreads_or(!ok)) {
            if (tid == 0) record_timeout(1);
            failed = true;
            break;
        }
        if constexpr (kEarly) {
            if (tid == 0 && i + 1 < ntiles) {
                const uint32_t si = (tbase + i + 1) % kStages;
                issue_tile(i + 1, t_begin + (int64_t)(i + 1) * kTT, s_raw[si], &s_full[si], tx_bytes, kBCT, &tm_u,
                           &tm_d, &tm_z, &tm_B, &tm_C, d0, b, has_z, kFull);
            }
            if (i + 1 < ntiles) issued = i + 2;
        }

#pragma unroll 1
        for (int g = 0; g < kGroups; ++g) {
            if (8 * g >= nt) break;
            const bool partial = 8 * g + 8 > nt;
            // ---- this lane's kSPG steps: Delta, Delta*u, D*u on packed pairs
            const uint32_t boff = (uint32_t)(8 * g * kES + j * kSPG * kES);  // byte offset in the row
            uint64_t u2[kSPG / 2], x2[kSPG / 2];
            if constexpr (kConv) {
                // x of this lane's four steps, and of the three before them
                const uint8_t* px = raw + msc::sw64(r, boff >> 4) + (boff & 15);
                const uint8_t* pd = raw + kRowTile + msc::sw64(r, boff >> 4) + (boff & 15);
                float xw[7];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    if constexpr (kBF16) {
                        const uint32_t wx = reinterpret_cast<const uint32_t*>(px)[e];
                        const uint32_t wd = reinterpret_cast<const uint32_t*>(pd)[e];
                        xw[3 + 2 * e] = msc::bf16lo(wx);
                        xw[4 + 2 * e] = msc::bf16hi(wx);
                        x2[e] = msc::pk2(msc::bf16lo(wd), msc::bf16hi(wd));
                    } else {
                        const float2 fx = reinterpret_cast<const float2*>(px)[e];
                        xw[3 + 2 * e] = fx.x;
                        xw[4 + 2 * e] = fx.y;
                        x2[e] = reinterpret_cast<const uint64_t*>(pd)[e];
                    }
                }
                // lane 0 of the row sends its steps 1..3 (lane 1's predecessors), lane 1
                // its previous group's steps 1..3 (lane 0's predecessors)
#pragma unroll
                for (int m = 0; m < 3; ++m) {
                    const float send = j == 0 ? xw[4 + m] : xprev[m];
                    xw[m] = __shfl_xor_sync(0xffffffffu, send, 1);
                }
                if (j == 1) {
#pragma unroll
                    for (int m = 0; m < 3; ++m) xprev[m] = xw[4 + m];
                }
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    uint64_t acc = cb2;
#pragma unroll
                    for (int m = 0; m < 4; ++m) acc = msc::fma2(cw2[m], msc::pk2(xw[2 * e + m], xw[2 * e + 1 + m]), acc);
                    u2[e] = msc::silu_2(acc);
                }
            } else if constexpr (kBF16) {
                const uint8_t* pu = raw + msc::sw64(r, boff >> 4) + (boff & 15);
                const uint8_t* pd = raw + kRowTile + msc::sw64(r, boff >> 4) + (boff & 15);
#pragma unroll
                for (int e = 0; e < kSPG / 2; ++e) {
                    const uint32_t wu = reinterpret_cast<const uint32_t*>(pu)[e];
                    const uint32_t wd = reinterpret_cast<const uint32_t*>(pd)[e];
                    u2[e] = msc::pk2(msc::bf16lo(wu), msc::bf16hi(wu));
                    x2[e] = msc::pk2(msc::bf16lo(wd), msc::bf16hi(wd));
                }
            } else {
                const uint8_t* pu = raw + msc::sw64(r, boff >> 4) + (boff & 15);
                const uint8_t* pd = raw + kRowTile + msc::sw64(r, boff >> 4) + (boff & 15);
#pragma unroll
                for (int e = 0; e < kSPG / 2; ++e) {
                    u2[e] = reinterpret_cast<const uint64_t*>(pu)[e];
                    x2[e] = reinterpret_cast<const uint64_t*>(pd)[e];
                }
            }
            const uint64_t bias2 = msc::pk2(bias, bias);
            uint64_t mdt2[kSPG / 2], mdtu2[kSPG / 2], mdu2[kSPG / 2];
#pragma unroll
            for (int e = 0; e < kSPG / 2; ++e) {
                uint64_t dt = msc::softplus_2(msc::add2(x2[e], bias2));
                if (partial) {
                    float a, c;
                    msc::upk2(dt, a, c);
                    const int k0 = 8 * g + j * kSPG + 2 * e;
                    dt = msc::pk2(k0 < nt ? a : 0.f, k0 + 1 < nt ? c : 0.f);  // past the end: abar = 1, input 0
                }
                mdt2[e] = dt;
                mdtu2[e] = msc::mul2(dt, u2[e]);
                if constexpr (kDisc == kDiscTrap) mdtu2[e] = msc::mul2(mdtu2[e], msc::pk2(0.5f, 0.5f));
                mdu2[e] = msc::mul2(msc::pk2(Dd, Dd), u2[e]);
                if (kMode == kModeAgg) {
                    float a, c;
                    msc::upk2(dt, a, c);
                    dsum += a + c;
                }
            }
            // ---- every lane of the group gets Delta, Delta*u of all 8 steps
            float mdt[kSPG], mdtu[kSPG];
#pragma unroll
            for (int e = 0; e < kSPG / 2; ++e) {
                msc::upk2(mdt2[e], mdt[2 * e], mdt[2 * e + 1]);
                msc::upk2(mdtu2[e], mdtu[2 * e], mdtu[2 * e + 1]);
            }
            float dts[8], dtus[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int src = glane0 | ((k / kSPG) << kJShift);
                if constexpr (kNG == 1) {
                    dts[k] = mdt[k];
                    dtus[k] = mdtu[k];
                } else {
                    dts[k] = __shfl_sync(0xffffffffu, mdt[k % kSPG], src);
                    dtus[k] = __shfl_sync(0xffffffffu, mdtu[k % kSPG], src);
                }
            }
            if (kWriteCk && row_ok) {
                // state entering this 8-step group, for the recomputing backward
                float* cp = p.ckpt + ((size_t)row * p.ckpt_groups + (size_t)((t0 + 8 * g) >> 3)) * kNS +
                            2 * kPPL * j;
#pragma unroll
                for (int q = 0; q < kPPL; q += 2)
                    *reinterpret_cast<ulonglong2*>(cp + 2 * q) = make_ulonglong2(h2[q], h2[q + 1]);
            }
            // ---- the scan: 8 steps, kPPL independent state pairs per step
            uint64_t acc[8];
            const float* bsrc = &s_bc[buf][0][j][16 * g];
            const float* csrc = &s_bc[buf][1][j][16 * g];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                uint64_t Bp[kPPL][2], Cp[kPPL][2];
#pragma unroll
                for (int q = 0; q < kPPL; ++q) {
                    const ulonglong2 vb = *reinterpret_cast<const ulonglong2*>(bsrc + q * kPitch + 4 * kk);
                    Bp[q][0] = vb.x; Bp[q][1] = vb.y;
                    if (kFull) {
                        const ulonglong2 vc = *reinterpret_cast<const ulonglong2*>(csrc + q * kPitch + 4 * kk);
                        Cp[q][0] = vc.x; Cp[q][1] = vc.y;
                    }
                }
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int k = 2 * kk + e;
                    const uint64_t dt2 = msc::pk2(dts[k], dts[k]);
                    const uint64_t dtu2 = msc::pk2(dtus[k], dtus[k]);
                    uint64_t acc_a = 0ull;
                    float rdt = 0.f;
                    if constexpr (kDisc == kDiscZoh) rdt = dts[k] > 0.f ? msc::rcp_approx(dts[k]) : 0.f;
                    if constexpr (kDisc == kDiscTrap) {
                        // the first step past the end drops the previous input term
                        if (partial && k == nt - 8 * g) {
#pragma unroll
                            for (int q = 0; q < kPPL; ++q) ep2[q] = 0ull;
                        }
                    }
#pragma unroll
                    for (int q = 0; q < kPPL; ++q) {
                        const uint64_t arg = msc::mul2(dt2, A2p[q]);
                        const uint64_t a = msc::ex2_2(arg);
                        if constexpr (kDisc == kDiscEuler) {
                            h2[q] = msc::fma2(a, h2[q], msc::mul2(dtu2, Bp[q][e]));
                        } else if constexpr (kDisc == kDiscZoh) {
                            const uint64_t x = msc::mul2(arg, msc::pk2(MSC_LN2, MSC_LN2));  // Delta A
                            uint64_t ps = msc::fma2(x, msc::pk2(1.f / 24.f, 1.f / 24.f), msc::pk2(1.f / 6.f, 1.f / 6.f));
                            ps = msc::fma2(x, ps, msc::pk2(0.5f, 0.5f));
                            ps = msc::fma2(x, ps, msc::pk2(1.f, 1.f));
                            const uint64_t pd = msc::mul2(msc::mul2(msc::add2(a, msc::pk2(-1.f, -1.f)), invA2[q]),
                                                          msc::pk2(rdt, rdt));
                            float x0, x1, s0, s1, d0, d1;
                            msc::upk2(x, x0, x1);
                            msc::upk2(ps, s0, s1);
                            msc::upk2(pd, d0, d1);
                            const uint64_t phi = msc::pk2(fabsf(x0) < 0.03f ? s0 : d0, fabsf(x1) < 0.03f ? s1 : d1);
                            h2[q] = msc::fma2(a, h2[q], msc::mul2(phi, msc::mul2(dtu2, Bp[q][e])));
                        } else {
                            const uint64_t e2 = msc::mul2(dtu2, Bp[q][e]);  // half the Euler term
                            h2[q] = msc::fma2(a, msc::add2(h2[q], ep2[q]), e2);
                            ep2[q] = e2;
                        }
                        // readout: one accumulator chain over the lane's pairs (the
                        // eight steps in flight hide its latency)
                        if (kFull) acc_a = q == 0 ? msc::mul2(Cp[q][e], h2[q]) : msc::fma2(Cp[q][e], h2[q], acc_a);
                    }
                    if (kFull) acc[k] = acc_a;
                }
            }
            // ---- readout + skip + gate of this lane's steps
            if (kFull) {
                float v[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    float lo, hi;
                    msc::upk2(acc[k], lo, hi);
                    v[k] = lo + hi;
                }
                // reduce-scatter over the group: lane j ends with steps j*kSPG ..
                if constexpr (kNG > 1) reduce_scatter_level<kNG / 2, 8, kJShift>(v, j);
                if constexpr (kNG == 4) reduce_scatter_level<1, 4, kJShift>(v, j);
                uint64_t y2[kSPG / 2];
#pragma unroll
                for (int e = 0; e < kSPG / 2; ++e) y2[e] = msc::add2(msc::pk2(v[2 * e], v[2 * e + 1]), mdu2[e]);
                if (has_z) {
                    const uint32_t zoff = boff;
                    const uint8_t* pz = raw + 2 * kRowTile + msc::sw64(r, zoff >> 4) + (zoff & 15);
#pragma unroll
                    for (int e = 0; e < kSPG / 2; ++e) {
                        uint64_t z2;
                        if constexpr (kBF16) {
                            const uint32_t wz = reinterpret_cast<const uint32_t*>(pz)[e];
                            z2 = msc::pk2(msc::bf16lo(wz), msc::bf16hi(wz));
                        } else {
                            z2 = reinterpret_cast<const uint64_t*>(pz)[e];
                        }
                        y2[e] = msc::mul2(y2[e], msc::silu_2(z2));
                    }
                }
                if constexpr (kStageY) {
                    static_assert(kSPG == 4, "staged y: four steps a lane");
                    const int c = (kBF16 ? 0 : (i & 1) * 4) + 2 * g + j;  // 16-byte chunk of the window
                    *reinterpret_cast<ulonglong2*>(&s_y[r][4 * c]) = make_ulonglong2(y2[0], y2[1]);
                } else if (row_ok) {
                    const int rem = nt - 8 * g - j * kSPG;
                    float* qy = p.y + row * p.L + t0 + 8 * g + j * kSPG;
                    if (rem >= kSPG) {
                        if constexpr (kSPG == 4)
                            __stcs(reinterpret_cast<ulonglong2*>(qy), make_ulonglong2(y2[0], y2[1]));
                        else
                            __stcs(reinterpret_cast<unsigned long long*>(qy), (unsigned long long)y2[0]);
                    } else {
                        float vv[kSPG];
#pragma unroll
                        for (int e = 0; e < kSPG / 2; ++e) msc::upk2(y2[e], vv[2 * e], vv[2 * e + 1]);
#pragma unroll
                        for (int k = 0; k < kSPG - 1; ++k)
                            if (k < rem) qy[k] = vv[k];
                    }
                }
            }
        }
        if constexpr (!kEarly) {
            __syncthreads();  // every thread is done with this tile's stage (and its y is staged)
            if (tid == 0 && issued < ntiles) {
                const uint32_t si = (tbase + issued) % kStages;
                issue_tile(issued, t_begin + (int64_t)issued * kTT, s_raw[si], &s_full[si], tx_bytes, kBCT, &tm_u,
                           &tm_d, &tm_z, &tm_B, &tm_C, d0, b, has_z, kFull);
            }
            ++issued;
            if constexpr (kStageY) {
                // the window is complete (or the item ends): eight lanes a row, 16 bytes
                // each; the next tile's groups write s_y only after its first barrier
                if (kBF16 || (i & 1) || i + 1 == ntiles) {
                    const int64_t tw = t_begin + (int64_t)(kBF16 ? i : (i & ~1)) * kTT;
                    const int nw = (int)imin64(32, t_end - tw);
                    for (int e = tid; e < kRows * 8; e += 32 * kNG) {
                        const int rr = e >> 3, c = e & 7;
                        if (rr < nrows && 4 * c < nw) {
                            const float4 v = *reinterpret_cast<const float4*>(&s_y[rr][4 * c]);
                            float* q = p.y + (b * p.dim + d0 + rr) * p.L + tw + 4 * c;
                            if (4 * c + 4 <= nw) {
                                __stcs(reinterpret_cast<float4*>(q), v);
                            } else {
                                q[0] = v.x;
                                if (4 * c + 1 < nw) q[1] = v.y;
                                if (4 * c + 2 < nw) q[2] = v.z;
                            }
                        }
                    }
                }
            }
        }
    }

    if (failed) {
        // drain loads still in flight before the shared memory is released
        if (tid == 0) {
            if (p.abort_word) atomicExch(p.abort_word, 1u);
            for (int jt = i; jt < issued && jt < ntiles; ++jt)
                (void)msc::wait_bounded(&s_full[(tbase + jt) % kStages], (uint32_t)(((tbase + jt) / kStages) & 1));
        }
        return;
    }
    if (kMode == kModeCkpt) return;
    if (!kFull) {
#pragma unroll
        for (int sl = 1; sl < kNG; sl *= 2) dsum += __shfl_xor_sync(0xffffffffu, dsum, sl << kJShift);
    }
    // a chained chunk that is not the row's last hands its state to the next chunk
    const bool publish = kFull && p.ctr && p.chained && t_end < p.L;
    if (row_ok) {
#pragma unroll
        for (int q = 0; q < kPPL; ++q) {
            float v0, v1;
            msc::upk2(h2[q], v0, v1);
            const int n = 2 * (kPPL * j + q);
            if (kFull) {
                if (publish) {
                    *reinterpret_cast<uint64_t*>(p.chain_state + row * kSN + n) = h2[q];
                } else if (p.h_last && t_end == p.L) {
                    if (n < N) p.h_last[row * N + n] = v0;
                    if (n + 1 < N) p.h_last[row * N + n + 1] = v1;
                }
            } else {
                if (n < N) p.seg_state[((size_t)row * p.G + seg) * N + n] = v0;
                if (n + 1 < N) p.seg_state[((size_t)row * p.G + seg) * N + n + 1] = v1;
            }
        }
        if (!kFull && j == 0) p.seg_dsum[(size_t)row * p.G + seg] = dsum;
    }
    if (!p.ctr) break;
    tbase += (uint32_t)ntiles;
    __syncthreads();  // this item's state is stored (and s_ticket may be rewritten)
    if (tid == 0 && publish) {
        __threadfence();
        asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(&p.flags[chain]), "r"((unsigned)(seg + 1)) : "memory");
    }
    }  // items
}

// Chains the segment aggregates of every (row, n): carry_0 = h0 (or 0),
// carry_{g+1} = exp(A sum Delta_g) carry_g + H_g.  Carries overwrite the
// aggregates in place (each is read before it is overwritten, by one thread).
__global__ void s6_seg_carry_kernel(const float* __restrict__ A, const float* __restrict__ h0,
                                    float* seg_state, const float* __restrict__ seg_dsum,
                                    int64_t rows, int64_t dim, int N, int G) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= rows * N) return;
    const int64_t row = idx / N;
    const int n = (int)(idx % N);
    const int64_t d = row % dim;
    const float a2 = __ldg(A + d * N + n) * MSC_LOG2E;
    float h = h0 ? __ldg(h0 + row * N + n) : 0.f;
    // The aggregates and sums of eight segments are loaded ahead of the
    // dependent chain (each slot is read before this thread overwrites it).
    // The aggregate pass writes segments 0 .. G-2; the last slot only receives
    // its carry.
    for (int g0 = 0; g0 < G; g0 += 8) {
        float agg[8], ds[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int g = g0 + k;
            agg[k] = g + 1 < G ? seg_state[((size_t)row * G + g) * N + n] : 0.f;
            ds[k] = g + 1 < G ? seg_dsum[(size_t)row * G + g] : 0.f;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int g = g0 + k;
            if (g >= G) break;
            seg_state[((size_t)row * G + g) * N + n] = h;
            if (g + 1 < G) h = fmaf(msc::ex2_approx(a2 * ds[k]), h, agg[k]);
        }
    }
}

// Sets steps [L, Lp) of every row of a padded copy to the bit pattern `fill`
// (4-byte or 2-byte elements).
__global__ void s6_pad_tail_kernel(void* dst, int64_t rows, int64_t L, int64_t Lp, int es, uint32_t fill) {
    const int64_t tail = Lp - L;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= rows * tail) return;
    const int64_t r = idx / tail, t = L + idx % tail;
    if (es == 4)
        reinterpret_cast<uint32_t*>(dst)[r * Lp + t] = fill;
    else
        reinterpret_cast<uint16_t*>(dst)[r * Lp + t] = (uint16_t)fill;
}

template <bool kBF16, bool kVec, int kDisc, bool kConv = false>
msc_status launch_rows(const FwdParams& p, int64_t batch, int G, int mode, cudaStream_t st) {
    dim3 grid((unsigned)((p.dim + kRows - 1) / kRows), (unsigned)batch, (unsigned)G);
    if (mode == kModeFull)
        s6_fwd_rows_kernel<kBF16, kVec, kModeFull, kDisc, kConv><<<grid, kRows, 0, st>>>(p);
    else
        s6_fwd_rows_kernel<kBF16, kVec, kModeAgg, kDisc, kConv><<<grid, kRows, 0, st>>>(p);
    return msc_host::check_launch("s6_fwd_rows");
}

template <bool kBF16, bool kVec>
msc_status launch_rows_disc(const FwdParams& p, int64_t batch, int G, int mode, int disc, cudaStream_t st) {
    if (p.conv_w) {
        if (disc != kDiscEuler)
            return msc_host::fail(MSC_ERR_UNSUPPORTED, "the fused conv front end runs with the exponential-Euler form");
        return launch_rows<kBF16, kVec, kDiscEuler, true>(p, batch, G, mode, st);
    }
    if (disc == kDiscZoh) return launch_rows<kBF16, kVec, kDiscZoh>(p, batch, G, mode, st);
    if (disc == kDiscTrap) return launch_rows<kBF16, kVec, kDiscTrap>(p, batch, G, mode, st);
    return launch_rows<kBF16, kVec, kDiscEuler>(p, batch, G, mode, st);
}

struct FwdMaps {
    CUtensorMap u, d, z, B, C;
};

// bc_rows: state rows between batch entries of B and C (0: N)
bool make_maps(FwdMaps& m, const FwdParams& p, int64_t batch, bool bf16, int64_t bc_rows = 0) {
    const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const uint64_t es = bf16 ? 2 : 4;
    const uint32_t tt = bf16 ? 32 : 16;
    const uint64_t rdims[3] = {(uint64_t)p.L, (uint64_t)p.dim, (uint64_t)batch};
    const uint64_t rstr[2] = {(uint64_t)p.L * es, (uint64_t)p.dim * p.L * es};
    const uint32_t rbox[3] = {tt, (uint32_t)kRows, 1};
    const uint64_t bdims[3] = {(uint64_t)p.L, (uint64_t)p.N, (uint64_t)batch};
    const uint64_t bstr[2] = {(uint64_t)p.L * es, (uint64_t)(bc_rows ? bc_rows : p.N) * p.L * es};
    const uint32_t bbox[3] = {tt, (uint32_t)state_slots(p.N), 1};
    const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_64B;
    if (!msc_host::encode_tmap(&m.u, dt, 3, p.u, rdims, rstr, rbox, sw)) return false;
    if (!msc_host::encode_tmap(&m.d, dt, 3, p.delta, rdims, rstr, rbox, sw)) return false;
    if (!msc_host::encode_tmap(&m.z, dt, 3, p.z ? p.z : p.u, rdims, rstr, rbox, sw)) return false;
    if (!msc_host::encode_tmap(&m.B, dt, 3, p.B, bdims, bstr, bbox, sw)) return false;
    if (!msc_host::encode_tmap(&m.C, dt, 3, p.C, bdims, bstr, bbox, sw)) return false;
    return true;
}

// Lanes per channel row of the TMA kernel.  Two beat four on the batch-8 x
// 5120 x 2048 workload (0.45 ms vs 0.54 ms): four lanes double the resident
// warps but add more exchange work than the extra latency hiding recovers.
constexpr int kLanesPerRow = 2;

// Resident CTAs per SM of a kernel instance, queried once per (instance,
// block size, device).  Keyed by the kernel's address: every instance of
// s6_fwd_tma_kernel has the same function type, so a cache per type would
// hand one instance's occupancy (8 CTAs per SM with 16 slots, 3 with 64) to
// all of them.
template <typename K>
int resident_ctas(K kernel, int threads) {
    static std::mutex mu;
    static std::map<std::tuple<const void*, int, int>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_tuple(reinterpret_cast<const void*>(kernel), threads, dev);
    std::lock_guard<std::mutex> lock(mu);
    const auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, 0) != cudaSuccess || n < 1) n = 1;
    cache.emplace(key, n);
    return n;
}

// A full pass: persistent CTAs taking (row block, chunk) tickets when the
// chained schedule's control block is set, else one CTA per (row block, batch
// entry, segment).
template <bool kBF16, int kMode, int kNG, int kDisc, bool kConv, int kSN, bool kLongRows = false>
void launch_full(const FwdMaps& m, const FwdParams& p, dim3 grid, cudaStream_t st) {
    auto kern = s6_fwd_tma_kernel<kBF16, kMode, kNG, kDisc, kConv, kSN, kLongRows>;
    if (p.ctr) {
        // persistent: at most one CTA per row block, so that the chunk before a
        // ticket's chunk was taken a full round earlier and is normally done
        const int64_t slots = (int64_t)resident_ctas(kern, 32 * kNG) * msc_host::num_sms();
        const int64_t n = std::min<int64_t>(slots, std::min<int64_t>(p.chains, p.total_items));
        kern<<<(unsigned)n, 32 * kNG, 0, st>>>(m.u, m.d, m.z, m.B, m.C, p);
    } else {
        kern<<<grid, 32 * kNG, 0, st>>>(m.u, m.d, m.z, m.B, m.C, p);
    }
}

// Rows of at least this many steps take the full pass that stages y (kLongRows).
constexpr int64_t kLongRowSteps = (int64_t)1 << 19;

template <bool kBF16, int kNG, int kDisc = kDiscEuler, bool kConv = false, int kSN = kNS>
msc_status launch_tma_ng(const FwdMaps& m, const FwdParams& p, int64_t batch, int G, int mode, cudaStream_t st) {
    constexpr bool kCkOk = kDisc == kDiscEuler && !kConv && kSN == kNS;
    dim3 grid((unsigned)((p.dim + kRows - 1) / kRows), (unsigned)batch, (unsigned)G);
    if (mode == kModeFull) {
        if (kSN == kNS && p.L >= kLongRowSteps)
            launch_full<kBF16, kModeFull, kNG, kDisc, kConv, kSN, kSN == kNS>(m, p, grid, st);
        else
            launch_full<kBF16, kModeFull, kNG, kDisc, kConv, kSN>(m, p, grid, st);
    } else if (mode == kModeAgg) {
        s6_fwd_tma_kernel<kBF16, kModeAgg, kNG, kDisc, kConv, kSN>
            <<<grid, 32 * kNG, 0, st>>>(m.u, m.d, m.z, m.B, m.C, p);
    } else if constexpr (kCkOk) {
        if (mode == kModeFullCkpt)
            launch_full<kBF16, kModeFullCkpt, kNG, kDisc, kConv, kSN>(m, p, grid, st);
        else
            s6_fwd_tma_kernel<kBF16, kModeCkpt, kNG><<<grid, 32 * kNG, 0, st>>>(m.u, m.d, m.z, m.B, m.C, p);
    } else {
        return msc_host::fail(MSC_ERR_UNSUPPORTED,
                              "checkpoints are kept for the exponential-Euler form with up to 16 states only");
    }
    return msc_host::check_launch("s6_fwd_tma");
}

// Up to 16 states: two lanes per row, eight states each.  17 to 32: four lanes
// of eight states; 33 to 64: four lanes of sixteen.  Slots past N hold A = 0,
// B = C = 0 (the TMA box reads zeros past the tensor's state extent), so they
// add nothing to the readout.
template <bool kBF16, int kSN>
msc_status launch_tma_sn(const FwdMaps& m, const FwdParams& p, int64_t batch, int G, int mode, int disc,
                         cudaStream_t st) {
    constexpr int kNG = kSN == kNS ? kLanesPerRow : 4;
    if (p.conv_w) {
        if constexpr (kSN == kNS) {
            if (disc != kDiscEuler)
                return msc_host::fail(MSC_ERR_UNSUPPORTED,
                                      "the fused conv front end runs with the exponential-Euler form");
            return launch_tma_ng<kBF16, 2, kDiscEuler, true>(m, p, batch, G, mode, st);
        } else {
            return msc_host::fail(MSC_ERR_UNSUPPORTED, "the fused conv front end runs with up to 16 states");
        }
    }
    if (disc == kDiscZoh) return launch_tma_ng<kBF16, kNG, kDiscZoh, false, kSN>(m, p, batch, G, mode, st);
    if (disc == kDiscTrap) return launch_tma_ng<kBF16, kNG, kDiscTrap, false, kSN>(m, p, batch, G, mode, st);
    return launch_tma_ng<kBF16, kNG, kDiscEuler, false, kSN>(m, p, batch, G, mode, st);
}

template <bool kBF16>
msc_status launch_tma(const FwdMaps& m, const FwdParams& p, int64_t batch, int G, int mode, int disc,
                      cudaStream_t st) {
    if (p.N <= 16) return launch_tma_sn<kBF16, 16>(m, p, batch, G, mode, disc, st);
    if (p.N <= 32) return launch_tma_sn<kBF16, 32>(m, p, batch, G, mode, disc, st);
    return launch_tma_sn<kBF16, 64>(m, p, batch, G, mode, disc, st);
}

// TMA needs every row stride to be a multiple of 16 bytes.
// The TMA path needs 16-byte row strides, and its tile coordinates (step, row)
// are signed 32-bit: longer rows or more channels take the plain-load kernel,
// whose indices are 64-bit.
bool tma_ok(const FwdParams& p, bool bf16) {
    constexpr int64_t kMaxCoord = ((int64_t)1 << 31) - 64;
    if (p.L > kMaxCoord || p.dim > kMaxCoord) return false;
    return bf16 ? (p.L % 8 == 0) : (p.L % 4 == 0);
}

msc_status launch_mode(const FwdParams& p, const FwdMaps* maps, bool bf16, bool vec, int64_t batch, int G,
                       int mode, int disc, cudaStream_t st) {
    if (maps)
        return bf16 ? launch_tma<true>(*maps, p, batch, G, mode, disc, st)
                    : launch_tma<false>(*maps, p, batch, G, mode, disc, st);
    if (mode == kModeFullCkpt)
        return msc_host::fail(MSC_ERR_UNSUPPORTED,
                              "the forward with checkpoints needs 16-byte row strides and seqlen, dim below 2^31");
    if (p.N > kNS)
        return msc_host::fail(MSC_ERR_UNSUPPORTED,
                              "more than 16 states need 16-byte row strides "
                              "(seqlen a multiple of 8 with bf16 inputs, of 4 with fp32) "
                              "and seqlen, dim below 2^31");
    if (bf16)
        return vec ? launch_rows_disc<true, true>(p, batch, G, mode, disc, st)
                   : launch_rows_disc<true, false>(p, batch, G, mode, disc, st);
    return vec ? launch_rows_disc<false, true>(p, batch, G, mode, disc, st)
               : launch_rows_disc<false, false>(p, batch, G, mode, disc, st);
}

}  // namespace

namespace msc_host {

namespace {
int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }
size_t align256(size_t x) { return (x + 255) / 256 * 256; }
}  // namespace

// Work plan of the forward.  A CTA of the two-lane kernel runs 32 channel rows
// ("row block"); eight are resident per SM in the full pass (64 threads, 126 to
// 128 registers, 21 KB of shared memory).
//  - Enough row blocks to fill the GPU: one pass.  Sequences of 512 steps or
//    more are cut into chained chunks (at least 256 steps, at most 4 per row)
//    taken by persistent CTAs in order, so that a row block's work moves
//    between SMs at chunk boundaries and the SMs that hold more warps do not
//    set the time.  Its workspace (ticket counter, flags, the state handed from
//    chunk to chunk) is optional: without it the pass runs one CTA per row block.
//  - Few row blocks and a long sequence: independent segments (aggregate pass,
//    carry pass, full pass) of at least 512 steps, about twelve per resident
//    CTA slot, at most as many as keep the scratch within max_required.  Its
//    workspace is required.
// Bytes of the padded copies (u, delta, z, B, C and y at a pitch of Lp steps,
// 4 bytes an element, which covers both input dtypes).
static size_t pad_bytes(int64_t batch, int64_t dim, int64_t Lp, int64_t dstate) {
    const size_t row = align256((size_t)batch * dim * Lp * 4), bc = align256((size_t)batch * dstate * Lp * 4);
    return 4 * row + 2 * bc;
}

static S6Plan plan_rows(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate, size_t max_required);

S6Plan s6_fwd_plan(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate, size_t max_required) {
    if (dstate > kNS && seqlen % 8 != 0) {
        // only the TMA kernel takes more than 16 states: rows of a pitch it can
        // stream (a multiple of 8 steps, which holds for both input dtypes) are
        // made in the workspace; the launch skips the copies for fp32 rows of a
        // multiple of 4 steps, which TMA streams as they are
        const int64_t Lp = cdiv64(seqlen, 8) * 8;
        S6Plan plan = plan_rows(batch, dim, Lp, dstate, max_required);
        plan.padded_len = Lp;
        plan.pad_off = align256(plan.workspace);
        plan.workspace = plan.pad_off + pad_bytes(batch, dim, Lp, dstate);
        plan.workspace_required = true;
        return plan;
    }
    return plan_rows(batch, dim, seqlen, dstate, max_required);
}

// The plan for rows of seqlen steps as they are.
static S6Plan plan_rows(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate, size_t max_required) {
    // Chunks per row and their least length: each item restarts the CTA's TMA
    // pipeline (a few microseconds), so that 4 chunks of 512 steps balance the
    // batch-8 x 5120 x 2048 workload as well as 8 of 256 (0.412 vs 0.414 ms on a
    // B300) and better than 16 of 128 (0.443 ms).
    constexpr int64_t kMaxChunks = 4, kMinChunk = 256;
    S6Plan plan;
    const int64_t rows = batch * dim;
    const int64_t chains = batch * cdiv64(dim, kRows);
    // full-pass CTAs resident per SM: 8 with up to 16 states (64 threads, 126-128
    // registers), 4 or 5 with 32 state slots, 3 with 64 (128 threads)
    const int slots = state_slots(dstate);
    const int64_t W = (slots == 16 ? 8 : slots == 32 ? 4 : 3) * (int64_t)num_sms();
    plan.G = 1;
    plan.seg_len = seqlen;
    plan.chunks = 1;
    plan.chunk = seqlen;
    if (chains * 2 >= W) {
        if (seqlen >= 512) {
            const int64_t chunk = std::max<int64_t>(kMinChunk, cdiv64(cdiv64(seqlen, kMaxChunks), kT) * kT);
            plan.chunk = chunk;
            plan.chunks = (int)cdiv64(seqlen, chunk);
        }
        if (plan.chunks > 1) {
            plan.ctrl_off = 0;
            plan.ctrl_bytes = align256(256 + (size_t)chains * sizeof(unsigned));
            plan.chain_state_off = plan.ctrl_bytes;
            plan.workspace = plan.chain_state_off + (size_t)rows * slots * sizeof(float);
            plan.workspace_required = false;
        }
        return plan;
    }
    // About twelve segments per resident CTA slot: CTAs that share an SM finish
    // at different times, and many short items keep that tail short (at
    // 1 x 1536 x 2^20: 17.5 ms with 154 segments, 17.1 with 296, 19.7 with 74).
    int bestG = 1;
    int64_t best_seg = seqlen;
    for (int64_t G = std::min<int64_t>({cdiv64(12 * W, chains), seqlen / 512, (int64_t)65535}); G >= 2; --G) {
        const int64_t seg = cdiv64(cdiv64(seqlen, G), kT) * kT;
        const int64_t Gc = cdiv64(seqlen, seg);
        const size_t need = align256((size_t)rows * Gc * (size_t)dstate * sizeof(float)) + (size_t)rows * Gc * sizeof(float);
        if (Gc >= 2 && need <= max_required) {
            bestG = (int)Gc;
            best_seg = seg;
            break;
        }
    }
    if (bestG > 1) {
        plan.G = bestG;
        plan.seg_len = best_seg;
        plan.seg_state_off = 0;
        plan.seg_dsum_off = align256((size_t)rows * bestG * (size_t)dstate * sizeof(float));
        plan.workspace = plan.seg_dsum_off + (size_t)rows * bestG * sizeof(float);
        plan.workspace_required = true;
    }
    return plan;
}

// Copies rows of L elements to a pitch of Lp (tail set to `fill`).
static msc_status pad_rows(void* dst, const void* src, size_t es, int64_t rows, int64_t L, int64_t Lp,
                           uint32_t fill, cudaStream_t st) {
    cudaError_t e = cudaMemcpy2DAsync(dst, Lp * es, src, L * es, L * es, rows, cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) return fail(MSC_ERR_CUDA, "padded copy: %s", cudaGetErrorString(e));
    const int64_t n = rows * (Lp - L);
    if (n > 0) {
        s6_pad_tail_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(dst, rows, L, Lp, (int)es, fill);
        return check_launch("s6_pad_tail");
    }
    return MSC_OK;
}

msc_status s6_fwd_launch(const S6FwdArgs& a, const S6Plan& plan, cudaStream_t st) {
    if (plan.padded_len > 0 && !a.bf16 && a.L % 4 == 0) {
        // fp32 rows of a multiple of 4 steps stream through TMA as they are
        const S6Plan direct = plan_rows(a.batch, a.dim, a.L, a.N, a.workspace_bytes);
        if (!direct.workspace_required || (a.workspace && a.workspace_bytes >= direct.workspace))
            return s6_fwd_launch(a, direct, st);
    }
    if (plan.padded_len > 0) {
        // Rows of a pitch TMA can stream: delta's padded steps are -inf, so that
        // Delta = softplus(-inf) = 0 there: the decay is 1 and the input term 0, and
        // the state (h_last included) passes them unchanged.  The trapezoid's
        // carried half-term would enter the first padded step, so it is refused.
        if (a.disc == kDiscTrap)
            return fail(MSC_ERR_UNSUPPORTED,
                        "the trapezoidal form with more than 16 states needs seqlen a multiple of 8 "
                        "with bf16 inputs, of 4 with fp32");
        if (a.conv_w) return fail(MSC_ERR_UNSUPPORTED, "the fused conv front end runs with up to 16 states");
        const int64_t L = a.L, Lp = plan.padded_len, rows = a.batch * a.dim, bcrows = a.batch * a.N;
        if (Lp > ((int64_t)1 << 31) - 64 || a.dim > ((int64_t)1 << 31) - 64)
            return fail(MSC_ERR_UNSUPPORTED, "seqlen and dim must be below 2^31");
        const size_t es = a.bf16 ? 2 : 4;
        const size_t rb = align256((size_t)rows * Lp * 4), bb = align256((size_t)bcrows * Lp * 4);
        char* pad = static_cast<char*>(a.workspace) + plan.pad_off;
        char *pu = pad, *pd = pu + rb, *pz = pd + rb, *py = pz + rb, *pB = py + rb, *pC = pB + bb;
        const uint32_t ninf = a.bf16 ? 0xFF80u : 0xFF800000u;
        msc_status s;
        if ((s = pad_rows(pu, a.u, es, rows, L, Lp, 0u, st)) != MSC_OK) return s;
        if ((s = pad_rows(pd, a.delta, es, rows, L, Lp, ninf, st)) != MSC_OK) return s;
        if (a.z && (s = pad_rows(pz, a.z, es, rows, L, Lp, 0u, st)) != MSC_OK) return s;
        if ((s = pad_rows(pB, a.B, es, bcrows, L, Lp, 0u, st)) != MSC_OK) return s;
        if ((s = pad_rows(pC, a.C, es, bcrows, L, Lp, 0u, st)) != MSC_OK) return s;
        S6FwdArgs b = a;
        b.L = Lp;
        b.u = pu; b.delta = pd; b.z = a.z ? pz : nullptr; b.B = pB; b.C = pC;
        b.y = reinterpret_cast<float*>(py);
        b.workspace_bytes = plan.pad_off;
        S6Plan inner = plan;  // the padded problem's plan, its scratch below pad_off
        inner.padded_len = 0;
        inner.pad_off = 0;
        inner.workspace = plan.pad_off;
        if ((s = s6_fwd_launch(b, inner, st)) != MSC_OK) return s;
        const cudaError_t e = cudaMemcpy2DAsync(a.y, L * 4, py, Lp * 4, L * 4, rows, cudaMemcpyDeviceToDevice, st);
        if (e != cudaSuccess) return fail(MSC_ERR_CUDA, "padded copy: %s", cudaGetErrorString(e));
        return MSC_OK;
    }
    FwdParams p{};
    p.u = a.u; p.delta = a.delta; p.z = a.z; p.B = a.B; p.C = a.C;
    p.A = a.A; p.D = a.D; p.delta_bias = a.delta_bias; p.h0 = a.h0;
    p.y = a.y; p.h_last = a.h_last;
    p.dim = a.dim; p.L = a.L; p.N = a.N; p.G = plan.G; p.seg_len = plan.seg_len;
    p.conv_w = a.conv_w; p.conv_b = a.conv_b; p.conv_k = a.conv_k;
    char* ws = static_cast<char*>(a.workspace);
    // 16-byte vector loads need every row and tile start 16-byte aligned:
    // bases are checked by the caller; rows start at row * L elements.
    const bool vec = (a.L % 8) == 0;
    FwdMaps maps;
    const FwdMaps* mp = nullptr;
    // MSC_S6_FWD_PLAIN (any value) sends rows that TMA could take to the
    // plain-load kernel as well, so that the two paths can be compared on the
    // same inputs; it changes which kernel runs, not what it computes.
    if (tma_ok(p, a.bf16) && std::getenv("MSC_S6_FWD_PLAIN") == nullptr) {
        if (!make_maps(maps, p, a.batch, a.bf16)) return MSC_ERR_CUDA;
        mp = &maps;
    }
    if (plan.G > 1) {
        p.seg_state = reinterpret_cast<float*>(ws + plan.seg_state_off);
        p.seg_dsum = reinterpret_cast<float*>(ws + plan.seg_dsum_off);
        msc_status s = launch_mode(p, mp, a.bf16, vec, a.batch, plan.G - 1, kModeAgg, a.disc, st);
        if (s != MSC_OK) return s;
        const int64_t total = a.batch * a.dim * a.N;
        const int threads = 256;
        s6_seg_carry_kernel<<<(unsigned)((total + threads - 1) / threads), threads, 0, st>>>(
            a.A, a.h0, p.seg_state, p.seg_dsum, a.batch * a.dim, a.dim, a.N, plan.G);
        s = check_launch("s6_seg_carry");
        if (s != MSC_OK) return s;
    } else if (plan.chunks > 1 && mp && ws && a.workspace_bytes >= plan.workspace) {
        // chained chunks on persistent CTAs (TMA path only); the control block
        // (ticket counter at 0, abort word at 16, flags from 256) starts at zero
        unsigned char* ctrl = reinterpret_cast<unsigned char*>(ws + plan.ctrl_off);
        const cudaError_t e = cudaMemsetAsync(ctrl, 0, plan.ctrl_bytes, st);
        if (e != cudaSuccess) return fail(MSC_ERR_CUDA, "workspace clear: %s", cudaGetErrorString(e));
        p.ctr = reinterpret_cast<unsigned long long*>(ctrl);
        p.abort_word = reinterpret_cast<unsigned*>(ctrl + 16);
        p.flags = reinterpret_cast<unsigned*>(ctrl + 256);
        p.chain_state = reinterpret_cast<float*>(ws + plan.chain_state_off);
        p.chunk = plan.chunk;
        p.nblk = cdiv64(a.dim, kRows);
        p.chains = a.batch * p.nblk;
        p.total_items = p.chains * plan.chunks;
        p.chained = 1;
    }
    if (a.ckpt) {
        // the training forward also keeps the state entering every 8-step group
        p.ckpt = a.ckpt;
        p.ckpt_groups = (a.L + 7) / 8;
    }
    return launch_mode(p, mp, a.bf16, vec, a.batch, plan.G, a.ckpt ? kModeFullCkpt : kModeFull, a.disc, st);
}

// Checkpoint pass of the backward: the state entering every 8-step group of
// every row, written to ckpt [batch * dim, ceil(L / 8), 16].  Rows must be
// TMA-describable (row stride a multiple of 16 bytes).
msc_status s6_fwd_checkpoints(const S6FwdArgs& a, float* ckpt, cudaStream_t st) {
    FwdParams p{};
    p.u = a.u; p.delta = a.delta; p.z = nullptr; p.B = a.B; p.C = a.C;
    p.A = a.A; p.D = nullptr; p.delta_bias = a.delta_bias; p.h0 = nullptr;
    p.y = nullptr; p.h_last = nullptr;
    p.dim = a.dim; p.L = a.L; p.N = a.N; p.G = 1; p.seg_len = a.L;
    p.ckpt = ckpt;
    p.ckpt_groups = (a.L + 7) / 8;
    if (!tma_ok(p, a.bf16))
        return fail(MSC_ERR_UNSUPPORTED, "checkpoint pass needs a 16-byte row stride and seqlen, dim below 2^31");
    FwdMaps maps;
    if (!make_maps(maps, p, a.batch, a.bf16, a.bc_rows)) return MSC_ERR_CUDA;
    return a.bf16 ? launch_tma_ng<true, 2>(maps, p, a.batch, 1, kModeCkpt, st)
                  : launch_tma_ng<false, 2>(maps, p, a.batch, 1, kModeCkpt, st);
}

// Reads and clears this module's device status word.
msc_status s6_fwd_take_status(unsigned int* code, unsigned int* site) {
    unsigned int w[2] = {0, 0};
    cudaError_t e = cudaMemcpyFromSymbol(w, g_s6_fwd_status, sizeof(w));
    if (e != cudaSuccess) return fail(MSC_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
    if (w[0] != 0) {
        const unsigned int z[2] = {0, 0};
        e = cudaMemcpyToSymbol(g_s6_fwd_status, z, sizeof(z));
        if (e != cudaSuccess) return fail(MSC_ERR_CUDA, "status clear: %s", cudaGetErrorString(e));
    }
    *code = w[0];
    *site = w[1];
    return MSC_OK;
}

}  // namespace msc_host
