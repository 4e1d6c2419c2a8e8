// msc_tc.cuh -- 5th-generation tensor core (tcgen05) helpers for sm_103a:
// tensor-memory allocation, shared-memory matrix descriptors, the instruction
// descriptor of kind::f16 MMAs, MMA issue / commit and TMEM loads, as inline PTX.
//
// Operand layout used throughout: "K-major, 128-byte swizzle".  A tile of R rows
// and K 16-bit elements is stored as K/64 column blocks; block kb holds rows
// 0..R-1 of elements [64 kb, 64 kb + 64) as 128-byte rows, and within every
// 8-row / 1024-byte atom the 16-byte chunk c of row r sits at chunk c ^ (r % 8).
// This is the layout TMA writes with CU_TENSOR_MAP_SWIZZLE_128B for a box whose
// inner extent is 64 elements; CUDA cores write it with sw128_offset().
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "msc_common.cuh"
#include "msc_tma.cuh"

namespace msc {

// Byte offset of element (row, k) of a 16-bit K-major SW128 tile with R rows.
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t k, uint32_t R) {
    const uint32_t kb = k >> 6, kk = k & 63;
    const uint32_t chunk = (kk >> 3) ^ (row & 7);
    return kb * (R * 128u) + row * 128u + (chunk << 4) + ((kk & 7) << 1);
}

// Shared-memory matrix descriptor (tcgen05 format) of a K-major SW128 tile whose
// first 1024-byte atom starts at smem address `addr` (1024-aligned, plus a
// multiple of 32 bytes to step K by 16 elements inside the 128-byte row).
// Stride between 8-row atoms (SBO) = 1024 bytes; LBO is unused for swizzled
// K-major layouts whose per-instruction K span stays inside one 128-byte row.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFFu);            // start address >> 4, bits 0-13
    d |= (uint64_t)(1u) << 16;                          // LBO (ignored), bits 16-29
    d |= (uint64_t)((1024u >> 4) & 0x3FFFu) << 32;      // SBO >> 4, bits 32-45
    d |= (uint64_t)1 << 46;                             // descriptor version, bits 46-47 = 0b01
    d |= (uint64_t)2 << 61;                             // layout: 128-byte swizzle, bits 61-63
    return d;
}

// Descriptor of an MN-major SW128 tile: 64-element MN blocks of K rows x 128
// bytes each (the layout TMA writes for a box {64 along MN, K rows} with
// SWIZZLE_128B); `lbo_bytes` = distance between consecutive 64-wide MN blocks,
// SBO = 1024 bytes between groups of 8 K rows.  Step K by 16 with +2048 bytes.
__device__ __forceinline__ uint64_t sdesc_sw128_mn(uint32_t addr, uint32_t lbo_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((1024u >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor of tcgen05.mma kind::f16 with fp32 accumulation.
// ab_bf16: operands bf16 (else fp16).  a_mn / b_mn: operand MN-major (else
// K-major).  M in {64, 128}, N % 16 == 0.
__host__ __device__ constexpr uint32_t idesc_f16(bool ab_bf16, int M, int N, bool a_mn = false,
                                                 bool b_mn = false) {
    return (1u << 4)                                    // D format: f32
         | ((ab_bf16 ? 1u : 0u) << 7)                   // A format
         | ((ab_bf16 ? 1u : 0u) << 10)                  // B format
         | ((a_mn ? 1u : 0u) << 15)                     // A major
         | ((b_mn ? 1u : 0u) << 16)                     // B major
         | ((uint32_t)(N >> 3) << 17)                   // N >> 3, bits 17-22
         | ((uint32_t)(M >> 4) << 24);                  // M >> 4, bits 24-28
}

// ---------------------------------------------------------------- TMEM
// Allocate `ncols` (power of two >= 32) tensor-memory columns; executed by all
// 32 lanes of one warp.  The base address is written to *dst_smem.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, issued by one thread.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when all previously issued MMAs of this thread complete.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// 16 consecutive fp32 columns of this warp's 32 TMEM lanes (lane = thread).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 2-D tiled TMA load (innermost coordinate first).
__device__ __forceinline__ void tma_load_2d(void* dst, const void* map, uint64_t* bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

// fp32 pair -> packed bf16x2 (round to nearest even), lo in the low half
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two-term bf16 split of an fp32 pair: hi = bf16(v), lo = bf16(v - hi), so that
// hi + lo carries 16 significant bits; tensor-core products of fp32 operands
// are formed as hi*hi + hi*lo + lo*hi with fp32 accumulation.
__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
    hi = pack_bf16x2(a, b);
    lo = pack_bf16x2(a - bf16lo(hi), b - bf16hi(hi));
}
// the same split of a packed fp32 pair, the residual formed by one packed subtract
__device__ __forceinline__ void split_bf16x2_packed(uint64_t v, uint32_t& hi, uint32_t& lo) {
    float a, b;
    upk2(v, a, b);
    hi = pack_bf16x2(a, b);
    const uint64_t r = add2(v, pk2(-bf16lo(hi), -bf16hi(hi)));
    float ra, rb;
    upk2(r, ra, rb);
    lo = pack_bf16x2(ra, rb);
}

// fp32 pair -> packed fp16x2 (round to nearest even)
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

}  // namespace msc
