// tc_gemm.cu -- test fixture (tcgen05 building blocks), not part of libmsc.
//
// One CTA computes D[128 x N] = A[128 x K] * B[N x K]^T with tcgen05.mma
// (kind::f16, fp32 accumulate in tensor memory) from K-major 128-byte-swizzled
// shared-memory tiles, then reads D back with tcgen05.ld.  The tiles are either
// written by CUDA cores (sw128_offset) or loaded by TMA with SWIZZLE_128B; both
// paths and the descriptor encodings of msc_tc.cuh are compared against a host
// matmul by tests/test_tc_gemm_gpu.py.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "msc_common.cuh"
#include "msc_tc.cuh"

namespace {

__device__ unsigned int g_tc_status;

__global__ void __launch_bounds__(128) tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                                                      const __grid_constant__ CUtensorMap tmB,
                                                      const uint16_t* A, const uint16_t* B, float* D, int K, int N,
                                                      int bf16, int use_tma, int a_mn, int b_mn) {
    extern __shared__ uint8_t s_dyn[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(s_dyn) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = base;                     // 128 x K
    uint8_t* sB = base + 128 * K * 2;       // N x K
    uint64_t* bar = reinterpret_cast<uint64_t*>(sB + N * K * 2);
    uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 2);
    const int tid = threadIdx.x, warp = tid >> 5;
    uint32_t ncols = 32;
    while ((int)ncols < N) ncols <<= 1;
    if (warp == 0) {
        msc::tmem_alloc(slot, ncols);
        msc::tmem_relinquish();
    }
    if (tid == 0) {
        msc::mbar_init(&bar[0], 1);
        msc::mbar_init(&bar[1], 1);
        msc::fence_barrier_init();
    }
    if (use_tma) {
        __syncthreads();
        if (tid == 0) {
            const uint32_t bytes = (uint32_t)(128 * K * 2 + N * K * 2);
            msc::mbar_arrive_expect_tx(&bar[1], bytes);
            if (a_mn) {  // A given as [K][128]: two 64-wide M blocks of K rows
                for (int mb = 0; mb < 2; ++mb) msc::tma_load_2d(sA + mb * K * 128, &tmA, &bar[1], mb * 64, 0);
            } else {
                for (int kb = 0; kb < K / 64; ++kb) msc::tma_load_2d(sA + kb * 128 * 128, &tmA, &bar[1], kb * 64, 0);
            }
            if (b_mn) {  // B given as [K][N]: N / 64 blocks of K rows
                for (int nb = 0; nb < N / 64; ++nb) msc::tma_load_2d(sB + nb * K * 128, &tmB, &bar[1], nb * 64, 0);
            } else {
                for (int kb = 0; kb < K / 64; ++kb) msc::tma_load_2d(sB + kb * N * 128, &tmB, &bar[1], kb * 64, 0);
            }
        }
        bool ok = msc::mbar_wait(&bar[1], 0, 1u << 24);
        if (!ok && tid == 0) atomicExch(&g_tc_status, 1u);
    } else {
        for (int e = tid; e < 128 * K; e += 128) {
            const int r = e / K, k = e % K;
            *reinterpret_cast<uint16_t*>(sA + msc::sw128_offset(r, k, 128)) = A[e];
        }
        for (int e = tid; e < N * K; e += 128) {
            const int r = e / K, k = e % K;
            *reinterpret_cast<uint16_t*>(sB + msc::sw128_offset(r, k, N)) = B[e];
        }
        msc::fence_proxy_async_smem();
    }
    __syncthreads();
    msc::tc_fence_after();
    const uint32_t tmem = *slot;
    if (tid == 0) {
        const uint32_t idesc = msc::idesc_f16(bf16 != 0, 128, N, a_mn != 0, b_mn != 0);
        for (int k = 0; k < K / 16; ++k) {
            const uint32_t koff = (uint32_t)((k & 3) * 32);
            const uint64_t ad = a_mn ? msc::sdesc_sw128_mn(msc::smem_u32(sA) + k * 2048, K * 128)
                                     : msc::sdesc_sw128(msc::smem_u32(sA + (k >> 2) * 128 * 128) + koff);
            const uint64_t bd = b_mn ? msc::sdesc_sw128_mn(msc::smem_u32(sB) + k * 2048, K * 128)
                                     : msc::sdesc_sw128(msc::smem_u32(sB + (k >> 2) * N * 128) + koff);
            msc::mma_f16(tmem, ad, bd, idesc, k > 0 ? 1u : 0u);
        }
        msc::mma_commit(&bar[0]);
    }
    const bool ok = msc::mbar_wait(&bar[0], 0, 1u << 24);
    if (!ok && tid == 0) atomicExch(&g_tc_status, 2u);
    msc::tc_fence_after();
    if (ok) {
        for (int c = 0; c < N; c += 16) {
            float v[16];
            msc::tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)c, v);
            msc::tmem_ld_wait();
            float* dst = D + (size_t)(32 * warp + (tid & 31)) * N + c;
#pragma unroll
            for (int i = 0; i < 16; ++i) dst[i] = v[i];
        }
    }
    msc::tc_fence_before();
    __syncthreads();
    if (warp == 0) msc::tmem_dealloc(tmem, ncols);
}

// 2-D map of a [rows][cols] tensor (cols contiguous) with boxes {64, box_rows}.
bool encode2d(CUtensorMap* m, const void* base, int rows, int cols, bool bf16) {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return false;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t str[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)rows};  // 64 contiguous elements x all rows
    cuuint32_t es[2] = {1, 1};
    return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
              const_cast<void*>(base), dims, str, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" {

// D[128 x N] = A[128 x K] B[N x K]^T; A, B, D device pointers (16-bit inputs).
// K in {64, 128}, N in {16 .. 256, multiple of 16}.  With a_mn (b_mn) the
// operand is given transposed, [K][128] ([K][N]), and used MN-major (TMA
// only; N a multiple of 64 for b_mn).  Returns 0 on success, -1 for bad
// arguments, -2 if a bounded wait ran out, else a CUDA error code.
int msc_probe_tc_gemm(const void* A, const void* B, float* D, int K, int N, int bf16, int use_tma, int a_mn,
                      int b_mn) {
    if (!(K == 64 || K == 128) || N < 16 || N > 256 || N % 16) return -1;
    if ((a_mn || b_mn) && !use_tma) return -1;
    if (b_mn && N % 64) return -1;
    CUtensorMap ta, tb;
    const bool ok_a = a_mn ? encode2d(&ta, A, K, 128, bf16 != 0) : encode2d(&ta, A, 128, K, bf16 != 0);
    const bool ok_b = b_mn ? encode2d(&tb, B, K, N, bf16 != 0) : encode2d(&tb, B, N, K, bf16 != 0);
    if (!ok_a || !ok_b) return -1;
    const int smem = 1024 + 128 * K * 2 + N * K * 2 + 64;
    cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return (int)e;
    unsigned int zero = 0;
    cudaMemcpyToSymbol(g_tc_status, &zero, sizeof(zero));
    tc_gemm_kernel<<<1, 128, smem>>>(ta, tb, static_cast<const uint16_t*>(A), static_cast<const uint16_t*>(B), D, K,
                                     N, bf16, use_tma, a_mn, b_mn);
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return (int)e;
    unsigned int st = 0;
    cudaMemcpyFromSymbol(&st, g_tc_status, sizeof(st));
    return st ? -2 : 0;
}

}  // extern "C"
