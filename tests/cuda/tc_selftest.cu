// Self-test of the tcgen05 / TMA / TMEM primitives in the library's tc.cuh:
// one CTA computes D[128][N] = A[128][K] * op(B) with bf16 operands and fp32
// accumulation, and the test compares D with a matmul on the host.
//   mode 0: A, B K-major in shared memory (B given as [N][K]), TMA-loaded.
//   mode 1: B MN-major in shared memory (B given as [K][N]), TMA-loaded.
//   mode 2: A read from tensor memory (written there with tcgen05.st),
//           B K-major as in mode 0.
//   mode 3: A MN-major in shared memory (A given as [K][128]), B K-major.
// Test-only code: built by tests/test_gpu_tc_selftest.py, never by the library.
#include <stdio.h>

#include "tc.cuh"

using namespace gdn;
using namespace gdn::tc;

__global__ void __launch_bounds__(128)
selftest_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                const __nv_bfloat16 *__restrict__ A, float *__restrict__ D, int N, int K, int mode,
                int *err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;                        // K/64 k-blocks x 128 rows x 128 B
    uint8_t *sB = smem + (K / 64) * 128 * 128; // mode 0/2: K/64 x N x 128 B; mode 1: N/64 x K x 128 B
    __shared__ uint64_t bar_load, bar_mma;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5;
    if (warp == 0) {
        tmem_alloc(&tmem_base, 256);
        tmem_relinquish();
    }
    if (tid == 0) {
        abort_flag = 0;
        mbar_init(&bar_load, 1);
        mbar_init(&bar_mma, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base;
    const uint32_t a_col = 128;                // A (mode 2) lives in columns [128, 128 + K/2)

    if (tid == 0) {
        uint32_t bytes = (mode == 2 ? 0u : 128u * K * 2u) + (uint32_t)N * K * 2u;
        mbar_arrive_expect_tx(&bar_load, bytes);
        if (mode == 3)
            for (int mb = 0; mb < 2; ++mb) tma_load_2d(sA + mb * K * 128, &mapA, &bar_load, mb * 64, 0);
        else if (mode != 2)
            for (int kb = 0; kb < K / 64; ++kb) tma_load_2d(sA + kb * 128 * 128, &mapA, &bar_load, kb * 64, 0);
        if (mode == 1) {
            for (int nb = 0; nb < N / 64; ++nb) tma_load_2d(sB + nb * K * 128, &mapB, &bar_load, nb * 64, 0);
        } else {
            for (int kb = 0; kb < K / 64; ++kb) tma_load_2d(sB + kb * N * 128, &mapB, &bar_load, kb * 64, 0);
        }
    }
    if (mode == 2) {
        // row tid of A into TMEM lane tid, bf16 pairs packed low-element-first
        const uint32_t lane_base = (uint32_t)(warp * 32);
        for (int c0 = 0; c0 < K; c0 += 64) {
            uint32_t r[32];
            for (int j = 0; j < 32; ++j)
                r[j] = pack_bf16(__bfloat162float(A[tid * K + c0 + 2 * j]),
                                 __bfloat162float(A[tid * K + c0 + 2 * j + 1]));
            tmem_st32(tmem_addr(tbase, lane_base, a_col + c0 / 2), r);
        }
        tmem_wait_st();
        tc_fence_before();
    }
    __syncthreads();
    if (tid == 0) {
        tc_fence_after();
        if (!mbar_wait(&bar_load, 0, &abort_flag)) atomicOr(err, 1);
        const uint32_t idesc = idesc_bf16(128, N, mode == 3, mode == 1);
        for (int s = 0; s < K / 16; ++s) {
            uint64_t bdesc;
            if (mode == 1)
                bdesc = sdesc_sw128(smem_u32(sB) + s * 16 * 128, K * 128, 1024);
            else
                bdesc = sdesc_sw128(smem_u32(sB) + (s / 4) * N * 128 + (s % 4) * 32, 16, 1024);
            if (mode == 2) {
                mma_ts(tbase, tbase + a_col + s * 8, bdesc, idesc, s > 0);
            } else if (mode == 3) {
                uint64_t adesc = sdesc_sw128(smem_u32(sA) + s * 16 * 128, K * 128, 1024);
                mma_ss(tbase, adesc, bdesc, idesc, s > 0);
            } else {
                uint64_t adesc = sdesc_sw128(smem_u32(sA) + (s / 4) * 128 * 128 + (s % 4) * 32, 16, 1024);
                mma_ss(tbase, adesc, bdesc, idesc, s > 0);
            }
        }
        mma_commit(&bar_mma);
    }
    if (!mbar_wait(&bar_mma, 0, &abort_flag)) atomicOr(err, 2);
    tc_fence_after();
    for (int c0 = 0; c0 < N; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tmem_addr(tbase, warp * 32, c0), r);
        for (int j = 0; j < 32; ++j) D[tid * N + c0 + j] = __uint_as_float(r[j]);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 256);
}

extern "C" int tc_selftest_gemm(const void *A, const void *B, float *D, int N, int K, int mode,
                                int *err_dev) {
    if ((N != 64 && N != 128) || (K != 64 && K != 128) || mode < 0 || mode > 3) return 1;
    CUtensorMap mA, mB;
    bool okA = mode == 3 ? encode_tmap_2d_bf16(&mA, A, 128, K, 128, 64, K)
                         : encode_tmap_2d_bf16(&mA, A, K, 128, K, 64, 128);
    if (!okA) return 2;
    bool ok = mode == 1 ? encode_tmap_2d_bf16(&mB, B, N, K, N, 64, K)
                        : encode_tmap_2d_bf16(&mB, B, K, N, K, 64, N);
    if (!ok) return 3;
    size_t smem = 1024 + (size_t)128 * K * 2 + (size_t)N * K * 2;
    cudaFuncSetAttribute(selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    selftest_kernel<<<1, 128, smem>>>(mA, mB, (const __nv_bfloat16 *)A, D, N, K, mode, err_dev);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        fprintf(stderr, "launch: %s\n", cudaGetErrorString(e));
        return 4;
    }
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        fprintf(stderr, "sync: %s\n", cudaGetErrorString(e));
        return 5;
    }
    return 0;
}
