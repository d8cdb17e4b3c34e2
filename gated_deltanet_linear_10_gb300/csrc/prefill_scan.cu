// The chunk-state scan of one long sequence (the long-context prefill of
// "[Feature] Qwen3-Next-80B-A3B Support", lmdeploy issue 3961: the model's
// native 262k context): the small kernels around the two-kernel prefill.
//
// The chain over a segment is affine in its initial state: S_end = S_0 A + B
// and o = o(0) + S_0 Phi, where A is the product of the chunk transitions and
// Phi the map from the state to the outputs.  The sequence is cut at a chunk
// boundary into segments 0 and 1; one chain launch runs segment 0 from the
// true initial state (final outputs, final state S_1), segment 1 from zero
// (outputs o(0) and state B) and segment 1 again from the identity with v = 0
// (state A, outputs Phi), so the serial chain is half as long.  Then
//   scan_combine_kernel:  S_final = S_1 A + B (fp32), and S_1 as a bf16
//                         tensor-core operand;
//   scan_correct_kernel:  o(segment 1) += S_1 Phi^T on tcgen05.
// scan_setup_kernel derives the segment bounds and slot lists on the device
// from cu_seqlens and the caller's slot indices.
#include "tc.cuh"
#include "common.cuh"
#include "prefill_scan.cuh"

namespace gdn {

GDN_DECLARE_STATUS_WORD(g_status_prefill_scan)
GDN_STATUS_READER(read_status_prefill_scan, g_status_prefill_scan)

namespace scan {
using namespace tc;

__global__ void scan_setup_kernel(const int32_t *__restrict__ cu, int64_t n_tokens,
                                  const int32_t *__restrict__ init_idx,
                                  const int32_t *__restrict__ final_idx, int64_t n_slots,
                                  ScanIdx *__restrict__ out) {
    if (threadIdx.x != 0) return;
    const int32_t a = cu[0], e = cu[1];
    ScanIdx r;
    if (a < 0 || e < a || e > n_tokens) {   // nothing runs, nothing is written
        flag_status(GDN_DEVSTAT_BAD_SEQLEN);
        r.cu_all[0] = r.cu_all[1] = r.cu_all[2] = 0;
        r.init[0] = r.init[1] = -1;
        r.fin[0] = r.fin[1] = -1;
        r.final_slot = -1;
    } else {
        const int64_t nch = ((int64_t)e - a + kChunk - 1) / kChunk;
        const int64_t m = (int64_t)a + kChunk * ((nch + 1) / 2);   // segment 0: the first half
        r.cu_all[0] = a;
        r.cu_all[1] = (int32_t)(m < e ? m : e);
        r.cu_all[2] = e;
        r.init[0] = init_idx ? init_idx[0] : -1;   // checked by the chain kernel
        r.init[1] = -1;                            // segment 1 from zero
        r.fin[0] = kSlotS1;
        r.fin[1] = kSlotB;
        int32_t fs = final_idx ? final_idx[0] : -1;
        if (fs >= n_slots) {
            flag_status(GDN_DEVSTAT_BAD_INDEX);
            fs = -1;
        }
        r.final_slot = fs;
    }
    *out = r;
}

// Four CTAs of 256 threads per V head, 32 state rows each: S_final = S_1 A +
// B in fp32 (thread (ty, tx) owns rows 2 ty, 2 ty + 1 of the CTA's rows and
// columns 8 tx .. 8 tx + 7), and those rows of S_1 rounded to bf16 in the
// 128-byte-swizzled K-major layout of a 128 x 128 tcgen05 A operand (two
// k-blocks of 128 rows x 128 B).
constexpr int kCombThreads = 256;
constexpr int kCombRows = 32;    // rows of S per CTA
constexpr int kKt = 16;          // k-tile
__global__ void __launch_bounds__(kCombThreads)
scan_combine_kernel(const float *__restrict__ states, int hv, const ScanIdx *__restrict__ idx,
                    float *__restrict__ pool, uint8_t *__restrict__ s1b) {
    __shared__ float As[kCombRows][kKt + 1];
    __shared__ float Bs[kKt][128 + 4];
    const int h = blockIdx.x, rb = blockIdx.y * kCombRows, t = threadIdx.x;
    const size_t slot = (size_t)hv * 128 * 128, head = (size_t)h * 128 * 128;
    const float *S1 = states + kSlotS1 * slot + head;
    const float *Bm = states + kSlotB * slot + head;
    const float *Am = states + kSlotA * slot + head;
    const int ty = t >> 4, tx = t & 15;
    const int r0 = rb + 2 * ty;
    float acc[2][8];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float4 b0 = *reinterpret_cast<const float4 *>(Bm + (r0 + i) * 128 + 8 * tx);
        const float4 b1 = *reinterpret_cast<const float4 *>(Bm + (r0 + i) * 128 + 8 * tx + 4);
        acc[i][0] = b0.x; acc[i][1] = b0.y; acc[i][2] = b0.z; acc[i][3] = b0.w;
        acc[i][4] = b1.x; acc[i][5] = b1.y; acc[i][6] = b1.z; acc[i][7] = b1.w;
    }
    for (int k0 = 0; k0 < 128; k0 += kKt) {
        for (int e = t; e < kCombRows * kKt; e += kCombThreads) {
            const int r = e / kKt, c = e % kKt;
            As[r][c] = S1[(rb + r) * 128 + k0 + c];
        }
        for (int e = t; e < kKt * 128; e += kCombThreads) {
            const int kr = e / 128, kc = e % 128;
            Bs[kr][kc] = Am[(k0 + kr) * 128 + kc];
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kKt; ++kk) {
            const float a0 = As[2 * ty][kk], a1 = As[2 * ty + 1][kk];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float b = Bs[kk][8 * tx + j];
                acc[0][j] = fmaf(a0, b, acc[0][j]);
                acc[1][j] = fmaf(a1, b, acc[1][j]);
            }
        }
        __syncthreads();
    }
    const int fs = idx->final_slot;
    if (fs >= 0) {
        float *dst = pool + (size_t)fs * slot + head;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            *reinterpret_cast<float4 *>(dst + (r0 + i) * 128 + 8 * tx) =
                make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
            *reinterpret_cast<float4 *>(dst + (r0 + i) * 128 + 8 * tx + 4) =
                make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
        }
    }
    // this CTA's rows of S_1 -> bf16 operand: one 16-byte chunk (8 columns) per step
    uint8_t *out = s1b + (size_t)h * kS1bBytes;
    for (int e = t; e < kCombRows * 16; e += kCombThreads) {
        const int r = rb + (e >> 4), ch = e & 15;   // row r, columns 8 ch .. 8 ch + 7
        const float4 x0 = *reinterpret_cast<const float4 *>(S1 + r * 128 + 8 * ch);
        const float4 x1 = *reinterpret_cast<const float4 *>(S1 + r * 128 + 8 * ch + 4);
        const uint4 w = make_uint4(pack_bf16(x0.x, x0.y), pack_bf16(x0.z, x0.w),
                                   pack_bf16(x1.x, x1.y), pack_bf16(x1.z, x1.w));
        *reinterpret_cast<uint4 *>(out + (ch >> 3) * 16384 + sw128_chunk(r, ch & 7)) = w;
    }
}

// One CTA of 256 threads per (128-token tile of segment 1, V head):
//   D[b][t] = sum_a S_1[b][a] Phi[t][a]        (tcgen05, M = N = K = 128)
//   o[t][h][b] += D[b][t]
// A = S_1 (bf16 operand from scan_combine_kernel, one bulk copy), B = the
// Phi tile (TMA, 128-byte swizzle); the o tile [t][b] comes in by TMA, is
// updated in shared memory and leaves by one TMA store.  Warp w reads TMEM
// lanes 32 (w % 4) .. + 31 (value rows b) for the tokens of its half, 64 (w / 4)
// .. + 63; each thread updates column b of those tokens.  Rows of the tile
// past segment 1 go back unchanged.
constexpr int kCorrThreads = 256;
constexpr uint32_t kCorrTmemCols = 128;
constexpr uint32_t kOTile = 128 * 128 * 2;
struct CorrBars {
    uint64_t full, mma_done;
    uint32_t tmem_base;
    int abort;
};
constexpr uint32_t kCorrSmem = 2 * kS1bBytes + kOTile + 128 + 1024;

__global__ void __launch_bounds__(kCorrThreads)
scan_correct_kernel(const __grid_constant__ CUtensorMap tm_phi,
                    const __grid_constant__ CUtensorMap tm_o, const uint8_t *__restrict__ s1b,
                    const ScanIdx *__restrict__ idx) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    uint8_t *at = sm, *bt = sm + kS1bBytes;
    __nv_bfloat16 *ot = reinterpret_cast<__nv_bfloat16 *>(sm + 2 * kS1bBytes);
    CorrBars &B = *reinterpret_cast<CorrBars *>(sm + 2 * kS1bBytes + kOTile);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = blockIdx.x, h = blockIdx.y;
    const int64_t r0 = idx->cu_all[1], r1 = idx->cu_all[2];
    if ((int64_t)tile * 128 >= r1 - r0) return;        // past segment 1 (CTA-uniform)
    const int row0 = (int)(r0 + (int64_t)tile * 128);

    if (warp == 0) {
        tmem_alloc(&B.tmem_base, kCorrTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&B.full, 1);
        mbar_init(&B.mma_done, 1);
        B.abort = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = B.tmem_base;
    volatile int *abort = &B.abort;

    if (tid == 0) {
        mbar_arrive_expect_tx(&B.full, 2 * kS1bBytes + kOTile);
        bulk_load(at, s1b + (size_t)h * kS1bBytes, kS1bBytes, &B.full);
        for (int kb = 0; kb < 2; ++kb)
            tma_load_2d(bt + kb * 16384, &tm_phi, &B.full, h * 128 + kb * 64, tile * 128);
        tma_load_2d(ot, &tm_o, &B.full, h * 128, row0);
        bool ok = mbar_wait(&B.full, 0, abort);
        if (!ok) {
            int z = 0;            // never leave with a copy in flight
            mbar_wait(&B.full, 0, &z);
        } else {
            tc_fence_after();
            const uint32_t id = idesc_bf16(128, 128);
            const uint32_t a0 = smem_u32(at), b0 = smem_u32(bt);
            for (int s = 0; s < 8; ++s) {
                const uint32_t off = (s >> 2) * 16384 + (s & 3) * 32;
                mma_ss(tbase, sdesc_sw128(a0 + off, 16, 1024), sdesc_sw128(b0 + off, 16, 1024), id,
                       s > 0);
            }
        }
        mma_commit(&B.mma_done);   // arrives at once when no MMA was issued
    }
    __syncwarp();
    const bool done = mbar_wait(&B.mma_done, 0, abort);
    tc_fence_after();
    const bool go = __all_sync(0xffffffffu, done && !*abort);   // warp-uniform: tcgen05.ld is .aligned
    if (go) {
        const int q4 = warp & 3, half = warp >> 2;
        const int b = q4 * 32 + lane;
        const int nrow = (int)min((int64_t)128, r1 - row0);     // rows of segment 1 in the tile
        for (int j = 2 * half; j < 2 * half + 2; ++j) {
            uint32_t r[32];
            tmem_ld32(tmem_addr(tbase, q4 * 32, 32 * j), r);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int t = 32 * j + i;
                if (t < nrow)
                    ot[t * 128 + b] = __float2bfloat16_rn(__bfloat162float(ot[t * 128 + b]) +
                                                         __uint_as_float(r[i]));
            }
        }
    }
    fence_async_smem();
    __syncthreads();
    if (tid == 0) {
        if (!*abort) {
            tma_store_2d(&tm_o, ot, h * 128, row0);
            bulk_commit();
            bulk_wait_read_all();
        }
        int z = 0;                // no MMA may still write TMEM when it is freed
        mbar_wait(&B.mma_done, 0, &z);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tbase, kCorrTmemCols);
    }
    if (tid == 0 && B.abort) flag_status(GDN_DEVSTAT_TIMEOUT);
}

}  // namespace scan

gdn_status scan_setup(const int32_t *cu, int64_t n_tokens, const int32_t *ii, const int32_t *fi,
                      int64_t n_slots, scan::ScanIdx *idx, cudaStream_t s) {
    scan::scan_setup_kernel<<<1, 32, 0, s>>>(cu, n_tokens, ii, fi, n_slots, idx);
    return launch_status();
}

gdn_status scan_finish(const float *states, int hv, const scan::ScanIdx *idx, float *pool,
                       uint8_t *s1b, const void *phi, int64_t phi_rows, void *o, int64_t n_tokens,
                       cudaStream_t s) {
    scan::scan_combine_kernel<<<dim3((unsigned)hv, 128 / scan::kCombRows), scan::kCombThreads, 0,
                                 s>>>(states, hv, idx, pool, s1b);
    gdn_status st = launch_status();
    if (st != GDN_OK) return st;
    CUtensorMap tm, tmo;
    if (!encode_tmap_2d_bf16(&tm, phi, (uint64_t)hv * 128, (uint64_t)phi_rows, (uint64_t)hv * 128,
                             64, 128, true) ||
        !encode_tmap_2d_bf16(&tmo, o, (uint64_t)hv * 128, (uint64_t)n_tokens, (uint64_t)hv * 128,
                             128, 128, false))
        return GDN_ERR_LAUNCH;
    const cudaError_t e = cudaFuncSetAttribute(
        scan::scan_correct_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)scan::kCorrSmem);
    if (e != cudaSuccess) {
        set_last_cuda_error(e);
        return GDN_ERR_LAUNCH;
    }
    const dim3 grid((unsigned)((phi_rows + 127) / 128), (unsigned)hv);
    scan::scan_correct_kernel<<<grid, scan::kCorrThreads, scan::kCorrSmem, s>>>(tm, tmo, s1b,
                                                                                 idx);
    return launch_status();
}

}  // namespace gdn
