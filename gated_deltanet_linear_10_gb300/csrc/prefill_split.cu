// Chunked prefill in two kernels, for callers that pass a workspace
// ("Flash Linear Attention operations for efficient chunked computations",
// "[model] Support Qwen3next", Highlights).  Same arithmetic as the fused
// tensor-core kernel (prefill_tc.cu), split where the dependency structure
// allows it:
//
//   1. prep_kernel: everything that does not depend on the state, for every
//      (chunk, V head) item at once -- chunk-parallel, several CTAs per SM:
//      G = [K;Q] K^T on the tensor cores, gates, norms, A and P, the UT solve
//      T = (I + A)^-1, and T1 = T diag(beta), T2 = -T diag(beta Gam r_k).
//      Each item's T1 | T2 | P | scalars block (25 KiB) is written to the
//      workspace in exactly the shared-memory layout the MMAs read.
//   2. chain_kernel: per (sequence, V head) only the state chain, with the
//      item blocks streamed in by 1-D bulk copies next to the K|Q and V tiles.
//
// Workspace: [chunk offsets, int32 x (n_seqs + 1), padded to 1 KiB]
//            [items: (ceil(n_tokens / 64) + n_seqs) x hv blocks of kItemBytes]
#include "prefill_common.cuh"

namespace gdn {

GDN_DECLARE_STATUS_WORD(g_status_prefill_split)
GDN_STATUS_READER(read_status_prefill_split, g_status_prefill_split)

namespace psp {
using namespace ptc;

// item block: T1 | T2 | P (bf16, 128-byte swizzle, K-major) | scalars
constexpr uint32_t kItemScal = 3 * kMatBytes;
struct ItemScal {
    float ks[C];      // D[last][j] r_k,j      (K'' row factors)
    float sq[C];      // scale Gam_i r_q,i     (Q' row factors)
    float gam_n;      // total decay of the chunk
    int n;            // valid rows
};
constexpr uint32_t kItemBytes = (kItemScal + sizeof(ItemScal) + 1023) / 1024 * 1024;

__host__ __device__ inline size_t header_bytes(int n_seqs) {
    return ((size_t)4 * (n_seqs + 1) + 1023) / 1024 * 1024;
}
__host__ __device__ inline int64_t chunk_bound(int64_t n_tokens, int n_seqs) {
    return (n_tokens + C - 1) / C + n_seqs;
}

// chunk_base[s] = sum over sequences before s of ceil(len / 64); one CTA.
// A sequence whose bounds are invalid gets no chunks (the chain kernel
// reports it).
__device__ __forceinline__ int seq_chunks(const int32_t *cu, int s, int64_t n_tokens) {
    const int32_t a = cu[s], e = cu[s + 1];
    return (a < 0 || e < a || e > n_tokens) ? 0 : (e - a + C - 1) / C;
}

__global__ void __launch_bounds__(1024) chunk_base_kernel(const int32_t *__restrict__ cu,
                                                          int n_seqs, int64_t n_tokens,
                                                          int32_t *__restrict__ base) {
    __shared__ int warp_tot[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (n_seqs + 1023) / 1024;
    const int s0 = min(n_seqs, tid * per), s1 = min(n_seqs, s0 + per);
    int local = 0;
    for (int s = s0; s < s1; ++s) local += seq_chunks(cu, s, n_tokens);
    int x = local;   // inclusive warp scan
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = warp_tot[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += y;
        }
        warp_tot[lane] = w;    // inclusive over warps
    }
    __syncthreads();
    int run = x - local + (warp > 0 ? warp_tot[warp - 1] : 0);   // exclusive
    for (int s = s0; s < s1; ++s) {
        base[s] = run;
        run += seq_chunks(cu, s, n_tokens);
    }
    if (tid == 1023) base[n_seqs] = warp_tot[31];
}

// ------------------------------------------------------------ prep kernel --
constexpr int kPrepWarps = 9;              // warp 0: TMA + MMA + TMEM; warps 1..8: prep
constexpr int kPrepKernelThreads = kPrepWarps * 32;
constexpr int kPrepThreads = 256;

struct PrepScal {
    float beta[C], gam[C], alpha[C], rk[C], rq[C], xs[C];
};
struct PrepBars {
    uint64_t kq_full, g_full;
    uint32_t tmem_base;
    int abort;
};
// The raw K|Q tile is dead once G is in TMEM and the norms are taken: its
// first kItemCopy bytes then stage the item block, the rest the solve scratch.
constexpr uint32_t kItemCopy = (kItemScal + sizeof(ItemScal) + 15) / 16 * 16;
constexpr uint32_t P_OFF_KQ = 0;
constexpr uint32_t P_OFF_WB = P_OFF_KQ + 25600;
constexpr uint32_t kPWbFloats = 8 * 16 * kWbLd + 16 * 16;
constexpr uint32_t P_OFF_AF = P_OFF_KQ + kKQBytes;
constexpr uint32_t P_OFF_TF = P_OFF_AF + C * kLd * 4;
constexpr uint32_t P_OFF_SCAL = P_OFF_TF + C * kLd * 4;
constexpr uint32_t P_OFF_BARS = P_OFF_SCAL + (sizeof(PrepScal) + 127) / 128 * 128;
constexpr uint32_t P_SMEM_BYTES = P_OFF_BARS + 128 + 1024;   // + slack to align to 1024
constexpr uint32_t kPrepTmemCols = 64;
static_assert(kItemCopy <= P_OFF_WB && P_OFF_WB + kPWbFloats * 4 <= kKQBytes, "staging layout");
static_assert(sizeof(PrepBars) <= 128, "barrier block");
static_assert(3 * (P_SMEM_BYTES + 1024) <= 233472, "three prep CTAs per SM");

// One CTA per (chunk, V head) item.  Warp 0: TMEM, TMA of the raw K|Q tile,
// M1 G = [K;Q] K^T; warps 1..8: the prep arithmetic (as in the fused kernel),
// then one bulk store of the item block.
__global__ void __launch_bounds__(kPrepKernelThreads, 3)
prep_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const float *__restrict__ g, const float *__restrict__ beta,
            const int32_t *__restrict__ cu, const int32_t *__restrict__ base, int n_seqs, int hv,
            int grp, float scale, int l2norm, uint8_t *__restrict__ items) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    PrepBars &B = *reinterpret_cast<PrepBars *>(sm + P_OFF_BARS);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int it = (int)(blockIdx.x / (unsigned)hv);
    const int h = (int)blockIdx.x - it * hv;
    if (it >= base[n_seqs]) return;
    int lo = 0, hi = n_seqs - 1;          // the sequence: last s with base[s] <= it
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (base[mid] <= it) lo = mid; else hi = mid - 1;
    }
    const int64_t c0 = cu[lo] + (int64_t)(it - base[lo]) * C;
    const int n = (int)min((int64_t)C, (int64_t)cu[lo + 1] - c0);
    const int hq = h / grp;
    uint8_t *kq = sm + P_OFF_KQ;

    if (warp == 0) {
        tmem_alloc(&B.tmem_base, kPrepTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&B.kq_full, 1);
        mbar_init(&B.g_full, 1);
        B.abort = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = B.tmem_base;
    volatile int *abort = &B.abort;

    if (warp == 0) {
        if (lane == 0) {
            mbar_arrive_expect_tx(&B.kq_full, kKQBytes);
            for (int kb = 0; kb < 2; ++kb) {
                tma_load_2d(kq + kb * kKBlk, &tm_k, &B.kq_full, hq * DH + kb * 64, (int)c0);
                tma_load_2d(kq + kb * kKBlk + 64 * 128, &tm_q, &B.kq_full, hq * DH + kb * 64, (int)c0);
            }
            if (mbar_wait(&B.kq_full, 0, abort)) {
                tc_fence_after();
                const uint32_t id64 = idesc_bf16(128, 64);
                const uint32_t kb0 = smem_u32(kq);
                for (int s = 0; s < 8; ++s) {
                    const uint32_t off = (s >> 2) * kKBlk + (s & 3) * 32;
                    mma_ss(tbase, sdesc_sw128(kb0 + off, 16, 1024), sdesc_sw128(kb0 + off, 16, 1024),
                           id64, s > 0);
                }
                mma_commit(&B.g_full);
                int z = 0;       // TMEM is freed at the end: the MMAs must be done
                mbar_wait(&B.g_full, 0, &z);
            } else {
                int z = 0;       // never leave with the copy in flight
                mbar_wait(&B.kq_full, 0, &z);
            }
        }
        __syncwarp();
    } else {
        const int t = tid - 32;                 // 0 .. 255
        const int pw = warp - 1;                // 0 .. 7
        const int q4 = warp & 3;                // TMEM lane quadrant
        const int p = q4 * 32 + lane;           // G row: 0..63 K rows, 64..127 Q rows
        const int chalf = pw >> 2;              // which 32 G columns this warp reads
        PrepScal &S = *reinterpret_cast<PrepScal *>(sm + P_OFF_SCAL);
        float *Af = reinterpret_cast<float *>(sm + P_OFF_AF);
        float *Tf = reinterpret_cast<float *>(sm + P_OFF_TF);
        float *Wb = reinterpret_cast<float *>(sm + P_OFF_WB);
        ItemScal &I = *reinterpret_cast<ItemScal *>(kq + kItemScal);
        float g0 = 0.f, g1 = 0.f, b0 = 0.f, b1 = 0.f;
        if (t < 32) {
            if (2 * t < n) {
                g0 = g[(c0 + 2 * t) * hv + h];
                b0 = beta[(c0 + 2 * t) * hv + h];
            }
            if (2 * t + 1 < n) {
                g1 = g[(c0 + 2 * t + 1) * hv + h];
                b1 = beta[(c0 + 2 * t + 1) * hv + h];
            }
        }
        mbar_wait(&B.kq_full, 0, abort);
        {
            const float r = kq_row_inv_norm(kq, t, l2norm);
            const int row = t >> 1;
            if ((t & 1) == 0) {
                if (row < C) S.rk[row] = r; else S.rq[row - C] = r;
            }
        }
        if (t < 32) {   // prefix sum of g, per-token decay alpha = exp(g)
            float x = g0 + g1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, x, off);
                if (lane >= off) x += y;
            }
            S.gam[2 * t] = x - g1;
            S.gam[2 * t + 1] = x;
            S.beta[2 * t] = b0;
            S.beta[2 * t + 1] = b1;
            S.alpha[2 * t] = __expf(g0);
            S.alpha[2 * t + 1] = __expf(g1);
        }
        named_sync(1, kPrepThreads);
        float ksv = 0.f, sqv = 0.f, gl = 0.f;
        if (t < C) {
            gl = S.gam[C - 1];                  // padded rows carry g = 0
            const float x = S.gam[t];
            const bool ok = t < n;
            const float ex = __expf(x);
            S.xs[t] = ok ? ex * S.rk[t] : 0.f;
            ksv = ok ? __expf(gl - x) * S.rk[t] : 0.f;
            sqv = ok ? scale * ex * S.rq[t] : 0.f;
        }
        mbar_wait(&B.g_full, 0, abort);
        tc_fence_after();
        uint32_t gr[32];
        tmem_ld32(tmem_addr(tbase, q4 * 32, 32 * chalf), gr);
        // the raw tile is dead from here on: it becomes the item staging area
        g_to_a_p(gr, p, chalf, n, S.beta, S.gam, S.alpha, S.rk, S.rq, scale, Af, kq + 2 * kMatBytes);
        if (t < C) {
            I.ks[t] = ksv;
            I.sq[t] = sqv;
            if (t == 0) {
                I.gam_n = __expf(gl);
                I.n = n;
            }
        }
        named_sync(1, kPrepThreads);
        ut_solve(Af, Tf, Wb, t, pw, lane, S.beta, S.xs, kq);
        fence_async_smem();
        named_sync(1, kPrepThreads);
        if (t == 0 && !*abort) {
            bulk_store(items + ((size_t)it * hv + h) * kItemBytes, kq, kItemCopy);
            bulk_commit();
            bulk_wait_all();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tbase, kPrepTmemCols);
    }
    if (tid == 0 && B.abort) flag_status(GDN_DEVSTAT_TIMEOUT);
}

// ------------------------------------------------------------ chain kernel --
// One CTA per (sequence, V head): only the state chain of the fused kernel
// (MU, M23, E1, M4, E2, M5, M6, E3), its per-chunk operands read from the
// item blocks.  Warp 0: TMA / bulk producer; warp 1: TMEM + MMA issue;
// warps 2..5: the epilogues.
constexpr int kChainWarps = 6;
constexpr int kChainKernelThreads = kChainWarps * 32;
constexpr int kChainThreads = 128;
constexpr int kKQStages = 3, kVStages = 2, kDStages = 3;
constexpr uint32_t kColS32 = 0, kColS16 = 128, kColU = 192, kColX = 256, kColO = 320,
                   kTmemCols = 512;   // X and O adjacent: one N = 128 MMA

struct ChainBars {
    uint64_t kq_full[kKQStages], kq_empty[kKQStages], v_full[kVStages], v_empty[kVStages],
        d_full[kDStages], d_empty[kDStages];
    uint64_t x_full, r_full, u_full, u2_full, s_full, s_next, mma_done;
    uint32_t tmem_base;
    int abort;
    int seq;
};
constexpr uint32_t C_OFF_KQ = 0;
constexpr uint32_t C_OFF_V = C_OFF_KQ + kKQStages * kKQBytes;
constexpr uint32_t C_OFF_D = C_OFF_V + kVStages * kVBytes;
constexpr uint32_t C_OFF_BARS = C_OFF_D + kDStages * kItemBytes;
constexpr uint32_t C_SMEM_BYTES = C_OFF_BARS + (sizeof(ChainBars) + 127) / 128 * 128 + 1024;
static_assert(kItemBytes % 1024 == 0, "item stages stay 1024-aligned");
static_assert(kDStages == kKQStages, "one stage index for K|Q and items");
static_assert(C_SMEM_BYTES <= 232448, "shared memory budget");

__global__ void __launch_bounds__(kChainKernelThreads, 1)
chain_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
             const __grid_constant__ CUtensorMap tm_v, const int32_t *__restrict__ cu,
             const int32_t *__restrict__ base, int n_seqs, int64_t n_tokens, int hv, int grp,
             const uint8_t *__restrict__ items, float *__restrict__ pool, int64_t n_slots,
             const int32_t *__restrict__ init_idx, const int32_t *__restrict__ final_idx,
             __nv_bfloat16 *__restrict__ o) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    ChainBars &B = *reinterpret_cast<ChainBars *>(sm + C_OFF_BARS);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const int rank = blockIdx.x / hv;
    const int h = blockIdx.x - rank * hv;
    const int hq = h / grp;
    const int seq = seq_for_rank(cu, n_seqs, rank, &B.seq);
    const int64_t s_start = cu[seq], s_end = cu[seq + 1];
    int64_t islot = init_idx ? init_idx[seq] : -1;
    int64_t fslot = final_idx ? final_idx[seq] : -1;
    if (islot >= n_slots || fslot >= n_slots) {
        if (tid == 0) flag_status(GDN_DEVSTAT_BAD_INDEX);
        if (islot >= n_slots) islot = -1;
        if (fslot >= n_slots) fslot = -1;
    }
    if (s_start < 0 || s_end < s_start || s_end > n_tokens) {
        if (tid == 0) flag_status(GDN_DEVSTAT_BAD_SEQLEN);
        return;
    }
    const int nch = (int)((s_end - s_start + C - 1) / C);
    const size_t head_off = (size_t)h * DH * DH;
    const size_t slot_stride = (size_t)hv * DH * DH;
    if (nch == 0) {   // empty sequence: the initial state (or zero) is the final state
        if (fslot >= 0)
            for (int e = tid; e < DH * DH; e += kChainKernelThreads)
                pool[fslot * slot_stride + head_off + e] =
                    islot >= 0 ? pool[islot * slot_stride + head_off + e] : 0.f;
        return;
    }
    const int64_t item0 = base[seq];

    if (warp == 1) {
        tmem_alloc(&B.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < kKQStages; ++s) { mbar_init(&B.kq_full[s], 1); mbar_init(&B.kq_empty[s], 1); }
        for (int s = 0; s < kVStages; ++s) { mbar_init(&B.v_full[s], 1); mbar_init(&B.v_empty[s], 1); }
        for (int s = 0; s < kDStages; ++s) {
            mbar_init(&B.d_full[s], 1);
            mbar_init(&B.d_empty[s], 1 + kChainThreads);   // the MMAs and the epilogues
        }
        mbar_init(&B.x_full, 1);
        mbar_init(&B.r_full, kChainThreads);
        mbar_init(&B.u_full, 1);
        mbar_init(&B.u2_full, kChainThreads);
        mbar_init(&B.s_full, 1);
        mbar_init(&B.s_next, kChainThreads);
        mbar_init(&B.mma_done, 1);
        B.abort = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = B.tmem_base;
    volatile int *abort = &B.abort;

    if (warp == 0) {
        // ------------------------------------------------ TMA / bulk producer
        if (lane == 0) {
            prefetch_tensormap(&tm_q);
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
            int kq_issued[kKQStages] = {0, 0, 0}, d_issued[kDStages] = {0, 0, 0},
                v_issued[kVStages] = {0, 0};
            for (int c = 0; c < nch && !*abort; ++c) {
                const int y = (int)(s_start + (int64_t)c * C);
                const int sk = c % kKQStages, sv = c % kVStages;
                if (c >= kKQStages) mbar_wait(&B.kq_empty[sk], ((c / kKQStages) - 1) & 1, abort);
                uint8_t *kq = sm + C_OFF_KQ + sk * kKQBytes;
                mbar_arrive_expect_tx(&B.kq_full[sk], kKQBytes);
                for (int kb = 0; kb < 2; ++kb) {
                    tma_load_2d(kq + kb * kKBlk, &tm_k, &B.kq_full[sk], hq * DH + kb * 64, y);
                    tma_load_2d(kq + kb * kKBlk + 64 * 128, &tm_q, &B.kq_full[sk], hq * DH + kb * 64, y);
                }
                kq_issued[sk] = c / kKQStages + 1;
                if (c >= kDStages) mbar_wait(&B.d_empty[sk], ((c / kDStages) - 1) & 1, abort);
                mbar_arrive_expect_tx(&B.d_full[sk], kItemCopy);
                bulk_load(sm + C_OFF_D + sk * kItemBytes, items + ((item0 + c) * hv + h) * kItemBytes,
                          kItemCopy, &B.d_full[sk]);
                d_issued[sk] = c / kDStages + 1;
                if (c >= kVStages) mbar_wait(&B.v_empty[sv], ((c / kVStages) - 1) & 1, abort);
                uint8_t *vt = sm + C_OFF_V + sv * kVBytes;
                mbar_arrive_expect_tx(&B.v_full[sv], kVBytes);
                for (int kb = 0; kb < 2; ++kb)
                    tma_load_2d(vt + kb * kVBlk, &tm_v, &B.v_full[sv], h * DH + kb * 64, y);
                v_issued[sv] = c / kVStages + 1;
            }
            // never leave with copies in flight: wait for the last load of every stage
            for (int s = 0; s < kKQStages; ++s)
                if (kq_issued[s]) { int z = 0; mbar_wait(&B.kq_full[s], (kq_issued[s] - 1) & 1, &z); }
            for (int s = 0; s < kDStages; ++s)
                if (d_issued[s]) { int z = 0; mbar_wait(&B.d_full[s], (d_issued[s] - 1) & 1, &z); }
            for (int s = 0; s < kVStages; ++s)
                if (v_issued[s]) { int z = 0; mbar_wait(&B.v_full[s], (v_issued[s] - 1) & 1, &z); }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t id64 = idesc_bf16(128, 64);
            const uint32_t id64amn = idesc_bf16(128, 64, true, false);
            const uint32_t id128 = idesc_bf16(128, 128);
            const uint32_t id128bmn = idesc_bf16(128, 128, false, true);
            for (int c = 0; c < nch; ++c) {
                const int sk = c % kKQStages, sv = c % kVStages;
                const uint32_t kqb = smem_u32(sm + C_OFF_KQ + sk * kKQBytes);
                const uint32_t dsm = smem_u32(sm + C_OFF_D + sk * kItemBytes);   // T1 | T2 | P
                const uint32_t vsm = smem_u32(sm + C_OFF_V + sv * kVBytes);
                mbar_wait(&B.d_full[sk], (c / kDStages) & 1, abort);
                mbar_wait(&B.kq_full[sk], (c / kKQStages) & 1, abort);
                mbar_wait(&B.s_next, c & 1, abort);      // S16 and Q' of this chunk ready
                mbar_wait(&B.v_full[sv], (c / kVStages) & 1, abort);
                tc_fence_after();
                for (int s = 0; s < 4; ++s)   // MU: U = T1 V  (A = V^T, MN-major)
                    mma_ss(tbase + kColU, sdesc_sw128(vsm + s * 16 * 128, kVBlk, 1024),
                           sdesc_sw128(dsm + s * 32, 16, 1024), id64amn, s > 0);
                mma_commit(&B.v_empty[sv]);
                for (int s = 0; s < 8; ++s) {   // M23: [X | O] = S [K; Q']^T
                    const uint32_t off = (s >> 2) * kKBlk + (s & 3) * 32;
                    mma_ts(tbase + kColX, tbase + kColS16 + s * 8, sdesc_sw128(kqb + off, 16, 1024),
                           id128, s > 0);
                }
                mma_commit(&B.x_full);
                mbar_wait(&B.r_full, c & 1, abort);
                tc_fence_after();
                for (int s = 0; s < 4; ++s)   // M4: U += T2 X^T
                    mma_ts(tbase + kColU, tbase + kColX + s * 8,
                           sdesc_sw128(dsm + kMatBytes + s * 32, 16, 1024), id64, 1);
                mma_commit(&B.u_full);
                mbar_wait(&B.u2_full, c & 1, abort);
                tc_fence_after();
                for (int s = 0; s < 4; ++s) {
                    // M5: O += U P^T ; M6: S += U K''  (K'' MN-major: 2 blocks of 64 keys)
                    mma_ts(tbase + kColO, tbase + kColU + s * 8,
                           sdesc_sw128(dsm + 2 * kMatBytes + s * 32, 16, 1024), id64, 1);
                    mma_ts(tbase + kColS32, tbase + kColU + s * 8,
                           sdesc_sw128(kqb + s * 16 * 128, kKBlk, 1024), id128bmn, 1);
                }
                mma_commit(&B.s_full);
                mma_commit(&B.kq_empty[sk]);
                mma_commit(&B.d_empty[sk]);
            }
            mma_commit(&B.mma_done);
            int z = 0;
            mbar_wait(&B.mma_done, 0, &z);
        }
        __syncwarp();
    } else {
        // --------------------------------------------------- chain (4 warps)
        const int tc4 = tid - 64;                 // 0 .. 127
        const int q4 = warp & 3;
        const int b = q4 * 32 + lane;            // value row of the state
        const uint32_t lrow = tmem_addr(tbase, q4 * 32, 0);
        auto item_scal = [&](int c) -> const ItemScal & {
            return *reinterpret_cast<const ItemScal *>(sm + C_OFF_D + (c % kDStages) * kItemBytes +
                                                       kItemScal);
        };
        // Q' = scale Gam_i r_q,i Q_i in place for chunk cq, before M23 of that chunk
        auto rescale_q = [&](int cq) {
            mbar_wait(&B.d_full[cq % kDStages], (cq / kDStages) & 1, abort);
            mbar_wait(&B.kq_full[cq % kKQStages], (cq / kKQStages) & 1, abort);
            uint8_t *kqq = sm + C_OFF_KQ + (cq % kKQStages) * kKQBytes;
            const int i = tc4 >> 1, kb = tc4 & 1;
            const float f = item_scal(cq).sq[i];
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                uint4 *pq = reinterpret_cast<uint4 *>(kqq + kb * kKBlk + sw128_chunk(C + i, ch));
                *pq = scale_chunk(*pq, f);
            }
            fence_async_smem();
        };
        // E0: initial state -> bf16 operand copy, and the fp32 accumulator
        //     pre-scaled by the first chunk's total decay
        {
            mbar_wait(&B.d_full[0], 0, abort);
            const float gn = item_scal(0).gam_n;
            const float *src = islot >= 0 ? pool + islot * slot_stride + head_off + (size_t)b * DH : nullptr;
            for (int c0 = 0; c0 < DH; c0 += 32) {
                uint32_t v[32], pk[16];
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const float4 f = src ? *reinterpret_cast<const float4 *>(src + c0 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
                    v[j] = __float_as_uint(f.x); v[j + 1] = __float_as_uint(f.y);
                    v[j + 2] = __float_as_uint(f.z); v[j + 3] = __float_as_uint(f.w);
                }
#pragma unroll
                for (int jj = 0; jj < 16; ++jj)
                    pk[jj] = pack_bf16(__uint_as_float(v[2 * jj]), __uint_as_float(v[2 * jj + 1]));
                tmem_st16(lrow + kColS16 + c0 / 2, pk);
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * gn);
                tmem_st32(lrow + kColS32 + c0, v);
            }
            tmem_wait_st();
            rescale_q(0);
            tc_fence_before();
            mbar_arrive(&B.s_next);
        }
        for (int c = 0; c < nch; ++c) {
            const int sd = c % kDStages;
            const ItemScal &I = item_scal(c);     // d_full(c) was waited by rescale_q(c)
            uint8_t *kq = sm + C_OFF_KQ + (c % kKQStages) * kKQBytes;
            const int64_t c0 = s_start + (int64_t)c * C;
            const bool last = c == nch - 1;
            const int n = I.n;
            // ---- E1: X -> bf16 in TMEM (X's columns)
            mbar_wait(&B.x_full, c & 1, abort);
            tc_fence_after();
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                uint32_t x[32], xx[16];
                tmem_ld32(lrow + kColX + 32 * h2, x);
#pragma unroll
                for (int jj = 0; jj < 16; ++jj)
                    xx[jj] = pack_bf16(__uint_as_float(x[2 * jj]), __uint_as_float(x[2 * jj + 1]));
                tmem_st16(lrow + kColX + 16 * h2, xx);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&B.r_full);
            // K'' = D[last][j] r_k,j K_j in place (M23 has consumed the raw rows)
            {
                const int j = tc4 >> 1, kb = tc4 & 1;
                const float f = I.ks[j];
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    uint4 *pk = reinterpret_cast<uint4 *>(kq + kb * kKBlk + sw128_chunk((uint32_t)j, ch));
                    *pk = scale_chunk(*pk, f);
                }
                fence_async_smem();
            }
            // ---- E2: U -> bf16 in TMEM (U's columns)
            mbar_wait(&B.u_full, c & 1, abort);
            tc_fence_after();
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                uint32_t u[32], uu[16];
                tmem_ld32(lrow + kColU + 32 * h2, u);
#pragma unroll
                for (int jj = 0; jj < 16; ++jj)
                    uu[jj] = pack_bf16(__uint_as_float(u[2 * jj]), __uint_as_float(u[2 * jj + 1]));
                tmem_st16(lrow + kColU + 16 * h2, uu);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&B.u2_full);
            if (!last) rescale_q(c + 1);   // overlaps M5 / M6
            // ---- E3a: S -> bf16 operand copy, fp32 pre-scaled for the next
            //      chunk (or the final state -> pool)
            mbar_wait(&B.s_full, c & 1, abort);
            tc_fence_after();
            const float gnext = last ? 1.f : item_scal(c + 1).gam_n;
            float *dstp = (last && fslot >= 0) ? pool + fslot * slot_stride + head_off + (size_t)b * DH : nullptr;
            for (int cc = 0; cc < DH; cc += 32) {
                uint32_t sv[32];
                tmem_ld32(lrow + kColS32 + cc, sv);
                if (!last) {
                    uint32_t pk[16];
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj)
                        pk[jj] = pack_bf16(__uint_as_float(sv[2 * jj]), __uint_as_float(sv[2 * jj + 1]));
                    tmem_st16(lrow + kColS16 + cc / 2, pk);
#pragma unroll
                    for (int j = 0; j < 32; ++j) sv[j] = __float_as_uint(__uint_as_float(sv[j]) * gnext);
                    tmem_st32(lrow + kColS32 + cc, sv);
                } else if (dstp) {
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4 *>(dstp + cc + j) = make_float4(
                            __uint_as_float(sv[j]), __uint_as_float(sv[j + 1]),
                            __uint_as_float(sv[j + 2]), __uint_as_float(sv[j + 3]));
                }
            }
            uint32_t ov0[32], ov1[32];
            tmem_ld32(lrow + kColO, ov0);
            tmem_ld32(lrow + kColO + 32, ov1);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&B.s_next);      // S16 ready and X | O free for the next chunk
            // ---- E3b: o <- O (from registers)
            {
                __nv_bfloat16 *orow = o + (c0 * hv + h) * (int64_t)DH + b;
                const int64_t ostride = (int64_t)hv * DH;
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (i < n) orow[i * ostride] = __float2bfloat16_rn(__uint_as_float(ov0[i]));
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (32 + i < n) orow[(32 + i) * ostride] = __float2bfloat16_rn(__uint_as_float(ov1[i]));
            }
            mbar_arrive(&B.d_empty[sd]);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
    }
    if (tid == 0 && B.abort) flag_status(GDN_DEVSTAT_TIMEOUT);
}

}  // namespace psp

size_t prefill_split_workspace(int n_seqs, int64_t n_tokens, int hv) {
    return psp::header_bytes(n_seqs) +
           (size_t)psp::chunk_bound(n_tokens, n_seqs) * (size_t)hv * psp::kItemBytes;
}

gdn_status prefill_split(const void *q, int64_t qs, const void *k, int64_t ks, const void *v,
                         int64_t vs, const float *g, const float *beta, const int32_t *cu,
                         int n_seqs, int64_t n_tokens, int hqk, int hv, float scale, int l2norm,
                         float *pool, int64_t n_slots, const int32_t *ii, const int32_t *fi,
                         void *o, void *ws, cudaStream_t s) {
    const int64_t items = psp::chunk_bound(n_tokens, n_seqs) * hv;
    if (items >= (1ll << 31)) return GDN_ERR_UNSUPPORTED;
    CUtensorMap tq, tk, tv;
    const uint64_t rows = (uint64_t)n_tokens;
    if (!encode_tmap_2d_bf16(&tq, q, (uint64_t)hqk * 128, rows, qs, 64, 64) ||
        !encode_tmap_2d_bf16(&tk, k, (uint64_t)hqk * 128, rows, ks, 64, 64) ||
        !encode_tmap_2d_bf16(&tv, v, (uint64_t)hv * 128, rows, vs, 64, 64))
        return GDN_ERR_LAUNCH;
    cudaError_t e = cudaFuncSetAttribute(psp::prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)psp::P_SMEM_BYTES);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(psp::chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)psp::C_SMEM_BYTES);
    if (e != cudaSuccess) {
        set_last_cuda_error(e);
        return GDN_ERR_LAUNCH;
    }
    int32_t *base = reinterpret_cast<int32_t *>(ws);
    uint8_t *item_blocks = reinterpret_cast<uint8_t *>(ws) + psp::header_bytes(n_seqs);
    psp::chunk_base_kernel<<<1, 1024, 0, s>>>(cu, n_seqs, n_tokens, base);
    gdn_status st = launch_status();
    if (st != GDN_OK) return st;
    psp::prep_kernel<<<(unsigned)items, psp::kPrepKernelThreads, psp::P_SMEM_BYTES, s>>>(
        tq, tk, g, beta, cu, base, n_seqs, hv, hv / hqk, scale, l2norm, item_blocks);
    st = launch_status();
    if (st != GDN_OK) return st;
    psp::chain_kernel<<<(unsigned)((int64_t)n_seqs * hv), psp::kChainKernelThreads,
                        psp::C_SMEM_BYTES, s>>>(tq, tk, tv, cu, base, n_seqs, n_tokens, hv,
                                                hv / hqk, item_blocks, pool, n_slots, ii, fi,
                                                (__nv_bfloat16 *)o);
    return launch_status();
}

}  // namespace gdn
