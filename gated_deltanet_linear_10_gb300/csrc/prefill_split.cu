// Chunked prefill in two kernels, for callers that pass a workspace
// ("Flash Linear Attention operations for efficient chunked computations",
// "[model] Support Qwen3next", Highlights).  Same recurrence as the fused
// tensor-core kernel (prefill_tc.cu), split where the dependency structure
// allows it:
//
//   1. prep_kernel: everything that does not depend on the state, for every
//      (chunk, V head) item at once -- chunk-parallel, several CTAs per SM:
//      G = [K;Q] K^T on the tensor cores, gates, norms, A and P, the UT solve
//      T = (I + A)^-1, T1 = T diag(beta), and on the tensor cores again
//      W = T diag(beta Gam r_k) K (the WY form's key term, kept negated).
//      Each item's T1 | P | W^T | row factors block is written to the
//      workspace in exactly the shared-memory layout the MMAs read.
//   2. chain_kernel: per (sequence, V head) only the state chain,
//        M2  U  = S W'^T                W' = -W
//        MU  U += T1 V                  so U = T1 V - W S^T
//        O   O  = S Q'^T                Q' = scale Gam r_q Q
//        E2  U -> bf16;  M6  S += U K'';  M5  O += U P^T
//        E3  S -> bf16 copy for the next chunk, S pre-scaled by its decay
//      with the item blocks streamed in by 1-D bulk copies next to the K|Q
//      and V tiles.  Against the fused kernel this drops the X = S K^T
//      round trip (and its epilogue) from the chain's critical path.
//
// Workspace: [chunk offsets, int32 x (n_seqs + 1), padded to 1 KiB]
//            [items: (ceil(n_tokens / 64) + n_seqs) x hv blocks of kItemBytes]
#include <stddef.h>

#include <algorithm>

#include "prefill_common.cuh"
#include "prefill_scan.cuh"

namespace gdn {

GDN_DECLARE_STATUS_WORD(g_status_prefill_split)
GDN_STATUS_READER(read_status_prefill_split, g_status_prefill_split)

// Debug control (gdn_debug_set_wait_limit): when set, the prep kernel issues
// no K|Q tile load, so its waits for that tile run out after the wait limit.
__device__ int g_prep_drop_loads = 0;

namespace psp {
using namespace ptc;

// item block: T1 [i][j] | P [i][j] (64 x 64 bf16, K-major) | W'^T [a][i]
// (128 x 64 bf16, 128 rows of 128 B) | row factors.  All 128-byte swizzled.
constexpr uint32_t kItemT1 = 0, kItemP = kMatBytes, kItemW = 2 * kMatBytes;
constexpr uint32_t kItemWBytes = 128 * 128;
constexpr uint32_t kItemOps = kItemW + kItemWBytes;            // 32 KiB of operands
struct ItemScal {
    float ks[C];      // D[last][j] r_k,j      (K'' row factors)
    float sq[C];      // scale Gam_i r_q,i     (Q' row factors)
    float gam_n;      // total decay of the chunk
    int n;            // valid rows
};
constexpr uint32_t kItemScalCopy = (sizeof(ItemScal) + 15) / 16 * 16;
constexpr uint32_t kItemBytes = (kItemOps + kItemScalCopy + 1023) / 1024 * 1024;

__host__ __device__ inline size_t header_bytes(int n_seqs) {
    return ((size_t)4 * (n_seqs + 1) + 1023) / 1024 * 1024;
}
__host__ __device__ inline int64_t chunk_bound(int64_t n_tokens, int n_seqs) {
    return (n_tokens + C - 1) / C + n_seqs;
}

// A sequence whose bounds are invalid gets no chunks (the chain kernel
// reports it).
__device__ __forceinline__ int seq_chunks(const int32_t *cu, int s, int64_t n_tokens) {
    const int32_t a = cu[s], e = cu[s + 1];
    return (a < 0 || e < a || e > n_tokens) ? 0 : (e - a + C - 1) / C;
}

// chunk_base[s] = sum over sequences before s of ceil(len / 64); one CTA.
__global__ void __launch_bounds__(1024) chunk_base_kernel(const int32_t *__restrict__ cu,
                                                          int n_seqs, int64_t n_tokens,
                                                          int32_t *__restrict__ base) {
    griddep_launch();        // the prep kernel behind it may start placing its CTAs
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
// The gate inputs of the prep kernel: g and beta, or (with a) the raw
// a, b [n_tokens][hv] bf16 and A_log, dt_bias [hv], from which the kernel
// forms g = -exp(A_log) softplus(a + dt_bias) and beta = sigmoid(b) itself
// (the same expressions as the gating kernel, so the same values).
struct RawGates {
    const __nv_bfloat16 *a, *b;
    const float *A_log, *dt_bias;
};
__device__ __forceinline__ void gate_of(const float *g, const float *beta, const RawGates &rg,
                                        int64_t row, int hv, int h, float &gv, float &bv) {
    const int64_t i = row * hv + h;
    if (rg.a) {
        const float x = __bfloat162float(rg.a[i]) + rg.dt_bias[h];
        gv = -expf(rg.A_log[h]) * (x > 20.0f ? x : log1pf(expf(x)));
        bv = 1.0f / (1.0f + expf(-__bfloat162float(rg.b[i])));
    } else {
        gv = g[i];
        bv = beta[i];
    }
}

constexpr int kPrepWarps = 9;              // warp 0: TMA + MMA + TMEM; warps 1..8: prep
constexpr int kPrepKernelThreads = kPrepWarps * 32;
constexpr int kPrepThreads = 256;
constexpr int kPrepCtasPerSm = 3;

struct PrepScal {
    float beta[C], gam[C], alpha[C], rk[C], rq[C], xs[C];
};
struct PrepBars {
    uint64_t kq_full, g_full, w_go, w_full;
    uint32_t tmem_base;
    int abort;
};
// Shared memory.  The raw K|Q tile keeps its K rows for the W MMA; its Q
// halves become the P and T1 staging once G is in TMEM.  T2 is written over
// the dead rows of Af (the last solve level reads only rows 48..63), and
// after the W MMA Af stages W'^T and Wb the row factors.
constexpr uint32_t P_OFF_KQ = 0;
constexpr uint32_t P_OFF_P = P_OFF_KQ + 64 * 128;              // Q rows of k-block 0
constexpr uint32_t P_OFF_T1 = P_OFF_KQ + kKBlk + 64 * 128;     // Q rows of k-block 1
constexpr uint32_t P_OFF_AF = P_OFF_KQ + kKQBytes;
constexpr uint32_t P_OFF_TF = P_OFF_AF + C * kLd * 4;
constexpr uint32_t P_OFF_WB = P_OFF_TF + C * kLd * 4;
constexpr uint32_t kPWbBytes = (8 * 16 * kWbLd + 16 * 16) * 4;
constexpr uint32_t P_OFF_SCAL = P_OFF_WB + kPWbBytes;
constexpr uint32_t P_OFF_BARS = P_OFF_SCAL + (sizeof(PrepScal) + 127) / 128 * 128;
constexpr uint32_t P_SMEM_BYTES = P_OFF_BARS + 128 + 1024;   // + slack to align to 1024
constexpr uint32_t kPrepTmemCols = 128;                      // G = [K;Q][K;Q]^T, then W'^T
static_assert(kItemWBytes <= C * kLd * 4 && sizeof(ItemScal) <= kPWbBytes, "staging");
static_assert(P_OFF_T1 + kMatBytes == P_OFF_AF && kMatBytes <= 48 * kLd * 4,
              "T2 lands on Af rows below 48");
static_assert(sizeof(PrepBars) <= 128, "barrier block");
static_assert(kPrepCtasPerSm * (P_SMEM_BYTES + 1024) <= 233472, "three prep CTAs per SM");

// A persistent grid (3 CTAs per SM) over the (chunk, V head) items.  Per
// item, warp 0: TMA of the raw K|Q tile,
// M1 G = [K;Q] [K;Q]^T (its diagonal gives the row norms), then
// MW W'^T = K^T T2^T; warps 1..8: the prep arithmetic, then bulk stores of
// the item block.
__global__ void __launch_bounds__(kPrepKernelThreads, kPrepCtasPerSm)
prep_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const float *__restrict__ g, const float *__restrict__ beta, RawGates rg,
            const int32_t *__restrict__ cu, const int32_t *__restrict__ base, int n_seqs, int hv,
            int grp, float scale, int l2norm, uint8_t *__restrict__ items) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    PrepBars &B = *reinterpret_cast<PrepBars *>(sm + P_OFF_BARS);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Launched behind the chunk-offset kernel: once every CTA of this grid
    // has started, the chain kernel may place its CTAs on the SMs that the
    // last items leave idle.  The chunk offsets are read after the wait.
    griddep_launch();
    griddep_wait();
    const int n_work = base[n_seqs] * hv;     // (chunk, V head) items
    if ((int)blockIdx.x >= n_work) return;
    uint8_t *kq = sm + P_OFF_KQ;

    if (warp == 0) {
        tmem_alloc(&B.tmem_base, kPrepTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&B.kq_full, 1);
        mbar_init(&B.g_full, 1);
        mbar_init(&B.w_go, kPrepThreads);
        mbar_init(&B.w_full, 1);
        B.abort = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = B.tmem_base;
    volatile int *abort = &B.abort;
    // persistent: CTA b takes the items n_work - 1 - b, n_work - 1 - b - grid,
    // ... (in reverse, so that the first chunks, which the chains read first,
    // are written last and can still be in L2 when the chains start: 0.3788
    // -> 0.3772 ms on the 8-sequence batch); the barriers' phase flips per
    // item, TMEM and the barriers are set up once
    for (int wk0 = blockIdx.x, kk = 0; wk0 < n_work; wk0 += gridDim.x, ++kk) {
        const uint32_t ph = kk & 1;
        const int wk = n_work - 1 - wk0;
        const int it = wk / hv;
        const int h = wk - it * hv;
        int lo = 0, hi = n_seqs - 1;          // the sequence: last s with base[s] <= it
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (base[mid] <= it) lo = mid; else hi = mid - 1;
        }
        const int64_t c0 = cu[lo] + (int64_t)(it - base[lo]) * C;
        const int n = (int)min((int64_t)C, (int64_t)cu[lo + 1] - c0);
        const int hq = h / grp;

        if (warp == 0) {
            if (lane == 0) {
                const bool drop = *(volatile int *)&g_prep_drop_loads != 0;
                if (!drop) {
                    mbar_arrive_expect_tx(&B.kq_full, kKQBytes);
                    for (int kb = 0; kb < 2; ++kb) {
                        tma_load_2d(kq + kb * kKBlk, &tm_k, &B.kq_full, hq * DH + kb * 64, (int)c0);
                        tma_load_2d(kq + kb * kKBlk + 64 * 128, &tm_q, &B.kq_full,
                                    hq * DH + kb * 64, (int)c0);
                    }
                }
                uint64_t *last = nullptr;   // the item's last commit: TMEM is reused after it
                if (mbar_wait(&B.kq_full, ph, abort)) {
                    tc_fence_after();
                    const uint32_t id128 = idesc_bf16(128, 128);
                    const uint32_t kb0 = smem_u32(kq);
                    for (int s = 0; s < 8; ++s) {
                        const uint32_t off = (s >> 2) * kKBlk + (s & 3) * 32;
                        mma_ss(tbase, sdesc_sw128(kb0 + off, 16, 1024),
                               sdesc_sw128(kb0 + off, 16, 1024),
                               id128, s > 0);
                    }
                    mma_commit(&B.g_full);
                    last = &B.g_full;
                    if (mbar_wait(&B.w_go, ph, abort)) {
                        // MW: W'^T[a][i] = sum_j K[j][a] T2[i][j]  (A = K^T, MN-major)
                        tc_fence_after();
                        const uint32_t id64amn = idesc_bf16(128, 64, true, false);
                        const uint32_t t2 = smem_u32(sm + P_OFF_AF);
                        for (int s = 0; s < 4; ++s)
                            mma_ss(tbase, sdesc_sw128(kb0 + s * 16 * 128, kKBlk, 1024),
                                   sdesc_sw128(t2 + s * 32, 16, 1024), id64amn, s > 0);
                        mma_commit(&B.w_full);
                        last = &B.w_full;
                    }
                } else if (!drop) {
                    int z = 0;       // never leave with the copy in flight
                    mbar_wait(&B.kq_full, ph, &z);
                }
                if (last) { int z = 0; mbar_wait(last, ph, &z); }
            }
            __syncwarp();
        } else {
            const int t = tid - 32;                 // 0 .. 255
            const int pw = warp - 1;                // 0 .. 7
            const int q4 = warp & 3;                // TMEM lane quadrant
            const int p = q4 * 32 + lane;           // G row: 0..63 K rows, 64..127 Q rows
            const int chalf = pw >> 2;              // which 32 TMEM columns this warp reads
            PrepScal &S = *reinterpret_cast<PrepScal *>(sm + P_OFF_SCAL);
            float *Af = reinterpret_cast<float *>(sm + P_OFF_AF);
            float *Tf = reinterpret_cast<float *>(sm + P_OFF_TF);
            float *Wb = reinterpret_cast<float *>(sm + P_OFF_WB);
            float g0 = 0.f, g1 = 0.f, b0 = 0.f, b1 = 0.f;
            if (t < 32) {
                if (2 * t < n) gate_of(g, beta, rg, c0 + 2 * t, hv, h, g0, b0);
                if (2 * t + 1 < n) gate_of(g, beta, rg, c0 + 2 * t + 1, hv, h, g1, b1);
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
            mbar_wait(&B.g_full, ph, abort);
            tc_fence_after();
            uint32_t gr[32];
            tmem_ld32(tmem_addr(tbase, q4 * 32, 32 * chalf), gr);
            {   // inverse L2 norms from the diagonal of G: row p's own column, p for
                // a K row, 64 + (p - 64) for a Q row (q . q); p % 32 is the lane
                // (both conditions are warp-uniform)
                float dg = 0.f;
                bool own = p < C && (p >> 5) == chalf;
                if (own) {
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) dg = jj == lane ? __uint_as_float(gr[jj]) : dg;
                }
                if (p >= C && ((p - C) >> 5) == chalf) {
                    uint32_t gq[32];
                    tmem_ld32(tmem_addr(tbase, q4 * 32, C + 32 * chalf), gq);
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) dg = jj == lane ? __uint_as_float(gq[jj]) : dg;
                    own = true;
                }
                if (own) {
                    const float r = l2norm ? rsqrtf(dg + kEps) : 1.f;
                    if (p < C) S.rk[p] = r; else S.rq[p - C] = r;
                }
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
            // the Q rows are dead: P goes to k-block 0's
            g_to_a_p(gr, p, chalf, n, S.beta, S.gam, S.alpha, S.rk, S.rq, scale, Af, sm + P_OFF_P);
            named_sync(1, kPrepThreads);
            // T1 over k-block 1's Q rows, T2 over Af's dead rows
            ut_solve_mma<true>(Af, Tf, Wb, t, pw, lane, S.beta, S.xs, sm + P_OFF_T1);
            fence_async_smem();
            tc_fence_before();
            mbar_arrive(&B.w_go);                  // T2 is in place: MW may run
            // the solve scratch is dead: the row factors go to Wb, W'^T to Af
            ItemScal &I = *reinterpret_cast<ItemScal *>(Wb);
            if (t < C) {
                I.ks[t] = ksv;
                I.sq[t] = sqv;
                if (t == 0) {
                    I.gam_n = __expf(gl);
                    I.n = n;
                }
            }
            mbar_wait(&B.w_full, ph, abort);
            tc_fence_after();
            {
                uint32_t wr[32];
                tmem_ld32(tmem_addr(tbase, q4 * 32, 32 * chalf), wr);
                uint8_t *wt = sm + P_OFF_AF;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w[e] = pack_bf16(__uint_as_float(wr[8 * cc + 2 * e]),
                                         __uint_as_float(wr[8 * cc + 2 * e + 1]));
                    *reinterpret_cast<uint4 *>(wt + sw128_chunk((uint32_t)p, 4 * chalf + cc)) =
                        make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            fence_async_smem();
            named_sync(1, kPrepThreads);
            if (t == 0 && !*abort) {
                uint8_t *item = items + ((size_t)it * hv + h) * kItemBytes;
                bulk_store(item + kItemT1, sm + P_OFF_T1, kMatBytes);
                bulk_store(item + kItemP, sm + P_OFF_P, kMatBytes);
                bulk_store(item + kItemW, sm + P_OFF_AF, kItemWBytes);
                bulk_store(item + kItemOps, Wb, kItemScalCopy);
                bulk_commit();
                bulk_wait_read_all();   // the staging may go; the writes complete on their own
            }
        }
        tc_fence_before();
        __syncthreads();                    // shared memory and TMEM are reused by the next item
        tc_fence_after();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tbase, kPrepTmemCols);
    }
    if (tid == 0 && B.abort) flag_status(GDN_DEVSTAT_TIMEOUT);
}

inline unsigned prep_grid(int64_t items) {   // the item bound caps it for tiny batches
    return (unsigned)std::min<int64_t>(items, (int64_t)kPrepCtasPerSm * sm_count());
}

// ------------------------------------------------------------ chain kernel --
// One CTA per (sequence, V head).  Per chunk c (S pre-scaled by the chunk's
// decay, S16 its bf16 copy; K, Q, V raw tiles; T1, P, W' from the item):
//   M2  U1  = S16[:, a < 64] W'^T,  U2 = S16[:, a >= 64] W'^T    (W' = T2 K)
//   MU  U2 += T1 V                    (behind U2's half of M2, same issuer)
//   E2  U = U1 + U2;  U16 = bf16(U), U16k = bf16(U diag(ks))     (ks: K'' rows)
//   M6  S += U16k K                   (= U K'')
//   O   O1 = S16 Q^T,  O2 = U16 P^T,  o = diag(sq) O1 + O2       (sq: Q' rows)
//   E3  S16 = bf16(S) for the next chunk, S *= its decay, o stores
// A tcgen05.mma costs its issuing thread about 60 cycles whatever N is, and
// an N = 64 product occupies the tensor pipe for about half that, so M2 is
// split by K over two issuing threads (warps 1 and 10) into separate
// accumulators that E2 adds.  The critical path is
//   s_next -> M2 -> E2 -> M6 -> E3a -> s_next;
// O1, O2 and the o stores fill the gaps.  (MU used to run a chunk ahead into
// U1, with M2 accumulating onto it: the next M2 then waited for MU, whose
// operands arrive late; behind M2 it adds ~2 % less time.)  Warp 0: TMA / bulk
// producer; warps 2..9: the epilogues as two warpgroups that each take half
// of the TMEM columns of S, U and O, and store o a 32 x 32 tile per warp
// through shared memory with TMA.
constexpr int kChainWarps = 11;
constexpr int kChainKernelThreads = kChainWarps * 32;
constexpr int kEpiThreads = 256;
constexpr int kKQStages = 3, kVStages = 2, kDStages = 2, kCStages = 4;
constexpr uint32_t kColS32 = 0, kColS16 = 128, kColU1 = 192, kColU2 = 256, kColO1 = 320,
                   kColO2 = 384, kColU16 = 448, kColU16k = 480, kTmemCols = 512;
constexpr uint32_t kCStageBytes = 1024;

struct ChainBars {
    uint64_t kq_full[kKQStages], kq_empty[kKQStages], v_full[kVStages], v_empty[kVStages],
        d_full[kDStages], d_empty[kDStages], c_full[kCStages], c_empty[kCStages];
    uint64_t u_full, u2_full, s_full, o1_full, o2_full, s_next, o_free, done_a, done_b;
    uint64_t zbar[8];             // per epilogue warp: its z tile of the chunk (gated output)
    uint32_t tmem_base;
    int abort;
    int seq;
};
constexpr uint32_t kOTileBytes = 32 * 32 * 2;               // one warp's o tile [i][b]
// gated output: [half][chunk parity][warp][token] sums of squares, then
// [warp][token] inverse norms
constexpr uint32_t kRedBytes = 2 * 2 * 4 * 32 * 4 + 8 * 32 * 4;
// Shared memory of the chain kernel.  The gated variant stages each warp's z
// tile in a buffer of its own (so the next chunk's z load waits for no o
// store) and pays for it with a K|Q ring of two stages instead of three.
template <bool kGated>
struct ChainSmem {
    static constexpr int kKQ = kGated ? 2 : kKQStages;     // K|Q ring depth
    static constexpr uint32_t KQ = 0;
    static constexpr uint32_t V = KQ + kKQ * kKQBytes;
    static constexpr uint32_t D = V + kVStages * kVBytes;
    static constexpr uint32_t Cs = D + kDStages * kItemOps;
    static constexpr uint32_t OT = Cs + kCStages * kCStageBytes;
    static constexpr uint32_t ZT = OT + 8 * kOTileBytes;   // gated: z tiles
    static constexpr uint32_t RED = ZT + (kGated ? 8 * kOTileBytes : 0);
    static constexpr uint32_t BARS = RED + (kGated ? kRedBytes : 0);
    static constexpr uint32_t BYTES = BARS + (sizeof(ChainBars) + 127) / 128 * 128 + 1024;
};
static_assert(kItemOps % 1024 == 0 && kItemScalCopy <= kCStageBytes, "stage layout");
static_assert(ChainSmem<false>::BYTES <= 232448 && ChainSmem<true>::BYTES <= 232448,
              "shared memory budget");

// Chains beyond the n_seqs * hv ordinary ones (the chunk-state scan): chain
// j runs sequence seq0 + j from the identity state with v = 0, so that its
// final state is the sequence's state transition A (S_end = S_0 A + B) and
// its outputs Phi the map from S_0 to o (o = o(S_0 = 0) + S_0 Phi); Phi rows
// are counted from the sequence start.  Its final state goes to pool_out
// slot final0 + j.
struct IdentChains {
    int n;
    int seq0;
    int final0;
};

// The gated output (kGated): y = o / sqrt(mean(o^2) + eps) * w * SiLU(z) per
// (token, V head) row, written instead of o.
struct GateArgs {
    const float *w;    // [128] fp32
    float eps;
};

template <bool kGated>
__global__ void __launch_bounds__(kChainKernelThreads, 1)
chain_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
             const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
             const __grid_constant__ CUtensorMap tm_phi, const __grid_constant__ CUtensorMap tm_z,
             GateArgs gate, const int32_t *__restrict__ cu,
             const int32_t *__restrict__ base, int n_seqs, int64_t n_tokens, int hv, int grp,
             const uint8_t *__restrict__ items, const float *__restrict__ pool_in, int64_t n_in,
             float *__restrict__ pool_out, int64_t n_out, const int32_t *__restrict__ init_idx,
             const int32_t *__restrict__ final_idx, __nv_bfloat16 *__restrict__ o,
             __nv_bfloat16 *__restrict__ phi, IdentChains ic) {
    using L = ChainSmem<kGated>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    ChainBars &B = *reinterpret_cast<ChainBars *>(sm + L::BARS);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // a kernel launched behind this one (a mixed batch's decode) may start on
    // the SMs the chains leave free
    griddep_launch();

    const int rank = blockIdx.x / hv;
    const int h = blockIdx.x - rank * hv;
    const int hq = h / grp;
    const bool ident = rank >= n_seqs;                // CTA-uniform
    const int seq = ident ? ic.seq0 + (rank - n_seqs) : seq_for_rank(cu, n_seqs, rank, &B.seq);
    const int64_t s_start = cu[seq], s_end = cu[seq + 1];
    int64_t islot = ident ? -1 : (init_idx ? init_idx[seq] : -1);
    int64_t fslot = ident ? ic.final0 + (rank - n_seqs) : (final_idx ? final_idx[seq] : -1);
    if (islot >= n_in || fslot >= n_out) {
        if (tid == 0) flag_status(GDN_DEVSTAT_BAD_INDEX);
        if (islot >= n_in) islot = -1;
        if (fslot >= n_out) fslot = -1;
    }
    if (s_start < 0 || s_end < s_start || s_end > n_tokens) {
        if (tid == 0) {
            flag_status(GDN_DEVSTAT_BAD_SEQLEN);
            griddep_wait();   // this grid completes after the prep kernel, on every path
        }
        return;
    }
    const int nch = (int)((s_end - s_start + C - 1) / C);
    const size_t head_off = (size_t)h * DH * DH;
    const size_t slot_stride = (size_t)hv * DH * DH;
    if (nch == 0) {   // empty sequence: the initial state (zero, identity) is the final state
        if (tid == 0) griddep_wait();
        if (fslot >= 0)
            for (int e = tid; e < DH * DH; e += kChainKernelThreads)
                pool_out[fslot * slot_stride + head_off + e] =
                    ident ? ((e >> 7) == (e & 127) ? 1.f : 0.f)
                          : (islot >= 0 ? pool_in[islot * slot_stride + head_off + e] : 0.f);
        return;
    }
    // the output rows: o at absolute rows, Phi from the sequence start
    const CUtensorMap *tm_out = ident ? &tm_phi : &tm_o;
    __nv_bfloat16 *out = ident ? phi : o;
    const int64_t row0 = ident ? s_start : 0;
    const int64_t item0 = base[seq];

    if (warp == 1) {
        tmem_alloc(&B.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < L::kKQ; ++s) { mbar_init(&B.kq_full[s], 1); mbar_init(&B.kq_empty[s], 1); }
        for (int s = 0; s < kVStages; ++s) { mbar_init(&B.v_full[s], 1); mbar_init(&B.v_empty[s], 1); }
        for (int s = 0; s < kDStages; ++s) { mbar_init(&B.d_full[s], 1); mbar_init(&B.d_empty[s], 1); }
        for (int s = 0; s < kCStages; ++s) { mbar_init(&B.c_full[s], 1); mbar_init(&B.c_empty[s], kEpiThreads); }
        mbar_init(&B.u_full, 2);                       // one commit from each issuer
        mbar_init(&B.u2_full, kEpiThreads);
        mbar_init(&B.s_full, 1);
        mbar_init(&B.o1_full, 1);
        mbar_init(&B.o2_full, 1);
        mbar_init(&B.s_next, kEpiThreads);
        mbar_init(&B.o_free, kEpiThreads);
        mbar_init(&B.done_a, 1);
        mbar_init(&B.done_b, 1);
        for (int w = 0; w < 8; ++w) mbar_init(&B.zbar[w], 1);
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
            if (!ident) prefetch_tensormap(&tm_v);
            int kq_n[L::kKQ] = {}, v_n[kVStages] = {0, 0}, d_n[kDStages] = {0, 0},
                c_n[kCStages] = {0, 0, 0, 0};
            for (int c = 0; c < nch && !*abort; ++c) {
                const int y = (int)(s_start + (int64_t)c * C);
                const uint8_t *item = items + ((item0 + c) * hv + h) * kItemBytes;
                const int sk = c % L::kKQ, sv = c % kVStages, sd = c % kDStages, sc = c % kCStages;
                if (c >= L::kKQ) mbar_wait(&B.kq_empty[sk], ((c / L::kKQ) - 1) & 1, abort);
                uint8_t *kq = sm + L::KQ + sk * kKQBytes;
                mbar_arrive_expect_tx(&B.kq_full[sk], kKQBytes);
                for (int kb = 0; kb < 2; ++kb) {
                    tma_load_2d(kq + kb * kKBlk, &tm_k, &B.kq_full[sk], hq * DH + kb * 64, y);
                    tma_load_2d(kq + kb * kKBlk + 64 * 128, &tm_q, &B.kq_full[sk], hq * DH + kb * 64, y);
                }
                kq_n[sk] = c / L::kKQ + 1;
                // launched behind the prep kernel: the item blocks are read
                // only once it has completed (K, Q, V and the initial state
                // come from earlier kernels)
                if (c == 0) griddep_wait();
                if (c >= kCStages) mbar_wait(&B.c_empty[sc], ((c / kCStages) - 1) & 1, abort);
                mbar_arrive_expect_tx(&B.c_full[sc], kItemScalCopy);
                bulk_load(sm + L::Cs + sc * kCStageBytes, item + kItemOps, kItemScalCopy, &B.c_full[sc]);
                c_n[sc] = c / kCStages + 1;
                if (c >= kDStages) mbar_wait(&B.d_empty[sd], ((c / kDStages) - 1) & 1, abort);
                mbar_arrive_expect_tx(&B.d_full[sd], kItemOps);
                bulk_load(sm + L::D + sd * kItemOps, item, kItemOps, &B.d_full[sd]);
                d_n[sd] = c / kDStages + 1;
                if (!ident) {   // v = 0 in an identity chain: no V tiles, no MU
                    if (c >= kVStages) mbar_wait(&B.v_empty[sv], ((c / kVStages) - 1) & 1, abort);
                    uint8_t *vt = sm + L::V + sv * kVBytes;
                    mbar_arrive_expect_tx(&B.v_full[sv], kVBytes);
                    for (int kb = 0; kb < 2; ++kb)
                        tma_load_2d(vt + kb * kVBlk, &tm_v, &B.v_full[sv], h * DH + kb * 64, y);
                    v_n[sv] = c / kVStages + 1;
                }
            }
            // never leave with copies in flight: wait for the last load of every stage
            for (int s = 0; s < L::kKQ; ++s)
                if (kq_n[s]) { int z = 0; mbar_wait(&B.kq_full[s], (kq_n[s] - 1) & 1, &z); }
            for (int s = 0; s < kCStages; ++s)
                if (c_n[s]) { int z = 0; mbar_wait(&B.c_full[s], (c_n[s] - 1) & 1, &z); }
            for (int s = 0; s < kDStages; ++s)
                if (d_n[s]) { int z = 0; mbar_wait(&B.d_full[s], (d_n[s] - 1) & 1, &z); }
            for (int s = 0; s < kVStages; ++s)
                if (v_n[s]) { int z = 0; mbar_wait(&B.v_full[s], (v_n[s] - 1) & 1, &z); }
        }
        __syncwarp();
    } else if (warp == 1 || warp == 10) {
        // ------------------------------------------------ the two MMA issuers
        // Issuer A (warp 1): M2 over a < 64 into U1, M6, O2.
        // Issuer B (warp 10): M2 over a >= 64 into U2, MU onto U2 right behind
        // it (one issuer, so the order on the accumulator is fixed), O1.
        if (lane == 0) {
            const bool isA = warp == 1;
            const uint32_t id64 = idesc_bf16(128, 64);
            const uint32_t id64amn = idesc_bf16(128, 64, true, false);
            const uint32_t id64bmn = idesc_bf16(128, 64, false, true);
            const uint32_t id128bmn = idesc_bf16(128, 128, false, true);
            const int s0 = isA ? 0 : 4;                  // this issuer's k-steps over a
            const uint32_t ucol = isA ? kColU1 : kColU2;
            auto issue_mu = [&](int c) {   // MU: U2 += T1 V  (A = V^T, MN-major)
                const int sd = c % kDStages, sv = c % kVStages;
                mbar_wait(&B.d_full[sd], (c / kDStages) & 1, abort);
                mbar_wait(&B.v_full[sv], (c / kVStages) & 1, abort);
                tc_fence_after();
                const uint32_t dsm = smem_u32(sm + L::D + sd * kItemOps);
                const uint32_t vsm = smem_u32(sm + L::V + sv * kVBytes);
                for (int s = 0; s < 4; ++s)   // onto this chunk's U2 (M2 over a >= 64)
                    mma_ss(tbase + kColU2, sdesc_sw128(vsm + s * 16 * 128, kVBlk, 1024),
                           sdesc_sw128(dsm + kItemT1 + s * 32, 16, 1024), id64amn, 1);
                mma_commit(&B.v_empty[sv]);
            };
            for (int c = 0; c < nch; ++c) {
                const int sk = c % L::kKQ, sd = c % kDStages;
                const uint32_t kqb = smem_u32(sm + L::KQ + sk * kKQBytes);
                const uint32_t dsm = smem_u32(sm + L::D + sd * kItemOps);
                mbar_wait(&B.kq_full[sk], (c / L::kKQ) & 1, abort);
                mbar_wait(&B.d_full[sd], (c / kDStages) & 1, abort);
                mbar_wait(&B.s_next, c & 1, abort);      // S16 of this chunk
                tc_fence_after();
                for (int s = s0; s < s0 + 4; ++s)   // M2: U(1|2) (+)= S16 W'^T over this a half
                    mma_ts(tbase + ucol, tbase + kColS16 + s * 8,
                           sdesc_sw128(dsm + kItemW + s * 16 * 128, 8192, 1024), id64bmn,
                           s > s0);
                if (!isA && !ident) issue_mu(c);         // U2 += T1 V, behind its M2 half
                mma_commit(&B.u_full);
                if (isA) {
                    mbar_wait(&B.u2_full, c & 1, abort);     // U16, U16k in TMEM
                    tc_fence_after();
                    for (int s = 0; s < 4; ++s)   // M6: S += U16k K  (K MN-major: 2 blocks of 64 keys)
                        mma_ts(tbase + kColS32, tbase + kColU16k + s * 8,
                               sdesc_sw128(kqb + s * 16 * 128, kKBlk, 1024), id128bmn, 1);
                    mma_commit(&B.s_full);
                    mbar_wait(&B.o_free, c & 1, abort);      // the last chunk's O read out
                    tc_fence_after();
                    for (int s = 0; s < 4; ++s)   // O2 = U16 P^T
                        mma_ts(tbase + kColO2, tbase + kColU16 + s * 8,
                               sdesc_sw128(dsm + kItemP + s * 32, 16, 1024), id64, s > 0);
                    mma_commit(&B.o2_full);
                    mbar_wait(&B.o1_full, c & 1, abort);     // B's reads of these stages are done
                    mma_commit(&B.kq_empty[sk]);
                    mma_commit(&B.d_empty[sd]);
                } else {
                    mbar_wait(&B.u_full, c & 1, abort);      // M2 done: E2 runs, the pipe is free
                    mbar_wait(&B.o_free, c & 1, abort);      // the last chunk's O read out
                    tc_fence_after();
                    for (int s = 0; s < 8; ++s) {   // O1 = S16 Q^T  (S16 still holds this chunk's S)
                        const uint32_t off = (s >> 2) * kKBlk + 64 * 128 + (s & 3) * 32;
                        mma_ts(tbase + kColO1, tbase + kColS16 + s * 8, sdesc_sw128(kqb + off, 16, 1024),
                               id64, s > 0);
                    }
                    mma_commit(&B.o1_full);
                }
            }
            mma_commit(isA ? &B.done_a : &B.done_b);
            int z = 0;
            mbar_wait(isA ? &B.done_a : &B.done_b, 0, &z);
        }
        __syncwarp();
    } else {
        // ------------------------------------------- epilogues (2 warpgroups)
        const int et = tid - 64;                  // 0 .. 255
        const int hf = et >> 7;                   // column half of S, U and O
        const int q4 = warp & 3;
        const int b = q4 * 32 + lane;            // value row of the state
        const uint32_t lrow = tmem_addr(tbase, q4 * 32, 0);
        const uint32_t s32 = lrow + kColS32 + hf * 64, s16 = lrow + kColS16 + hf * 32;
        auto scal = [&](int c) -> const ItemScal & {
            return *reinterpret_cast<const ItemScal *>(sm + L::Cs + (c % kCStages) * kCStageBytes);
        };
        __nv_bfloat16 *ot = reinterpret_cast<__nv_bfloat16 *>(sm + L::OT + (warp - 2) * kOTileBytes);
        __nv_bfloat16 *zt = reinterpret_cast<__nv_bfloat16 *>(sm + L::ZT + (warp - 2) * kOTileBytes);
        // gated: this warp's z tile (32 tokens x 32 value rows) of chunk c,
        // TMA-loaded one chunk ahead
        auto load_z = [&](int c) {
            mbar_arrive_expect_tx(&B.zbar[warp - 2], kOTileBytes);
            tma_load_2d(zt, &tm_z, &B.zbar[warp - 2], h * DH + q4 * 32,
                        (int)(s_start + (int64_t)c * C + 32 * hf));
        };
        float wb = 0.f;
        if constexpr (kGated) {
            wb = gate.w[b];
            if (lane == 0) load_z(0);
        }
        // E0: this half of the initial state -> bf16 operand copy, and the
        //     fp32 accumulator pre-scaled by the first chunk's total decay
        {
            mbar_wait(&B.c_full[0], 0, abort);
            const float gn = scal(0).gam_n;
            const float *src = islot >= 0 ? pool_in + islot * slot_stride + head_off + (size_t)b * DH + hf * 64
                                          : nullptr;
            for (int c0 = 0; c0 < 64; c0 += 32) {
                uint32_t v[32], pk[16];
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const float4 f = src ? *reinterpret_cast<const float4 *>(src + c0 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
                    v[j] = __float_as_uint(f.x); v[j + 1] = __float_as_uint(f.y);
                    v[j + 2] = __float_as_uint(f.z); v[j + 3] = __float_as_uint(f.w);
                }
                if (ident) {   // S_0 = I: row b holds a one in column b
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(hf * 64 + c0 + j == b ? 1.f : 0.f);
                }
#pragma unroll
                for (int jj = 0; jj < 16; ++jj)
                    pk[jj] = pack_bf16(__uint_as_float(v[2 * jj]), __uint_as_float(v[2 * jj + 1]));
                tmem_st16(s16 + c0 / 2, pk);
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * gn);
                tmem_st32(s32 + c0, v);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&B.s_next);
            mbar_arrive(&B.o_free);
        }
        for (int c = 0; c < nch; ++c) {
            const ItemScal &I = scal(c);             // c_full(c) was waited one chunk earlier
            const int64_t c0 = s_start + (int64_t)c * C;
            const bool last = c == nch - 1;
            const int n = (int)min((int64_t)C, s_end - c0);   // rows of this chunk (bounds from cu)
            // ---- E2: U = U1 + U2 (this half) -> U16 = bf16(U), U16k = bf16(U diag(ks))
            mbar_wait(&B.u_full, c & 1, abort);
            tc_fence_after();
            {
                uint32_t u1[32], u2[32], uu[16], uk[16];
                tmem_ld32x2(lrow + kColU1 + 32 * hf, lrow + kColU2 + 32 * hf, u1, u2);
                const uint64_t *ks2 = reinterpret_cast<const uint64_t *>(I.ks + 32 * hf);
#pragma unroll
                for (int q = 0; q < 16; ++q) {   // pairs of columns, packed fp32
                    const uint64_t x = f2_add(f2_make(__uint_as_float(u1[2 * q]), __uint_as_float(u1[2 * q + 1])),
                                              f2_make(__uint_as_float(u2[2 * q]), __uint_as_float(u2[2 * q + 1])));
                    const uint64_t xk = f2_mul(x, ks2[q]);
                    float x0, x1, k0, k1;
                    f2_split(x, x0, x1);
                    f2_split(xk, k0, k1);
                    uu[q] = pack_bf16(x0, x1);
                    uk[q] = pack_bf16(k0, k1);
                }
                tmem_st16(lrow + kColU16k + 16 * hf, uk);
                tmem_st16(lrow + kColU16 + 16 * hf, uu);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&B.u2_full);
            // ---- E3a: S -> bf16 operand copy first (the next chunk's M2 waits
            //      on it), then the fp32 state pre-scaled by the next decay
            mbar_wait(&B.s_full, c & 1, abort);
            mbar_wait(&B.o1_full, c & 1, abort);     // O1 has read the old S16
            tc_fence_after();
            uint32_t sv[64];
            tmem_ld32x2(s32, s32 + 32, *reinterpret_cast<uint32_t(*)[32]>(sv),
                        *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
            if (!last) {
#pragma unroll
                for (int cc = 0; cc < 64; cc += 32) {
                    uint32_t pk[16];
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj)
                        pk[jj] = pack_bf16(__uint_as_float(sv[cc + 2 * jj]), __uint_as_float(sv[cc + 2 * jj + 1]));
                    tmem_st16(s16 + cc / 2, pk);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&B.s_next);
                mbar_wait(&B.c_full[(c + 1) % kCStages], ((c + 1) / kCStages) & 1, abort);
                const float gnext = scal(c + 1).gam_n;
                const uint64_t g2 = f2_make(gnext, gnext);
#pragma unroll
                for (int cc = 0; cc < 64; cc += 32) {
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        float a0, a1;
                        f2_split(f2_mul(f2_make(__uint_as_float(sv[cc + j]), __uint_as_float(sv[cc + j + 1])), g2),
                                 a0, a1);
                        sv[cc + j] = __float_as_uint(a0);
                        sv[cc + j + 1] = __float_as_uint(a1);
                    }
                    tmem_st32(s32 + cc, *reinterpret_cast<uint32_t(*)[32]>(sv + cc));
                }
            } else if (fslot >= 0) {
                float *dstp = pool_out + fslot * slot_stride + head_off + (size_t)b * DH + hf * 64;
#pragma unroll
                for (int j = 0; j < 64; j += 4)
                    *reinterpret_cast<float4 *>(dstp + j) = make_float4(
                        __uint_as_float(sv[j]), __uint_as_float(sv[j + 1]),
                        __uint_as_float(sv[j + 2]), __uint_as_float(sv[j + 3]));
            }
            // ---- o = diag(sq) O1 + O2 for rows 32 hf .. 32 hf + 31
            mbar_wait(&B.o2_full, c & 1, abort);
            tc_fence_after();
            uint32_t o1[32], o2[32];
            tmem_ld32x2(lrow + kColO1 + 32 * hf, lrow + kColO2 + 32 * hf, o1, o2);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&B.o_free);
            {
                // o rows 32 hf + i of column b; a full tile leaves through TMA,
                // a partial last one through plain stores
                const uint64_t *sq2 = reinterpret_cast<const uint64_t *>(I.sq + 32 * hf);
                float f[32];
#pragma unroll
                for (int q = 0; q < 16; ++q)   // pairs of tokens, packed fp32
                    f2_split(f2_fma(sq2[q],
                                    f2_make(__uint_as_float(o1[2 * q]), __uint_as_float(o1[2 * q + 1])),
                                    f2_make(__uint_as_float(o2[2 * q]), __uint_as_float(o2[2 * q + 1]))),
                             f[2 * q], f[2 * q + 1]);
                if constexpr (kGated) {
                    // sum of o^2 over the 128 value rows of each token: the
                    // warp's 32 rows by a reduce-scatter (lane l: token l),
                    // then the warpgroup's four warps through shared memory
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const uint64_t fi = f2_make(f[i], f[i + 1]);
                        f2_split(f2_mul(fi, fi), v[i], v[i + 1]);
                    }
                    reduce_scatter_step<32>(v, lane);
                    reduce_scatter_step<16>(v, lane);
                    reduce_scatter_step<8>(v, lane);
                    reduce_scatter_step<4>(v, lane);
                    reduce_scatter_step<2>(v, lane);
                    float *red = reinterpret_cast<float *>(sm + L::RED) + (hf * 2 + (c & 1)) * 128;
                    red[q4 * 32 + lane] = v[0];
                    named_sync(1 + hf, 128);
                    const float ss = red[lane] + red[32 + lane] + red[64 + lane] + red[96 + lane];
                    // each lane's token norm, read back by every lane as 8 float4
                    float *rs = reinterpret_cast<float *>(sm + L::RED) + 512 + (warp - 2) * 32;
                    rs[lane] = rsqrtf(ss * (1.0f / DH) + gate.eps);
                    __syncwarp();
                    mbar_wait(&B.zbar[warp - 2], c & 1, abort);
                    // y = o rstd w SiLU(z), SiLU by the one-instruction tanh
                    // form (below the bf16 rounding of y): the epilogue is
                    // issue-bound, and SiLU with an exact reciprocal cost a
                    // third of the chain's time
                    const uint64_t wb2 = f2_make(wb, wb), half2 = f2_make(0.5f, 0.5f);
#pragma unroll
                    for (int q = 0; q < 16; ++q) {   // pairs of tokens, packed fp32
                        const uint64_t rr2 = reinterpret_cast<const uint64_t *>(rs)[q];
                        const uint64_t h2 = f2_mul(f2_make(__bfloat162float(zt[(2 * q) * 32 + lane]),
                                                           __bfloat162float(zt[(2 * q + 1) * 32 + lane])),
                                                   half2);      // SiLU(z) = h + h tanh(h), h = z / 2
                        float h0, h1;
                        f2_split(h2, h0, h1);
                        const uint64_t sz = f2_fma(h2, f2_make(tanh_approx(h0), tanh_approx(h1)), h2);
                        f2_split(f2_mul(f2_make(f[2 * q], f[2 * q + 1]), f2_mul(f2_mul(rr2, wb2), sz)),
                                 f[2 * q], f[2 * q + 1]);
                    }
                    fence_async_smem();      // z reads (generic) before the next z load (async)
                    __syncwarp();
                    if (c + 1 < nch && lane == 0 && !*abort) load_z(c + 1);
                }
                if (32 * hf + 32 <= n) {
                    if (lane == 0) bulk_wait_read_all();     // the last tile has left
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 32; ++i) ot[i * 32 + lane] = __float2bfloat16_rn(f[i]);
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(tm_out, ot, h * DH + q4 * 32, (int)(c0 - row0 + 32 * hf));
                        bulk_commit();
                    }
                } else {
                    const int64_t ostride = (int64_t)hv * DH;
                    __nv_bfloat16 *orow = out + ((c0 - row0 + 32 * hf) * hv + h) * (int64_t)DH + b;
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (32 * hf + i < n) orow[i * ostride] = __float2bfloat16_rn(f[i]);
                }
            }
            mbar_arrive(&B.c_empty[c % kCStages]);
        }
        if (lane == 0) bulk_wait_read_all();         // the staged o tiles have been read
        if constexpr (kGated) {
            if (lane == 0) {   // never leave with a z load in flight
                int z = 0;
                mbar_wait(&B.zbar[warp - 2], (nch - 1) & 1, &z);
            }
        }
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
    }
    if (tid == 0 && B.abort) flag_status(GDN_DEVSTAT_TIMEOUT);
    if (tid == 0) griddep_wait();   // no-op once the producer has waited
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
                         void *o, void *ws, cudaStream_t s, const void *z, int64_t zs,
                         const float *norm_w, float norm_eps, const void *ga, const void *gb,
                         const float *A_log, const float *dt_bias) {
    const psp::RawGates rg{(const __nv_bfloat16 *)ga, (const __nv_bfloat16 *)gb, A_log, dt_bias};
    const int64_t items = psp::chunk_bound(n_tokens, n_seqs) * hv;
    if (items >= (1ll << 31)) return GDN_ERR_UNSUPPORTED;
    CUtensorMap tq, tk, tv, to, tz;
    const uint64_t rows = (uint64_t)n_tokens;
    const bool gated = z != nullptr;
    if (!encode_tmap_2d_bf16(&tq, q, (uint64_t)hqk * 128, rows, qs, 64, 64) ||
        !encode_tmap_2d_bf16(&tk, k, (uint64_t)hqk * 128, rows, ks, 64, 64) ||
        !encode_tmap_2d_bf16(&tv, v, (uint64_t)hv * 128, rows, vs, 64, 64) ||
        !encode_tmap_2d_bf16(&to, o, (uint64_t)hv * 128, rows, (uint64_t)hv * 128, 32, 32, false) ||
        (gated && !encode_tmap_2d_bf16(&tz, z, (uint64_t)hv * 128, rows, (uint64_t)zs, 32, 32, false)))
        return GDN_ERR_LAUNCH;
    cudaError_t e = cudaFuncSetAttribute(psp::prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)psp::P_SMEM_BYTES);
    if (e == cudaSuccess)
        e = gated ? cudaFuncSetAttribute(psp::chain_kernel<true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)psp::ChainSmem<true>::BYTES)
                  : cudaFuncSetAttribute(psp::chain_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)psp::ChainSmem<false>::BYTES);
    if (e != cudaSuccess) {
        set_last_cuda_error(e);
        return GDN_ERR_LAUNCH;
    }
    int32_t *base = reinterpret_cast<int32_t *>(ws);
    uint8_t *item_blocks = reinterpret_cast<uint8_t *>(ws) + psp::header_bytes(n_seqs);
    psp::chunk_base_kernel<<<1, 1024, 0, s>>>(cu, n_seqs, n_tokens, base);
    gdn_status st = launch_status();
    if (st != GDN_OK) return st;
    e = launch_after(psp::prep_kernel, dim3(psp::prep_grid(items)), dim3(psp::kPrepKernelThreads),
                     psp::P_SMEM_BYTES, s, tq, tk, g, beta, rg, cu, (const int32_t *)base, n_seqs,
                     hv, hv / hqk, scale, l2norm, item_blocks);
    if (e != cudaSuccess) {
        set_last_cuda_error(e);
        return GDN_ERR_LAUNCH;
    }
    const dim3 grid((unsigned)((int64_t)n_seqs * hv));
    if (gated)
        e = launch_after(psp::chain_kernel<true>, grid, dim3(psp::kChainKernelThreads),
                         psp::ChainSmem<true>::BYTES, s, tq, tk, tv, to, to, tz,
                         psp::GateArgs{norm_w, norm_eps}, cu, (const int32_t *)base, n_seqs,
                         n_tokens, hv, hv / hqk, (const uint8_t *)item_blocks,
                         (const float *)pool, n_slots, pool, n_slots, ii, fi,
                         (__nv_bfloat16 *)o, (__nv_bfloat16 *)nullptr, psp::IdentChains{0, 0, 0});
    else
        e = launch_after(psp::chain_kernel<false>, grid, dim3(psp::kChainKernelThreads),
                         psp::ChainSmem<false>::BYTES, s, tq, tk, tv, to, to, to,
                         psp::GateArgs{nullptr, 0.f}, cu, (const int32_t *)base, n_seqs,
                         n_tokens, hv, hv / hqk, (const uint8_t *)item_blocks,
                         (const float *)pool, n_slots, pool, n_slots, ii, fi,
                         (__nv_bfloat16 *)o, (__nv_bfloat16 *)nullptr, psp::IdentChains{0, 0, 0});
    if (e != cudaSuccess) {
        set_last_cuda_error(e);
        return GDN_ERR_LAUNCH;
    }
    return GDN_OK;
}

// ------------------------------------------------- chunk-state scan (host) --
// One sequence of at least kScanMinChunks chunks runs as two segments (see
// prefill_scan.cu): one prep launch over both, one chain launch of 3 x hv
// CTAs (segment 0 from the true initial state, segment 1 from zero and from
// the identity), then the combine and the output correction.
namespace psp {
constexpr int64_t kScanMinChunks = 64;

inline size_t align1k(size_t x) { return (x + 1023) / 1024 * 1024; }
inline int64_t scan_phi_rows(int64_t n_tokens) {   // rows of segment 1 at most
    const int64_t nch = (n_tokens + C - 1) / C;
    return (int64_t)C * (nch - (nch + 1) / 2);
}
struct ScanLayout {
    size_t base, idx, items, states, s1b, phi, total;
};
inline ScanLayout scan_layout(int64_t n_tokens, int hv) {
    ScanLayout L;
    L.base = 0;                        // chunk offsets of the two segments
    L.idx = 1024;                      // scan::ScanIdx
    L.items = 2048;
    L.states = align1k(L.items + (size_t)chunk_bound(n_tokens, 2) * hv * kItemBytes);
    L.s1b = L.states + (size_t)scan::kScratchSlots * hv * DH * DH * 4;
    L.phi = L.s1b + (size_t)hv * scan::kS1bBytes;
    L.total = align1k(L.phi + (size_t)scan_phi_rows(n_tokens) * hv * DH * 2);
    return L;
}
}  // namespace psp

bool prefill_scan_sized(int n_seqs, int64_t n_tokens) {
    return n_seqs == 1 && (n_tokens + psp::C - 1) / psp::C >= psp::kScanMinChunks;
}
// The scan pays only while its 3 x hv chain CTAs run at once, one per SM.
bool prefill_scan_fits(int hv) { return 3 * hv <= sm_count(); }
size_t prefill_scan_workspace(int64_t n_tokens, int hv) {
    return psp::scan_layout(n_tokens, hv).total;
}

gdn_status prefill_scan(const void *q, int64_t qs, const void *k, int64_t ks, const void *v,
                        int64_t vs, const float *g, const float *beta, const int32_t *cu,
                        int64_t n_tokens, int hqk, int hv, float scale, int l2norm, float *pool,
                        int64_t n_slots, const int32_t *ii, const int32_t *fi, void *o, void *ws,
                        cudaStream_t s, const void *ga, const void *gb, const float *A_log,
                        const float *dt_bias) {
    const psp::RawGates rg{(const __nv_bfloat16 *)ga, (const __nv_bfloat16 *)gb, A_log, dt_bias};
    const psp::ScanLayout L = psp::scan_layout(n_tokens, hv);
    const int64_t items = psp::chunk_bound(n_tokens, 2) * hv;
    if (items >= (1ll << 31)) return GDN_ERR_UNSUPPORTED;
    uint8_t *w = reinterpret_cast<uint8_t *>(ws);
    int32_t *base = reinterpret_cast<int32_t *>(w + L.base);
    scan::ScanIdx *idx = reinterpret_cast<scan::ScanIdx *>(w + L.idx);
    const int32_t *cu_all = reinterpret_cast<const int32_t *>(w + L.idx + offsetof(scan::ScanIdx, cu_all));
    const int32_t *seg_init = reinterpret_cast<const int32_t *>(w + L.idx + offsetof(scan::ScanIdx, init));
    const int32_t *seg_fin = reinterpret_cast<const int32_t *>(w + L.idx + offsetof(scan::ScanIdx, fin));
    uint8_t *item_blocks = w + L.items;
    float *states = reinterpret_cast<float *>(w + L.states);
    void *phi = w + L.phi;
    const int64_t phi_rows = psp::scan_phi_rows(n_tokens);
    CUtensorMap tq, tk, tv, to, tphi;
    const uint64_t rows = (uint64_t)n_tokens;
    if (!encode_tmap_2d_bf16(&tq, q, (uint64_t)hqk * 128, rows, qs, 64, 64) ||
        !encode_tmap_2d_bf16(&tk, k, (uint64_t)hqk * 128, rows, ks, 64, 64) ||
        !encode_tmap_2d_bf16(&tv, v, (uint64_t)hv * 128, rows, vs, 64, 64) ||
        !encode_tmap_2d_bf16(&to, o, (uint64_t)hv * 128, rows, (uint64_t)hv * 128, 32, 32, false) ||
        !encode_tmap_2d_bf16(&tphi, phi, (uint64_t)hv * 128, (uint64_t)phi_rows,
                             (uint64_t)hv * 128, 32, 32, false))
        return GDN_ERR_LAUNCH;
    cudaError_t e = cudaFuncSetAttribute(psp::prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)psp::P_SMEM_BYTES);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(psp::chain_kernel<false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)psp::ChainSmem<false>::BYTES);
    if (e != cudaSuccess) {
        set_last_cuda_error(e);
        return GDN_ERR_LAUNCH;
    }
    gdn_status st = scan_setup(cu, n_tokens, ii, fi, n_slots, idx, s);
    if (st != GDN_OK) return st;
    psp::chunk_base_kernel<<<1, 1024, 0, s>>>(cu_all, 2, n_tokens, base);
    if ((st = launch_status()) != GDN_OK) return st;
    e = launch_after(psp::prep_kernel, dim3(psp::prep_grid(items)), dim3(psp::kPrepKernelThreads),
                     psp::P_SMEM_BYTES, s, tq, tk, g, beta, rg, cu_all, (const int32_t *)base, 2, hv,
                     hv / hqk, scale, l2norm, item_blocks);
    if (e == cudaSuccess)
        e = launch_after(psp::chain_kernel<false>, dim3((unsigned)(3 * hv)),
                         dim3(psp::kChainKernelThreads), psp::ChainSmem<false>::BYTES, s, tq, tk,
                         tv, to, tphi, tphi, psp::GateArgs{nullptr, 0.f}, cu_all,
                         (const int32_t *)base, 2, n_tokens, hv, hv / hqk,
                         (const uint8_t *)item_blocks, (const float *)pool, n_slots, states,
                         (int64_t)scan::kScratchSlots, seg_init, seg_fin, (__nv_bfloat16 *)o,
                         (__nv_bfloat16 *)phi, psp::IdentChains{1, 1, scan::kSlotA});
    if (e != cudaSuccess) {
        set_last_cuda_error(e);
        return GDN_ERR_LAUNCH;
    }
    return scan_finish(states, hv, idx, pool, w + L.s1b, phi, phi_rows, o, n_tokens, s);
}

}  // namespace gdn

using namespace gdn;

// Test control of the failure path of the two-kernel prefill: the wait limit
// of its kernels and the prep kernel's K|Q loads (see gdn.h).
extern "C" gdn_status gdn_debug_set_wait_limit(uint64_t limit_ns, int32_t drop_prep_loads,
                                               void *stream) {
    const uint64_t lim = limit_ns ? limit_ns : tc::kWaitLimitNs;
    const int drop = drop_prep_loads != 0;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaMemcpyToSymbolAsync(tc::g_wait_limit_ns, &lim, sizeof(lim), 0,
                                            cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbolAsync(g_prep_drop_loads, &drop, sizeof(drop), 0,
                                    cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);   // the sources live on this stack
    if (e != cudaSuccess) {
        set_last_cuda_error(e);
        return GDN_ERR_CUDA;
    }
    return GDN_OK;
}
