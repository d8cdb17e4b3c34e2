// Chunked varlen prefill of the gated delta rule on the 5th-generation tensor
// cores (tcgen05 + TMEM + TMA), bf16 activations, dk = dv = 128, chunk 64
// ("Flash Linear Attention operations for efficient chunked computations",
// "[model] Support Qwen3next", Highlights).
//
// One CTA per (sequence, V head) chain; 14 warps:
//   warp 0        TMA producer: raw K|Q tiles (3 stages) and V tiles (2 stages)
//   warp 1        TMEM owner + the single thread that issues every tcgen05.mma
//   warps 2..9    "prep": everything that does not depend on the state, one
//                 chunk ahead of the chain (gating prefix sums, q/k norms,
//                 the UT transform T = (I + A)^-1 by a blocked fp32 solve, P)
//   warps 10..13  "chain": the state-dependent epilogues
//
// Per chunk (rows i, j = tokens, b = value index, a = key index; S is the
// fp32 state [b][a]; gc = prefix sum of g, Gam = exp(gc); D = exp(gc_i-gc_j);
// r_k, r_q = inverse L2 norms):
//   M1  G  = [K;Q] K^T                  prep: A (K rows) and P (Q rows) from G
//   MU  U  = T1 V                       T1 = T diag(beta)         (V^T read MN-major)
//   M23 [X | O] = S [K; Q']^T           one N = 128 MMA; X[b][j], O[b][i];
//                                       A operand: bf16 copy of S in TMEM;
//                                       Q' = scale Gam r_q Q (rows rescaled in place)
//   E1  X -> bf16 in TMEM
//   M4  U += T2 X^T                     T2 = -T diag(beta Gam r_k), so that
//                                       U = T diag(beta) (V - diag(Gam r_k) K S^T)
//   E2  U -> bf16 in TMEM
//   M5  O += U P^T       P[i][j] = scale D_ij r_q,i r_k,j (q_i . k_j), j <= i
//   M6  S += U K''       K''_j = D[last][j] r_k,j K_j (rows rescaled in place);
//                        S was pre-scaled by Gam_last by the previous epilogue
//   E3  S -> bf16 copy (and pre-scaled for the next chunk) and O -> registers,
//       hand-off to the next chunk, then the o stores
// Padded rows of a partial last chunk get beta = g = 0 and explicit zero masks.
#include "prefill_common.cuh"

namespace gdn {

GDN_DECLARE_STATUS_WORD(g_status_prefill_tc)
GDN_STATUS_READER(read_status_prefill_tc, g_status_prefill_tc)

namespace ptc {
using namespace tc;

constexpr int kWarps = 14;
constexpr int kThreads = kWarps * 32;
constexpr int kPrepThreads = 256;
constexpr int kChainThreads = 128;
constexpr int kKQStages = 3;
constexpr int kVStages = 2;
constexpr uint32_t kDBytes = 3 * kMatBytes;      // derived stage: T1, T2, P

// TMEM columns
constexpr uint32_t kColS32 = 0, kColS16 = 128, kColG = 192, kColU = 256, kColX = 320,
                   kColO = 384, kTmemCols = 512;   // X and O adjacent: one N = 128 MMA

struct Scal {
    float beta[C], gam[C], alpha[C], rk[C], rq[C], xs[C], ks[C];
    float gam_n;
    int n;
};

struct Bars {
    uint64_t kq_full[kKQStages], kq_empty[kKQStages], v_full[kVStages], v_empty[kVStages];
    uint64_t g_full, g_free, prep_done[2], gn_ready[2], d_free[2], x_full, r_full, u_full,
        u2_full, s_full, s_next, mma_done;
    uint32_t tmem_base;
    int abort;
    int seq;
    float tot0;
};

constexpr uint32_t OFF_KQ = 0;
constexpr uint32_t OFF_V = OFF_KQ + kKQStages * kKQBytes;
constexpr uint32_t OFF_D = OFF_V + kVStages * kVBytes;
constexpr uint32_t OFF_AF = OFF_D + 2 * kDBytes;
constexpr uint32_t OFF_TF = OFF_AF + C * kLd * 4;
constexpr uint32_t OFF_WB = OFF_TF + C * kLd * 4;
constexpr uint32_t kWbFloats = 8 * 16 * kWbLd + 16 * 16;   // 8 warps' 16x8 scratch + Z30
constexpr uint32_t OFF_SCAL = OFF_WB + kWbFloats * 4;
constexpr uint32_t kScalBytes = (sizeof(Scal) + 127) / 128 * 128;
constexpr uint32_t OFF_BARS = OFF_SCAL + 2 * kScalBytes;
constexpr uint32_t SMEM_USED = OFF_BARS + (sizeof(Bars) + 127) / 128 * 128;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;    // slack to align the base to 1024
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const float *__restrict__ g,
                  const float *__restrict__ beta, const int32_t *__restrict__ cu, int n_seqs,
                  int64_t n_tokens, int hv, int grp, float scale, int l2norm,
                  float *__restrict__ pool, int64_t n_slots, const int32_t *__restrict__ init_idx,
                  const int32_t *__restrict__ final_idx, __nv_bfloat16 *__restrict__ o) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    Bars &B = *reinterpret_cast<Bars *>(sm + OFF_BARS);
    float *Af = reinterpret_cast<float *>(sm + OFF_AF);
    float *Tf = reinterpret_cast<float *>(sm + OFF_TF);
    float *Wb = reinterpret_cast<float *>(sm + OFF_WB);
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
            for (int e = tid; e < DH * DH; e += kThreads)
                pool[fslot * slot_stride + head_off + e] =
                    islot >= 0 ? pool[islot * slot_stride + head_off + e] : 0.f;
        return;
    }

    if (warp == 1) {
        tmem_alloc(&B.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < kKQStages; ++s) { mbar_init(&B.kq_full[s], 1); mbar_init(&B.kq_empty[s], 1); }
        for (int s = 0; s < kVStages; ++s) { mbar_init(&B.v_full[s], 1); mbar_init(&B.v_empty[s], 1); }
        mbar_init(&B.g_full, 1);
        mbar_init(&B.g_free, kPrepThreads);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&B.prep_done[s], kPrepThreads);
            mbar_init(&B.gn_ready[s], C);
            mbar_init(&B.d_free[s], kChainThreads);
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
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tensormap(&tm_q);
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
            int kq_issued[kKQStages] = {0, 0, 0}, v_issued[kVStages] = {0, 0};
            for (int c = 0; c < nch && !*abort; ++c) {
                const int y = (int)(s_start + (int64_t)c * C);
                const int sk = c % kKQStages, sv = c % kVStages;
                if (c >= kKQStages) mbar_wait(&B.kq_empty[sk], ((c / kKQStages) - 1) & 1, abort);
                uint8_t *kq = sm + OFF_KQ + sk * kKQBytes;
                mbar_arrive_expect_tx(&B.kq_full[sk], kKQBytes);
                for (int kb = 0; kb < 2; ++kb) {
                    tma_load_2d(kq + kb * kKBlk, &tm_k, &B.kq_full[sk], hq * DH + kb * 64, y);
                    tma_load_2d(kq + kb * kKBlk + 64 * 128, &tm_q, &B.kq_full[sk], hq * DH + kb * 64, y);
                }
                kq_issued[sk] = c / kKQStages + 1;
                if (c >= kVStages) mbar_wait(&B.v_empty[sv], ((c / kVStages) - 1) & 1, abort);
                uint8_t *vt = sm + OFF_V + sv * kVBytes;
                mbar_arrive_expect_tx(&B.v_full[sv], kVBytes);
                for (int kb = 0; kb < 2; ++kb)
                    tma_load_2d(vt + kb * kVBlk, &tm_v, &B.v_full[sv], h * DH + kb * 64, y);
                v_issued[sv] = c / kVStages + 1;
            }
            // never leave with copies in flight: wait for the last load of every stage
            for (int s = 0; s < kKQStages; ++s)
                if (kq_issued[s]) { int z = 0; mbar_wait(&B.kq_full[s], (kq_issued[s] - 1) & 1, &z); }
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
            auto kq_base = [&](int c) { return smem_u32(sm + OFF_KQ + (c % kKQStages) * kKQBytes); };
            auto issue_g = [&](int c) {   // M1: G = [K;Q] K^T
                const uint32_t base = kq_base(c);
                for (int s = 0; s < 8; ++s) {
                    const uint32_t off = (s >> 2) * kKBlk + (s & 3) * 32;
                    mma_ss(tbase + kColG, sdesc_sw128(base + off, 16, 1024),
                           sdesc_sw128(base + off, 16, 1024), id64, s > 0);
                }
                mma_commit(&B.g_full);
            };
            mbar_wait(&B.kq_full[0], 0, abort);
            tc_fence_after();
            issue_g(0);
            for (int c = 0; c < nch; ++c) {
                const int sd = c & 1, sv = c % kVStages;
                const uint32_t base = kq_base(c);
                const uint32_t dsm = smem_u32(sm + OFF_D + sd * kDBytes);   // T1 | T2 | P
                const uint32_t vsm = smem_u32(sm + OFF_V + sv * kVBytes);
                // the next chunk's G as soon as the prep group has read this one
                mbar_wait(&B.g_free, c & 1, abort);
                if (c + 1 < nch) {
                    mbar_wait(&B.kq_full[(c + 1) % kKQStages], ((c + 1) / kKQStages) & 1, abort);
                    tc_fence_after();
                    issue_g(c + 1);
                }
                mbar_wait(&B.prep_done[sd], (c >> 1) & 1, abort);
                mbar_wait(&B.s_next, c & 1, abort);
                mbar_wait(&B.v_full[sv], (c / kVStages) & 1, abort);
                tc_fence_after();
                for (int s = 0; s < 4; ++s)   // MU: U = T1 V  (A = V^T, MN-major)
                    mma_ss(tbase + kColU, sdesc_sw128(vsm + s * 16 * 128, kVBlk, 1024),
                           sdesc_sw128(dsm + s * 32, 16, 1024), id64amn, s > 0);
                mma_commit(&B.v_empty[sv]);
                for (int s = 0; s < 8; ++s) {   // M23: [X | O] = S [K; Q']^T
                    const uint32_t off = (s >> 2) * kKBlk + (s & 3) * 32;
                    mma_ts(tbase + kColX, tbase + kColS16 + s * 8, sdesc_sw128(base + off, 16, 1024),
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
                           sdesc_sw128(base + s * 16 * 128, kKBlk, 1024), id128bmn, 1);
                }
                mma_commit(&B.s_full);
                mma_commit(&B.kq_empty[c % kKQStages]);
            }
            mma_commit(&B.mma_done);
            int z = 0;
            mbar_wait(&B.mma_done, 0, &z);
        }
        __syncwarp();
    } else if (warp < 10) {
        // ---------------------------------------------------- prep (8 warps)
        const int t = tid - 64;                  // 0 .. 255
        const int pw = warp - 2;                 // 0 .. 7
        const int q4 = warp & 3;                 // TMEM lane quadrant
        const int p = q4 * 32 + lane;            // G row: 0..63 K rows, 64..127 Q rows
        const int chalf = pw >> 2;               // which 32 G columns this warp reads
        for (int c = 0; c < nch; ++c) {
            const int sd = c & 1, sk = c % kKQStages;
            Scal &S = *reinterpret_cast<Scal *>(sm + OFF_SCAL + sd * kScalBytes);
            uint8_t *kq = sm + OFF_KQ + sk * kKQBytes;
            uint8_t *dst = sm + OFF_D + sd * kDBytes;
            const int64_t c0 = s_start + (int64_t)c * C;
            const int n = (int)min((int64_t)C, s_end - c0);
            // warp 0 of the group holds the chunk's gates, rows 2l and 2l+1 per lane
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
            if (c >= 2) mbar_wait(&B.d_free[sd], ((c >> 1) - 1) & 1, abort);
            mbar_wait(&B.kq_full[sk], (c / kKQStages) & 1, abort);
            // ---- inverse norms of the K rows (0..63) and Q rows (64..127)
            {
                const float r = kq_row_inv_norm(kq, t, l2norm);
                const int row = t >> 1;
                if ((t & 1) == 0) {
                    if (row < C) S.rk[row] = r; else S.rq[row - C] = r;
                }
            }
            // ---- prefix sum of g (one warp), per-token decay alpha = exp(g)
            if (t < 32) {
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
            if (t < C) {
                const float gl = S.gam[C - 1];      // padded rows carry g = 0
                const float x = S.gam[t];
                const bool ok = t < n;
                S.xs[t] = ok ? __expf(x) * S.rk[t] : 0.f;
                S.ks[t] = ok ? __expf(gl - x) * S.rk[t] : 0.f;
                if (t == 0) {
                    S.gam_n = __expf(gl);
                    S.n = n;
                }
                mbar_arrive(&B.gn_ready[sd]);   // the chain needs these early
            }
            // ---- G -> A (K rows, fp32 scratch) and P (Q rows, bf16 operand)
            mbar_wait(&B.g_full, c & 1, abort);
            tc_fence_after();
            uint32_t gr[32];
            tmem_ld32(tmem_addr(tbase, q4 * 32, kColG + 32 * chalf), gr);
            tc_fence_before();
            mbar_arrive(&B.g_free);
            g_to_a_p(gr, p, chalf, n, S.beta, S.gam, S.alpha, S.rk, S.rq, scale, Af, dst + 2 * kMatBytes);
            named_sync(1, kPrepThreads);
            // ---- T = (I + A)^-1 and the T1 / T2 operands
            ut_solve<true>(Af, Tf, Wb, t, pw, lane, S.beta, S.xs, dst);
            fence_async_smem();
            mbar_arrive(&B.prep_done[sd]);
            named_sync(1, kPrepThreads);   // the solve scratch is free again
        }
    } else {
        // --------------------------------------------------- chain (4 warps)
        const int tc4 = tid - 320;                // 0 .. 127
        const int q4 = warp & 3;
        const int b = q4 * 32 + lane;            // value row of the state
        const uint32_t lrow = tmem_addr(tbase, q4 * 32, 0);
        // Q' = scale Gam_i r_q,i Q_i in place for chunk cq, once its scalars are
        // out and M1 has read the raw rows (g_free); before M23 of that chunk.
        auto rescale_q = [&](int cq) {
            const int sq = cq & 1;
            mbar_wait(&B.gn_ready[sq], (cq >> 1) & 1, abort);
            mbar_wait(&B.g_free, cq & 1, abort);
            const Scal &Sq = *reinterpret_cast<const Scal *>(sm + OFF_SCAL + sq * kScalBytes);
            uint8_t *kqq = sm + OFF_KQ + (cq % kKQStages) * kKQBytes;
            const int i = tc4 >> 1, kb = tc4 & 1;
            const float f = i < Sq.n ? scale * __expf(Sq.gam[i]) * Sq.rq[i] : 0.f;
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
            mbar_wait(&B.gn_ready[0], 0, abort);
            const float gn = reinterpret_cast<const Scal *>(sm + OFF_SCAL)->gam_n;
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
            const int sd = c & 1, sk = c % kKQStages;
            const Scal &S = *reinterpret_cast<const Scal *>(sm + OFF_SCAL + sd * kScalBytes);
            uint8_t *kq = sm + OFF_KQ + sk * kKQBytes;
            const int64_t c0 = s_start + (int64_t)c * C;
            const bool last = c == nch - 1;
            mbar_wait(&B.prep_done[sd], (c >> 1) & 1, abort);
            const int n = S.n;
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
            // K'' = D[last][j] r_k,j K_j in place (M1, M2 have consumed the raw rows)
            {
                const int j = tc4 >> 1, kb = tc4 & 1;
                const float f = S.ks[j];
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
            float gnext = 1.f;
            if (!last) {
                mbar_wait(&B.gn_ready[sd ^ 1], ((c + 1) >> 1) & 1, abort);
                gnext = reinterpret_cast<const Scal *>(sm + OFF_SCAL + (sd ^ 1) * kScalBytes)->gam_n;
            }
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
            tc_fence_before();
            mbar_arrive(&B.d_free[sd]);
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

}  // namespace ptc

static bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

bool prefill_tc_supported(int dtype, int dk, int dv, int chunk, const void *q, int64_t qs,
                          const void *k, int64_t ks, const void *v, int64_t vs) {
    return dtype == GDN_BF16 && dk == 128 && dv == 128 && chunk == 64 && aligned16(q) &&
           aligned16(k) && aligned16(v) && (qs * 2) % 16 == 0 && (ks * 2) % 16 == 0 &&
           (vs * 2) % 16 == 0;
}

gdn_status prefill_tc(const void *q, int64_t qs, const void *k, int64_t ks, const void *v,
                      int64_t vs, const float *g, const float *beta, const int32_t *cu,
                      int n_seqs, int64_t n_tokens, int hqk, int hv, float scale, int l2norm,
                      float *pool, int64_t n_slots, const int32_t *ii, const int32_t *fi,
                      void *o, cudaStream_t s) {
    CUtensorMap tq, tk, tv;
    const uint64_t rows = (uint64_t)n_tokens;
    if (!encode_tmap_2d_bf16(&tq, q, (uint64_t)hqk * 128, rows, qs, 64, 64) ||
        !encode_tmap_2d_bf16(&tk, k, (uint64_t)hqk * 128, rows, ks, 64, 64) ||
        !encode_tmap_2d_bf16(&tv, v, (uint64_t)hv * 128, rows, vs, 64, 64))
        return GDN_ERR_LAUNCH;
    cudaError_t e = cudaFuncSetAttribute(ptc::prefill_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)ptc::SMEM_BYTES);
    if (e != cudaSuccess) {
        set_last_cuda_error(e);
        return GDN_ERR_LAUNCH;
    }
    const int64_t blocks = (int64_t)n_seqs * hv;
    ptc::prefill_tc_kernel<<<(unsigned)blocks, ptc::kThreads, ptc::SMEM_BYTES, s>>>(
        tq, tk, tv, g, beta, cu, n_seqs, n_tokens, hv, hv / hqk, scale, l2norm, pool, n_slots,
        ii, fi, (__nv_bfloat16 *)o);
    return launch_status();
}

}  // namespace gdn
