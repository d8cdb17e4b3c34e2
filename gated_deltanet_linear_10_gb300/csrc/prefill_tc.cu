// Chunked varlen prefill of the gated delta rule on the 5th-generation tensor
// cores (tcgen05 + TMEM + TMA), bf16 activations, dk = dv = 128, chunk 64
// ("Flash Linear Attention operations for efficient chunked computations",
// "[model] Support Qwen3next", Highlights).
//
// One CTA per (sequence, V head) chain; 10 warps:
//   warp 0      TMA producer: raw K|Q tiles (3 stages) and V tiles (2 stages)
//   warp 1      TMEM owner + the single thread that issues every tcgen05.mma
//   warps 2..5  "prep": everything that does not depend on the state, one
//               chunk ahead of the chain (gating prefix sums, q/k norms, the
//               UT transform T = (I + A)^-1 by a blocked fp32 solve, P)
//   warps 6..9  "chain": the state-dependent epilogues
//
// Per chunk (rows i, j = tokens, b = value index, a = key index; S is the
// fp32 state [b][a]; gc = prefix sum of g, Gam = exp(gc); D = exp(gc_i-gc_j)):
//   M1  G  = [K;Q] K^T                    (prep: A from the K rows, P from the Q rows)
//   M2  X  = S K^T          X[b][j]       (A operand: bf16 copy of S in TMEM)
//   M3  O  = S Q'^T         Q' = scale Gam r_q Q (rows rescaled in place)
//   E1  R[b][j] = beta_j (V[j][b] - Gam_j r_k,j X[b][j])   -> bf16 into TMEM
//   M4  U  = R T^T          U[b][i] = (T R)[i][b]
//   E2  U -> bf16 in TMEM
//   M5  O += U P^T          P[i][j] = scale D_ij r_q,i r_k,j (q_i . k_j), j <= i
//   M6  S += U K''          K''_j = D[last][j] r_k,j K_j (rows rescaled in place),
//                           S pre-scaled by Gam_last in E1
//   E3  o <- O, S -> bf16 copy for the next chunk (final state -> pool)
// Padded rows of a partial last chunk get beta = g = 0 and explicit zero masks.
#include "common.cuh"
#include "tc.cuh"

namespace gdn {

GDN_DECLARE_STATUS_WORD(g_status_prefill_tc)
GDN_STATUS_READER(read_status_prefill_tc, g_status_prefill_tc)

namespace ptc {
using namespace tc;

constexpr int C = 64;                  // chunk
constexpr int DH = 128;                // dk = dv
constexpr int kThreads = 320;
constexpr int kKQStages = 3;
constexpr int kVStages = 2;
constexpr uint32_t kKQBytes = 2 * 128 * 128;     // 2 k-blocks x (64 K rows + 64 Q rows) x 128 B
constexpr uint32_t kKBlk = 128 * 128;            // k-block stride inside a K|Q stage
constexpr uint32_t kVBytes = 2 * 64 * 128;       // 2 k-blocks x 64 rows x 128 B
constexpr uint32_t kVBlk = 64 * 128;
constexpr uint32_t kTBytes = 64 * 128;           // T[i][j], one k-block
constexpr uint32_t kPBytes = 64 * 128;           // P[i][j]
constexpr int kLd = 68;                          // fp32 row stride of the solve scratch
constexpr float kEps = 1e-6f;

// TMEM columns
constexpr uint32_t kColS32 = 0, kColS16 = 128, kColG = 192, kColX = 256, kColU = 320,
                   kColO = 384, kTmemCols = 512;

struct Scal {
    float beta[C], gam[C], rk[C], rq[C], xs[C], ks[C];
    float gam_n;
    int n;
};

struct Bars {
    uint64_t kq_full[kKQStages], kq_empty[kKQStages], v_full[kVStages], v_empty[kVStages];
    uint64_t g_full, prep_done[2], d_free[2], x_full, r_full, u_full, u2_full, s_full, s_next,
        mma_done;
    uint32_t tmem_base;
    int abort;
    int seq;
};

constexpr uint32_t OFF_KQ = 0;
constexpr uint32_t OFF_V = OFF_KQ + kKQStages * kKQBytes;
constexpr uint32_t OFF_T = OFF_V + kVStages * kVBytes;
constexpr uint32_t OFF_P = OFF_T + 2 * kTBytes;
constexpr uint32_t OFF_AF = OFF_P + 2 * kPBytes;
constexpr uint32_t OFF_TF = OFF_AF + C * kLd * 4;
constexpr uint32_t OFF_WB = OFF_TF + C * kLd * 4;
constexpr uint32_t OFF_SCAL = OFF_WB + 4 * 16 * 20 * 4;
constexpr uint32_t kScalBytes = (sizeof(Scal) + 127) / 128 * 128;
constexpr uint32_t OFF_BARS = OFF_SCAL + 2 * kScalBytes;
constexpr uint32_t SMEM_USED = OFF_BARS + (sizeof(Bars) + 127) / 128 * 128;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;    // slack to align the base to 1024
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Rank -> sequence in decreasing-length order (ties by index), so that the
// longest chains start first.  Every thread tests a share of the candidates.
__device__ int seq_for_rank(const int32_t *cu, int n_seqs, int rank, int *slot) {
    if (n_seqs > 1024) return rank;
    if (threadIdx.x == 0) *slot = -1;
    __syncthreads();
    for (int i = threadIdx.x; i < n_seqs; i += blockDim.x) {
        const int li = cu[i + 1] - cu[i];
        int r = 0;
        for (int j = 0; j < n_seqs; ++j) {
            const int lj = cu[j + 1] - cu[j];
            r += (lj > li) || (lj == li && j < i);
        }
        if (r == rank) *slot = i;
    }
    __syncthreads();
    return *slot < 0 ? rank : *slot;
}

// 16x16 block products for the blocked UT solve.  A warp owns one block;
// lane (r = lane/2, hh = lane%2) holds row r, columns 8hh .. 8hh+7.
__device__ __forceinline__ void blk_mac(float (&acc)[8], const float *X, int xr, int xc,
                                        const float *Y, int yr, int yc, int r, int hh) {
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
        const float x = X[(xr + r) * kLd + xc + kk];
        const float4 y0 = *reinterpret_cast<const float4 *>(Y + (yr + kk) * kLd + yc + 8 * hh);
        const float4 y1 = *reinterpret_cast<const float4 *>(Y + (yr + kk) * kLd + yc + 8 * hh + 4);
        acc[0] = fmaf(x, y0.x, acc[0]); acc[1] = fmaf(x, y0.y, acc[1]);
        acc[2] = fmaf(x, y0.z, acc[2]); acc[3] = fmaf(x, y0.w, acc[3]);
        acc[4] = fmaf(x, y1.x, acc[4]); acc[5] = fmaf(x, y1.y, acc[5]);
        acc[6] = fmaf(x, y1.z, acc[6]); acc[7] = fmaf(x, y1.w, acc[7]);
    }
}

// Tf[bi][bj] = -Tf[bi][bi] * W, W (in acc) staged through the warp's scratch.
__device__ __forceinline__ void blk_finish(float (&acc)[8], float *Tf, float *wb, int bi, int bj,
                                           int r, int hh) {
    float *w = wb;   // 16 x 20
#pragma unroll
    for (int k = 0; k < 8; ++k) w[r * 20 + 8 * hh + k] = acc[k];
    __syncwarp();
    float out[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
        const float d = Tf[(16 * bi + r) * kLd + 16 * bi + kk];
#pragma unroll
        for (int k = 0; k < 8; ++k) out[k] = fmaf(d, w[kk * 20 + 8 * hh + k], out[k]);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) Tf[(16 * bi + r) * kLd + 16 * bj + 8 * hh + k] = -out[k];
    __syncwarp();
}

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
    if (nch == 0) {   // empty sequence: the initial state (or zero) is the final state
        if (fslot >= 0)
            for (int e = tid; e < DH * DH; e += kThreads)
                pool[(size_t)fslot * hv * DH * DH + head_off + e] =
                    islot >= 0 ? pool[(size_t)islot * hv * DH * DH + head_off + e] : 0.f;
        return;
    }

    if (warp == 1) {
        tmem_alloc(&B.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < kKQStages; ++s) { mbar_init(&B.kq_full[s], 1); mbar_init(&B.kq_empty[s], 1); }
        for (int s = 0; s < kVStages; ++s) { mbar_init(&B.v_full[s], 1); mbar_init(&B.v_empty[s], 128); }
        mbar_init(&B.g_full, 1);
        for (int s = 0; s < 2; ++s) { mbar_init(&B.prep_done[s], 128); mbar_init(&B.d_free[s], 128); }
        mbar_init(&B.x_full, 1);
        mbar_init(&B.r_full, 128);
        mbar_init(&B.u_full, 1);
        mbar_init(&B.u2_full, 128);
        mbar_init(&B.s_full, 1);
        mbar_init(&B.s_next, 128);
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
            const uint32_t id128mn = idesc_bf16(128, 128, false, true);
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
                const int sd = c & 1;
                const uint32_t base = kq_base(c);
                mbar_wait(&B.prep_done[sd], (c >> 1) & 1, abort);
                mbar_wait(&B.s_next, c & 1, abort);
                tc_fence_after();
                for (int s = 0; s < 8; ++s) {   // M2: X = S K^T ; M3: O = S Q'^T
                    const uint32_t off = (s >> 2) * kKBlk + (s & 3) * 32;
                    mma_ts(tbase + kColX, tbase + kColS16 + s * 8, sdesc_sw128(base + off, 16, 1024),
                           id64, s > 0);
                    mma_ts(tbase + kColO, tbase + kColS16 + s * 8,
                           sdesc_sw128(base + 64 * 128 + off, 16, 1024), id64, s > 0);
                }
                mma_commit(&B.x_full);
                if (c + 1 < nch) {
                    mbar_wait(&B.kq_full[(c + 1) % kKQStages], ((c + 1) / kKQStages) & 1, abort);
                    tc_fence_after();
                    issue_g(c + 1);
                }
                mbar_wait(&B.r_full, c & 1, abort);
                tc_fence_after();
                const uint32_t tsm = smem_u32(sm + OFF_T + sd * kTBytes);
                for (int s = 0; s < 4; ++s)   // M4: U = R T^T
                    mma_ts(tbase + kColU, tbase + kColX + s * 8, sdesc_sw128(tsm + s * 32, 16, 1024),
                           id64, s > 0);
                mma_commit(&B.u_full);
                mbar_wait(&B.u2_full, c & 1, abort);
                tc_fence_after();
                const uint32_t psm = smem_u32(sm + OFF_P + sd * kPBytes);
                for (int s = 0; s < 4; ++s) {
                    // M5: O += U P^T ; M6: S += U K''  (K'' MN-major: 2 blocks of 64 keys)
                    mma_ts(tbase + kColO, tbase + kColU + s * 8, sdesc_sw128(psm + s * 32, 16, 1024),
                           id64, 1);
                    mma_ts(tbase + kColS32, tbase + kColU + s * 8,
                           sdesc_sw128(base + s * 16 * 128, kKBlk, 1024), id128mn, 1);
                }
                mma_commit(&B.s_full);
                mma_commit(&B.kq_empty[c % kKQStages]);
            }
            mma_commit(&B.mma_done);
            int z = 0;
            mbar_wait(&B.mma_done, 0, &z);
        }
        __syncwarp();
    } else if (warp < 6) {
        // ---------------------------------------------------- prep (4 warps)
        const int q4 = warp & 3;                 // TMEM lane quadrant
        const int p = q4 * 32 + lane;            // G row: 0..63 K rows, 64..127 Q rows
        const int pw = warp - 2;                 // 0..3 within the group
        for (int c = 0; c < nch; ++c) {
            const int sd = c & 1, sk = c % kKQStages;
            Scal &S = *reinterpret_cast<Scal *>(sm + OFF_SCAL + sd * kScalBytes);
            uint8_t *kq = sm + OFF_KQ + sk * kKQBytes;
            const int64_t c0 = s_start + (int64_t)c * C;
            const int n = (int)min((int64_t)C, s_end - c0);
            if (c >= 2) mbar_wait(&B.d_free[sd], ((c >> 1) - 1) & 1, abort);
            mbar_wait(&B.kq_full[sk], (c / kKQStages) & 1, abort);
            // gating values and the row norms of K (p < 64) / Q (p >= 64)
            if (p < C) {
                S.gam[p] = p < n ? g[(c0 + p) * hv + h] : 0.f;
                S.beta[p] = p < n ? beta[(c0 + p) * hv + h] : 0.f;
            }
            {
                float ss = 0.f;
                const uint32_t row = (uint32_t)p;
                for (int kb = 0; kb < 2; ++kb)
                    for (int ch = 0; ch < 8; ++ch) {
                        const uint4 w = *reinterpret_cast<const uint4 *>(kq + kb * kKBlk + sw128_chunk(row, ch));
                        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = unpack_bf16(ws[e]);
                            ss = fmaf(f.x, f.x, fmaf(f.y, f.y, ss));
                        }
                    }
                const float r = l2norm ? rsqrtf(ss + kEps) : 1.f;
                if (p < C) S.rk[p] = r; else S.rq[p - C] = r;
            }
            named_sync(1, 128);
            if (p < C) {
                float run = 0.f;
                for (int j = 0; j <= p; ++j) run += S.gam[j];
                named_sync(1, 128);      // everyone has read the raw g values
                S.gam[p] = run;
            } else {
                named_sync(1, 128);
            }
            named_sync(1, 128);
            const float gl = S.gam[C - 1];     // padded rows carry g = 0
            if (p < C) {
                const bool ok = p < n;
                S.xs[p] = ok ? expf(S.gam[p]) * S.rk[p] : 0.f;
                S.ks[p] = ok ? expf(gl - S.gam[p]) * S.rk[p] : 0.f;
                if (!ok) S.beta[p] = 0.f;
                if (p == 0) { S.gam_n = expf(gl); S.n = n; }
            }
            // G row -> A (K rows) or P (Q rows)
            mbar_wait(&B.g_full, c & 1, abort);
            tc_fence_after();
            uint32_t graw[64];
            {
                uint32_t t0[32], t1[32];
                tmem_ld32(tmem_addr(tbase, q4 * 32, kColG), t0);
                tmem_ld32(tmem_addr(tbase, q4 * 32, kColG + 32), t1);
#pragma unroll
                for (int j = 0; j < 32; ++j) { graw[j] = t0[j]; graw[32 + j] = t1[j]; }
            }
            tc_fence_before();
            named_sync(1, 128);          // scalars complete
            if (p < C) {
                const int i = p;
                const float bi = S.beta[i], gi = S.gam[i], ri = S.rk[i];
                const bool ok = i < n;
                float *arow = Af + i * kLd;
#pragma unroll
                for (int j = 0; j < C; ++j) {
                    float v = 0.f;
                    if (ok && j < i) v = bi * expf(gi - S.gam[j]) * ri * S.rk[j] * __uint_as_float(graw[j]);
                    arow[j] = v;
                }
            } else {
                const int i = p - C;
                const bool ok = i < n;
                const float gi = S.gam[i], ri = scale * S.rq[i];
                uint8_t *pt = sm + OFF_P + sd * kPBytes;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int j0 = ch * 8 + 2 * e, j1 = j0 + 1;
                        const float v0 = (ok && j0 <= i) ? expf(gi - S.gam[j0]) * ri * S.rk[j0] * __uint_as_float(graw[j0]) : 0.f;
                        const float v1 = (ok && j1 <= i) ? expf(gi - S.gam[j1]) * ri * S.rk[j1] * __uint_as_float(graw[j1]) : 0.f;
                        w[e] = pack_bf16(v0, v1);
                    }
                    *reinterpret_cast<uint4 *>(pt + sw128_chunk(i, ch)) = make_uint4(w[0], w[1], w[2], w[3]);
                }
                // Q' = scale Gam_i r_q,i Q_i, in place (M1 has consumed the raw rows)
                const float f = ok ? expf(gi) * ri : 0.f;
                for (int kb = 0; kb < 2; ++kb)
                    for (int ch = 0; ch < 8; ++ch) {
                        uint4 *pq = reinterpret_cast<uint4 *>(kq + kb * kKBlk + sw128_chunk(C + i, ch));
                        uint4 w = *pq;
                        uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 v = unpack_bf16(ws[e]);
                            ws[e] = pack_bf16(v.x * f, v.y * f);
                        }
                        *pq = make_uint4(ws[0], ws[1], ws[2], ws[3]);
                    }
            }
            named_sync(1, 128);
            // ---- T = (I + A)^-1, blocked 4 x 16: diagonal blocks by forward
            //      substitution (one warp each), then the block rows below.
            {
                const int r = lane >> 1, hh = lane & 1;
                const int bb = pw;                       // diagonal block of this warp
                const int R = 16 * bb + r;
                float t[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) t[k] = (8 * hh + k == r) ? 1.f : 0.f;
                for (int m = 0; m < 15; ++m) {
                    const float a = Af[R * kLd + 16 * bb + m];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float vm = __shfl_sync(0xffffffffu, t[k], 2 * m + hh);
                        if (r > m) t[k] = fmaf(-a, vm, t[k]);
                    }
                }
#pragma unroll
                for (int k = 0; k < 8; ++k) Tf[R * kLd + 16 * bb + 8 * hh + k] = t[k];
                named_sync(1, 128);
                float *wb = Wb + pw * 16 * 20;
                float acc[8];
                // level 1: T10, T21, T32
                if (pw < 3) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) acc[k] = 0.f;
                    blk_mac(acc, Af, 16 * (pw + 1), 16 * pw, Tf, 16 * pw, 16 * pw, r, hh);
                    blk_finish(acc, Tf, wb, pw + 1, pw, r, hh);
                }
                named_sync(1, 128);
                // level 2: T20, T31 and the partial sum Z30 = A30 T00 + A31 T10
                if (pw < 3) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) acc[k] = 0.f;
                    if (pw == 0) {
                        blk_mac(acc, Af, 32, 0, Tf, 0, 0, r, hh);
                        blk_mac(acc, Af, 32, 16, Tf, 16, 0, r, hh);
                        blk_finish(acc, Tf, wb, 2, 0, r, hh);
                    } else if (pw == 1) {
                        blk_mac(acc, Af, 48, 16, Tf, 16, 16, r, hh);
                        blk_mac(acc, Af, 48, 32, Tf, 32, 16, r, hh);
                        blk_finish(acc, Tf, wb, 3, 1, r, hh);
                    } else {
                        blk_mac(acc, Af, 48, 0, Tf, 0, 0, r, hh);
                        blk_mac(acc, Af, 48, 16, Tf, 16, 0, r, hh);
#pragma unroll
                        for (int k = 0; k < 8; ++k) Wb[3 * 16 * 20 + r * 20 + 8 * hh + k] = acc[k];
                    }
                }
                named_sync(1, 128);
                // level 3: T30 = -T33 (Z30 + A32 T20)
                if (pw == 0) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) acc[k] = Wb[3 * 16 * 20 + r * 20 + 8 * hh + k];
                    blk_mac(acc, Af, 48, 32, Tf, 32, 0, r, hh);
                    blk_finish(acc, Tf, wb, 3, 0, r, hh);
                }
                named_sync(1, 128);
            }
            // T (lower triangular) -> bf16, K-major [i][j]
            {
                const int i = p >> 1, half = p & 1;
                uint8_t *tt = sm + OFF_T + sd * kTBytes;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int ch = half * 4 + cc;
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int j0 = ch * 8 + 2 * e;
                        const float v0 = j0 <= i ? Tf[i * kLd + j0] : 0.f;
                        const float v1 = j0 + 1 <= i ? Tf[i * kLd + j0 + 1] : 0.f;
                        w[e] = pack_bf16(v0, v1);
                    }
                    *reinterpret_cast<uint4 *>(tt + sw128_chunk(i, ch)) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            fence_async_smem();
            mbar_arrive(&B.prep_done[sd]);
            named_sync(1, 128);          // the solve scratch is free again
        }
    } else {
        // --------------------------------------------------- chain (4 warps)
        const int q4 = warp & 3;
        const int b = q4 * 32 + lane;            // value row of the state
        const uint32_t lrow = tmem_addr(tbase, q4 * 32, 0);
        // E0: initial state -> fp32 accumulator + bf16 operand copy
        {
            const float *src = islot >= 0 ? pool + (size_t)islot * hv * DH * DH + head_off + (size_t)b * DH : nullptr;
            for (int c0 = 0; c0 < DH; c0 += 32) {
                uint32_t r[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(src ? src[c0 + j] : 0.f);
                tmem_st32(lrow + kColS32 + c0, r);
            }
            for (int c0 = 0; c0 < DH; c0 += 64) {
                uint32_t r[32];
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    r[j] = pack_bf16(src ? src[c0 + 2 * j] : 0.f, src ? src[c0 + 2 * j + 1] : 0.f);
                tmem_st32(lrow + kColS16 + c0 / 2, r);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&B.s_next);
        }
        for (int c = 0; c < nch; ++c) {
            const int sd = c & 1, sk = c % kKQStages, sv = c % kVStages;
            const Scal &S = *reinterpret_cast<const Scal *>(sm + OFF_SCAL + sd * kScalBytes);
            uint8_t *kq = sm + OFF_KQ + sk * kKQBytes;
            const uint8_t *vt = sm + OFF_V + sv * kVBytes;
            const int64_t c0 = s_start + (int64_t)c * C;
            mbar_wait(&B.prep_done[sd], (c >> 1) & 1, abort);
            const int n = S.n;
            // ---- E1: R = beta (V - Gam r_k X) -> bf16 in TMEM (X's columns)
            mbar_wait(&B.x_full, c & 1, abort);
            tc_fence_after();
            mbar_wait(&B.v_full[sv], (c / kVStages) & 1, abort);
            {
                uint32_t x0[32], x1[32];
                tmem_ld32(lrow + kColX, x0);
                tmem_ld32(lrow + kColX + 32, x1);
                const uint8_t *vcol = vt + (b >> 6) * kVBlk;
                const uint32_t be = (uint32_t)(b & 63);
                uint32_t rr[32];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    float v2[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int j = 2 * jj + e;
                        const float x = __uint_as_float(j < 32 ? x0[j] : x1[j - 32]);
                        const float vv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(vcol + sw128_off((uint32_t)j, be)));
                        v2[e] = j < n ? S.beta[j] * (vv - S.xs[j] * x) : 0.f;
                    }
                    rr[jj] = pack_bf16(v2[0], v2[1]);
                }
                tmem_st32(lrow + kColX, rr);
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(&B.r_full);
            mbar_arrive(&B.v_empty[sv]);
            // K'' = D[last][j] r_k,j K_j in place (M1, M2 have consumed the raw rows)
            {
                const int j = tid - 192 >= 0 ? ((tid - 192) >> 1) : 0;
                const int kb = (tid - 192) & 1;
                const float f = S.ks[j];
                for (int ch = 0; ch < 8; ++ch) {
                    uint4 *pk = reinterpret_cast<uint4 *>(kq + kb * kKBlk + sw128_chunk((uint32_t)j, ch));
                    uint4 w = *pk;
                    uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 v = unpack_bf16(ws[e]);
                        ws[e] = pack_bf16(v.x * f, v.y * f);
                    }
                    *pk = make_uint4(ws[0], ws[1], ws[2], ws[3]);
                }
                fence_async_smem();
            }
            // S <- Gam_last S ahead of M6
            {
                const float gn = S.gam_n;
                for (int cc = 0; cc < DH; cc += 32) {
                    uint32_t r[32];
                    tmem_ld32(lrow + kColS32 + cc, r);
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * gn);
                    tmem_st32(lrow + kColS32 + cc, r);
                }
                tmem_wait_st();
            }
            // ---- E2: U -> bf16 in TMEM (U's columns)
            mbar_wait(&B.u_full, c & 1, abort);
            tc_fence_after();
            {
                uint32_t u0[32], u1[32], uu[32];
                tmem_ld32(lrow + kColU, u0);
                tmem_ld32(lrow + kColU + 32, u1);
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    uu[jj] = pack_bf16(__uint_as_float(u0[2 * jj]), __uint_as_float(u0[2 * jj + 1]));
                    uu[16 + jj] = pack_bf16(__uint_as_float(u1[2 * jj]), __uint_as_float(u1[2 * jj + 1]));
                }
                tmem_st32(lrow + kColU, uu);
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(&B.u2_full);
            // ---- E3: o <- O ; S -> bf16 copy ; final state
            mbar_wait(&B.s_full, c & 1, abort);
            tc_fence_after();
            {
                uint32_t o0[32], o1[32];
                tmem_ld32(lrow + kColO, o0);
                tmem_ld32(lrow + kColO + 32, o1);
                __nv_bfloat16 *orow = o + (c0 * hv + h) * (int64_t)DH + b;
                const int64_t ostride = (int64_t)hv * DH;
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (i < n) orow[i * ostride] = __float2bfloat16_rn(__uint_as_float(o0[i]));
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (32 + i < n) orow[(32 + i) * ostride] = __float2bfloat16_rn(__uint_as_float(o1[i]));
            }
            const bool last = c == nch - 1;
            float *dst = (last && fslot >= 0) ? pool + (size_t)fslot * hv * DH * DH + head_off + (size_t)b * DH : nullptr;
            for (int cc = 0; cc < DH; cc += 64) {
                uint32_t s0[32], s1[32], pk[32];
                tmem_ld32(lrow + kColS32 + cc, s0);
                tmem_ld32(lrow + kColS32 + cc + 32, s1);
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    pk[jj] = pack_bf16(__uint_as_float(s0[2 * jj]), __uint_as_float(s0[2 * jj + 1]));
                    pk[16 + jj] = pack_bf16(__uint_as_float(s1[2 * jj]), __uint_as_float(s1[2 * jj + 1]));
                }
                if (!last) tmem_st32(lrow + kColS16 + cc / 2, pk);
                if (dst) {
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        *reinterpret_cast<float4 *>(dst + cc + j) = make_float4(
                            __uint_as_float(s0[j]), __uint_as_float(s0[j + 1]),
                            __uint_as_float(s0[j + 2]), __uint_as_float(s0[j + 3]));
                        *reinterpret_cast<float4 *>(dst + cc + 32 + j) = make_float4(
                            __uint_as_float(s1[j]), __uint_as_float(s1[j + 1]),
                            __uint_as_float(s1[j + 2]), __uint_as_float(s1[j + 3]));
                    }
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&B.s_next);
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
