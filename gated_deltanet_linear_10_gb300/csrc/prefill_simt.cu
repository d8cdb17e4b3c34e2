// Chunked varlen prefill of the gated delta rule in WY/UT form, fp32 SIMT
// ("Flash Linear Attention operations for efficient chunked computations",
// "[model] Support Qwen3next", Highlights).  This is the generic kernel: any
// dk = dv in {16, 32, 64, 128}, chunk in {16, 32, 64}, fp32 or bf16
// activations, all arithmetic in fp32.  (The bf16 dk = 128 / chunk 64 case
// has a tensor-core kernel of its own.)
//
// One CTA per (sequence, V head, 32-wide slice of dv): rows of S evolve
// independently, so slices of dv are independent chains.  Per chunk of C
// tokens, with S0 the incoming state slice [BV][dk] and, inside the chunk,
// gc = prefix sum of g, Gam = exp(gc), D[i][j] = exp(gc_i - gc_j) (j <= i):
//   A  = strictly-lower beta_i D_ij (k_i . k_j)      T = (I + A)^-1
//   R  = diag(beta) (V - diag(Gam) K S0^T)            U = T R
//   O  = scale (diag(Gam) Q S0^T + (D .* Q K^T) U)
//   S  = Gam_last S0 + U^T diag(D[last][.]) K
// A partial last chunk is padded with k = q = v = 0, beta = g = 0, which
// leaves every product above unchanged for the real rows.
#include "common.cuh"

namespace gdn {

GDN_DECLARE_STATUS_WORD(g_status_prefill_simt)
GDN_STATUS_READER(read_status_prefill_simt, g_status_prefill_simt)

constexpr int kSimtThreads = 256;
constexpr float kPrefillL2Eps = 1e-6f;

template <int DK, int CH>
struct SimtSmem {
    static constexpr int BV = DK < 32 ? DK : 32;
    static constexpr int LK = DK + 1;    // padded row strides (bank-conflict free columns)
    static constexpr int LV = BV + 1;
    static constexpr int LC = CH + 1;
    static constexpr int floats = 2 * CH * LK + 2 * CH * LV + 2 * CH * LC + BV * LK + 2 * CH + 8;
    static constexpr size_t bytes = (size_t)floats * sizeof(float);
};

// Rank of sequence `which` in decreasing-length order (ties by index), so
// that the longest chains start first.  Computed redundantly per CTA.
__device__ int seq_of_rank(const int32_t *cu, int n_seqs, int rank, int *s_seq) {
    if (n_seqs > 1024) return rank;   // large batches: keep launch order
    if (threadIdx.x == 0) *s_seq = -1;
    __syncthreads();
    for (int i = threadIdx.x; i < n_seqs; i += blockDim.x) {
        const int li = cu[i + 1] - cu[i];
        int r = 0;
        for (int j = 0; j < n_seqs; ++j) {
            const int lj = cu[j + 1] - cu[j];
            r += (lj > li) || (lj == li && j < i);
        }
        if (r == rank) *s_seq = i;
    }
    __syncthreads();
    const int s = *s_seq;
    return s < 0 ? rank : s;
}

template <int DK, int CH, typename T>
__global__ void __launch_bounds__(kSimtThreads)
prefill_simt_kernel(const T *__restrict__ q, int64_t qs, const T *__restrict__ k, int64_t ks,
                    const T *__restrict__ v, int64_t vs, const float *__restrict__ g,
                    const float *__restrict__ beta, const int32_t *__restrict__ cu, int n_seqs,
                    int64_t n_tokens, int hv, int grp, float scale, int l2norm,
                    float *__restrict__ pool, int64_t n_slots,
                    const int32_t *__restrict__ init_idx, const int32_t *__restrict__ final_idx,
                    T *__restrict__ o) {
    using L = SimtSmem<DK, CH>;
    constexpr int BV = L::BV, LK = L::LK, LV = L::LV, LC = L::LC;
    constexpr int DV = DK;
    constexpr int NT = kSimtThreads;
    constexpr int tiles = DV / BV;

    extern __shared__ float sm[];
    float *Kn = sm;                 // [CH][LK]
    float *Qn = Kn + CH * LK;       // [CH][LK]
    float *Vb = Qn + CH * LK;       // [CH][LV]  V, then R
    float *Ub = Vb + CH * LV;       // [CH][LV]
    float *Tm = Ub + CH * LV;       // [CH][LC]
    float *Am = Tm + CH * LC;       // [CH][LC]  A, then D .* Q K^T
    float *S = Am + CH * LC;        // [BV][LK]
    float *gc = S + BV * LK;        // [CH]
    float *bt = gc + CH;            // [CH]
    int *misc = reinterpret_cast<int *>(bt + CH);

    const int tid = threadIdx.x;
    const int per_seq = hv * tiles;
    const int rank = blockIdx.x / per_seq;
    const int rem = blockIdx.x - rank * per_seq;
    const int h = rem / tiles;
    const int b0 = (rem - h * tiles) * BV;
    const int hq = h / grp;
    const int seq = seq_of_rank(cu, n_seqs, rank, misc);

    const int64_t s_start = cu[seq], s_end = cu[seq + 1];
    if (s_start < 0 || s_end < s_start || s_end > n_tokens) {
        if (tid == 0) flag_status(GDN_DEVSTAT_BAD_SEQLEN);
        return;
    }
    int64_t islot = init_idx ? init_idx[seq] : -1;
    int64_t fslot = final_idx ? final_idx[seq] : -1;
    if (islot >= n_slots || fslot >= n_slots) {
        if (tid == 0) flag_status(GDN_DEVSTAT_BAD_INDEX);
        if (islot >= n_slots) islot = -1;
        if (fslot >= n_slots) fslot = -1;
    }

    // initial state slice
    for (int e = tid; e < BV * DK; e += NT) {
        const int b = e / DK, a = e - b * DK;
        S[b * LK + a] = islot >= 0 ? pool[((islot * hv + h) * DV + b0 + b) * (int64_t)DK + a] : 0.f;
    }

    for (int64_t c0 = s_start; c0 < s_end; c0 += CH) {
        const int n = (int)min((int64_t)CH, s_end - c0);
        // ---- 1. load the chunk (zero-padded past n)
        for (int e = tid; e < CH * DK; e += NT) {
            const int i = e / DK, a = e - i * DK;
            float kv = 0.f, qv = 0.f;
            if (i < n) {
                kv = Io<T>::load(k + (c0 + i) * ks + (int64_t)hq * DK + a);
                qv = Io<T>::load(q + (c0 + i) * qs + (int64_t)hq * DK + a);
            }
            Kn[i * LK + a] = kv;
            Qn[i * LK + a] = qv;
        }
        for (int e = tid; e < CH * BV; e += NT) {
            const int i = e / BV, b = e - i * BV;
            Vb[i * LV + b] = i < n ? Io<T>::load(v + (c0 + i) * vs + (int64_t)h * DV + b0 + b) : 0.f;
        }
        if (tid < CH) {
            gc[tid] = tid < n ? g[(c0 + tid) * hv + h] : 0.f;
            bt[tid] = tid < n ? beta[(c0 + tid) * hv + h] : 0.f;
        }
        __syncthreads();
        // ---- 2. L2-normalise q, k rows (one warp per row); prefix-sum g
        if (l2norm) {
            const int warp = tid >> 5, lane = tid & 31;
            for (int i = warp; i < 2 * CH; i += NT / 32) {
                float *row = i < CH ? Kn + i * LK : Qn + (i - CH) * LK;
                float ss = 0.f;
                for (int a = lane; a < DK; a += 32) ss += row[a] * row[a];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                const float inv = rsqrtf(ss + kPrefillL2Eps);
                for (int a = lane; a < DK; a += 32) row[a] *= inv;
            }
        }
        if (tid == 0) {
            float run = 0.f;
            for (int i = 0; i < CH; ++i) {
                run += gc[i];
                gc[i] = run;
            }
        }
        __syncthreads();
        // ---- 3. A (strictly lower) and T = I
        for (int e = tid; e < CH * CH; e += NT) {
            const int i = e / CH, j = e - i * CH;
            float val = 0.f;
            if (j < i) {
                float acc = 0.f;
                for (int a = 0; a < DK; ++a) acc = fmaf(Kn[i * LK + a], Kn[j * LK + a], acc);
                val = bt[i] * expf(gc[i] - gc[j]) * acc;
            }
            Am[i * LC + j] = val;
            Tm[i * LC + j] = (i == j) ? 1.f : 0.f;
        }
        __syncthreads();
        // ---- 4. T = (I + A)^-1: after step m row m is final; rows i > m take
        //         T[i][:] -= A[i][m] T[m][:] (T[m] is nonzero on columns <= m).
        for (int m = 0; m < CH - 1; ++m) {
            const int rows = CH - 1 - m, cols = m + 1;
            for (int e = tid; e < rows * cols; e += NT) {
                const int i = m + 1 + e / cols, c = e % cols;
                Tm[i * LC + c] -= Am[i * LC + m] * Tm[m * LC + c];
            }
            __syncthreads();
        }
        // ---- 5. P = D .* (Q K^T) (into Am) and R = diag(beta)(V - diag(Gam) K S0^T)
        for (int e = tid; e < CH * CH; e += NT) {
            const int i = e / CH, j = e - i * CH;
            float val = 0.f;
            if (j <= i) {
                float acc = 0.f;
                for (int a = 0; a < DK; ++a) acc = fmaf(Qn[i * LK + a], Kn[j * LK + a], acc);
                val = expf(gc[i] - gc[j]) * acc;
            }
            Am[i * LC + j] = val;
        }
        for (int e = tid; e < CH * BV; e += NT) {
            const int j = e / BV, b = e - j * BV;
            float acc = 0.f;
            for (int a = 0; a < DK; ++a) acc = fmaf(Kn[j * LK + a], S[b * LK + a], acc);
            Vb[j * LV + b] = bt[j] * (Vb[j * LV + b] - expf(gc[j]) * acc);
        }
        __syncthreads();
        // ---- 6. U = T R
        for (int e = tid; e < CH * BV; e += NT) {
            const int i = e / BV, b = e - i * BV;
            float acc = 0.f;
            for (int j = 0; j <= i; ++j) acc = fmaf(Tm[i * LC + j], Vb[j * LV + b], acc);
            Ub[i * LV + b] = acc;
        }
        __syncthreads();
        // ---- 7. O = scale (diag(Gam) Q S0^T + P U)
        for (int e = tid; e < CH * BV; e += NT) {
            const int i = e / BV, b = e - i * BV;
            if (i < n) {
                float qs0 = 0.f;
                for (int a = 0; a < DK; ++a) qs0 = fmaf(Qn[i * LK + a], S[b * LK + a], qs0);
                float acc = expf(gc[i]) * qs0;
                for (int j = 0; j <= i; ++j) acc = fmaf(Am[i * LC + j], Ub[j * LV + b], acc);
                Io<T>::store(o + ((c0 + i) * hv + h) * (int64_t)DV + b0 + b, scale * acc);
            }
        }
        __syncthreads();
        // ---- 8. S = Gam_last S0 + U^T diag(D[last][.]) K
        {
            const float glast = gc[CH - 1];
            for (int e = tid; e < BV * DK; e += NT) {
                const int b = e / DK, a = e - b * DK;
                float acc = expf(glast) * S[b * LK + a];
                for (int j = 0; j < CH; ++j)
                    acc = fmaf(Ub[j * LV + b] * expf(glast - gc[j]), Kn[j * LK + a], acc);
                S[b * LK + a] = acc;
            }
        }
        __syncthreads();
    }

    if (fslot >= 0)
        for (int e = tid; e < BV * DK; e += NT) {
            const int b = e / DK, a = e - b * DK;
            pool[((fslot * hv + h) * DV + b0 + b) * (int64_t)DK + a] = S[b * LK + a];
        }
}

template <int DK, int CH, typename T>
static gdn_status launch_simt(const void *q, int64_t qs, const void *k, int64_t ks, const void *v,
                              int64_t vs, const float *g, const float *beta, const int32_t *cu,
                              int n_seqs, int64_t n_tokens, int hqk, int hv, float scale,
                              int l2norm, float *pool, int64_t n_slots, const int32_t *ii,
                              const int32_t *fi, void *o, cudaStream_t s) {
    using L = SimtSmem<DK, CH>;
    auto kern = prefill_simt_kernel<DK, CH, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)L::bytes);
    if (e != cudaSuccess) {
        set_last_cuda_error(e);
        return GDN_ERR_LAUNCH;
    }
    const int64_t blocks = (int64_t)n_seqs * hv * (DK / L::BV);
    kern<<<(unsigned)blocks, kSimtThreads, L::bytes, s>>>(
        (const T *)q, qs, (const T *)k, ks, (const T *)v, vs, g, beta, cu, n_seqs, n_tokens, hv,
        hv / hqk, scale, l2norm, pool, n_slots, ii, fi, (T *)o);
    return launch_status();
}

template <typename T>
static gdn_status dispatch_simt(int dk, int chunk, const void *q, int64_t qs, const void *k,
                                int64_t ks, const void *v, int64_t vs, const float *g,
                                const float *beta, const int32_t *cu, int n_seqs,
                                int64_t n_tokens, int hqk, int hv, float scale, int l2norm,
                                float *pool, int64_t n_slots, const int32_t *ii,
                                const int32_t *fi, void *o, cudaStream_t s) {
#define GDN_SIMT(DK, CH)                                                                   \
    if (dk == DK && chunk == CH)                                                           \
        return launch_simt<DK, CH, T>(q, qs, k, ks, v, vs, g, beta, cu, n_seqs, n_tokens, hqk, \
                                      hv, scale, l2norm, pool, n_slots, ii, fi, o, s);
    GDN_SIMT(16, 16) GDN_SIMT(16, 32) GDN_SIMT(16, 64)
    GDN_SIMT(32, 16) GDN_SIMT(32, 32) GDN_SIMT(32, 64)
    GDN_SIMT(64, 16) GDN_SIMT(64, 32) GDN_SIMT(64, 64)
    GDN_SIMT(128, 16) GDN_SIMT(128, 32) GDN_SIMT(128, 64)
#undef GDN_SIMT
    return GDN_ERR_UNSUPPORTED;
}

gdn_status prefill_simt(int dtype, int dk, int chunk, const void *q, int64_t qs, const void *k,
                        int64_t ks, const void *v, int64_t vs, const float *g, const float *beta,
                        const int32_t *cu, int n_seqs, int64_t n_tokens, int hqk, int hv,
                        float scale, int l2norm, float *pool, int64_t n_slots, const int32_t *ii,
                        const int32_t *fi, void *o, cudaStream_t s) {
    if (dtype == GDN_F32)
        return dispatch_simt<float>(dk, chunk, q, qs, k, ks, v, vs, g, beta, cu, n_seqs, n_tokens,
                                    hqk, hv, scale, l2norm, pool, n_slots, ii, fi, o, s);
    return dispatch_simt<__nv_bfloat16>(dk, chunk, q, qs, k, ks, v, vs, g, beta, cu, n_seqs,
                                        n_tokens, hqk, hv, scale, l2norm, pool, n_slots, ii, fi,
                                        o, s);
}

}  // namespace gdn
