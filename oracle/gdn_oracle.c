/*
 * Gated DeltaNet (GDN) layer — CPU oracle, fp64.  TEST INFRASTRUCTURE ONLY.
 *
 * This file is the plain, slow, obviously correct definition that the CUDA
 * path is checked against.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load it; the library's own path never
 * does, and this file shares no code, header or constant with the CUDA
 * sources.
 *
 * What the method computes.  The pages describing the layer are the LightLLM
 * pull request "[model] support Qwen3next" (Highlights: causal 1D
 * convolutions, fused recurrent GDN, fused gating), the LightLLM issue
 * "[model] Support Qwen3next" (Highlights: causal 1D convolution, fused GDN
 * gating, chunked and recurrent linear-attention operations) and the lmdeploy
 * issue "[Feature] Qwen3-Next-80B-A3B Support" (New attention kernels: 16 QK
 * heads, 32 V heads, head_dim 128).  They name the operations but print no
 * formula.  The reading taken here is the standard gated delta rule:
 *
 *   g_t   = -exp(A_log[h]) * softplus(a_t + dt_bias[h])        (gating)
 *   beta_t = sigmoid(b_t)
 *   y     = SiLU(bias + sum_w W[c][w] * x[t-(W-1)+w][c])       (causal conv)
 *   S_t   = exp(g_t) * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *   o_t   = scale * S_t q_t      with q, k L2-normalised per head.
 *
 * S is dv x dk (row = value index).  Every function below is single-threaded
 * and loops in the order the formula reads.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

/* softplus(x) = log(1 + e^x), written so that e^x never overflows. */
static double softplus(double x)
{
    if (x > 0.0)
        return x + log1p(exp(-x));
    return log1p(exp(x));
}

/* sigmoid(x) = 1 / (1 + e^-x), written so that e^-x never overflows. */
static double sigmoid(double x)
{
    if (x >= 0.0)
        return 1.0 / (1.0 + exp(-x));
    double e = exp(x);
    return e / (1.0 + e);
}

static double silu(double z) { return z * sigmoid(z); }

/*
 * Fused gating ("fused GDN gating", Qwen3next pages, Highlights).
 * a, b: [n_tokens][hv]; A_log, dt_bias: [hv]; g, beta: [n_tokens][hv].
 */
void oracle_gating(const double *a, const double *b, const double *A_log,
                   const double *dt_bias, long n_tokens, int hv, double *g,
                   double *beta)
{
    for (long t = 0; t < n_tokens; ++t)
        for (int h = 0; h < hv; ++h) {
            long i = t * hv + h;
            g[i] = -exp(A_log[h]) * softplus(a[i] + dt_bias[h]);
            beta[i] = sigmoid(b[i]);
        }
}

/*
 * Causal depthwise conv1d over one sequence ("causal 1D convolutions",
 * Qwen3next pages, Highlights).
 *
 * x: [T][C] (contiguous), weight: [C][W] (tap W-1 multiplies the current
 * token), bias: [C] or NULL, hist: [(W-1)][C] inputs that precede the
 * sequence, oldest first, or NULL for zeros.  y: [T][C].
 * state_out: [(W-1)][C] = the last W-1 pre-activation inputs of the extended
 * sequence hist ++ x, oldest first (may alias hist).
 */
void oracle_conv1d_seq(const double *x, long T, int C, int W,
                       const double *weight, const double *bias,
                       const double *hist, int apply_silu, double *y,
                       double *state_out)
{
    const int H = W - 1;
    /* Extended input e[n], n in [-H, T): e[n] = hist[H + n] for n < 0. */
    double *ext = (double *)calloc((size_t)(T + H) * C, sizeof(double));
    if (hist)
        memcpy(ext, hist, (size_t)H * C * sizeof(double));
    memcpy(ext + (size_t)H * C, x, (size_t)T * C * sizeof(double));

    for (long t = 0; t < T; ++t)
        for (int c = 0; c < C; ++c) {
            double acc = bias ? bias[c] : 0.0;
            for (int w = 0; w < W; ++w) {
                long n = t - H + w;              /* index into e[] */
                acc += weight[c * W + w] * ext[(size_t)(n + H) * C + c];
            }
            y[t * C + c] = apply_silu ? silu(acc) : acc;
        }

    if (state_out)
        for (int r = 0; r < H; ++r) {
            long n = T - H + r;
            for (int c = 0; c < C; ++c)
                state_out[r * C + c] = ext[(size_t)(n + H) * C + c];
        }
    free(ext);
}

/* x_hat = x / sqrt(sum x^2 + eps), row by row.  x, out: [n][d]. */
void oracle_l2norm(const double *x, long n, int d, double eps, double *out)
{
    for (long i = 0; i < n; ++i) {
        double ss = 0.0;
        for (int j = 0; j < d; ++j)
            ss += x[i * d + j] * x[i * d + j];
        double inv = 1.0 / sqrt(ss + eps);
        for (int j = 0; j < d; ++j)
            out[i * d + j] = x[i * d + j] * inv;
    }
}

/*
 * Token-by-token gated delta rule for one (sequence, V head) chain
 * ("fused recurrent GDN", Qwen3next pages, Highlights).
 *
 * q, k: [T][dk]; v: [T][dv]; g, beta: [T].  S: [dv][dk], in: initial state,
 * out: final state.  o: [T][dv].  snaps: NULL or [T][dv][dk], the state
 * after each token.  If l2norm, q and k are normalised first.
 *
 * One token, with alpha = exp(g):
 *   S <- alpha S (I - beta k k^T) + beta v k^T
 *      = alpha S + u k^T,   u = beta (v - alpha S k)        (same algebra)
 *   o  = scale * S q        (the updated S)
 */
void oracle_gdn_recurrent(const double *q, const double *k, const double *v,
                          const double *g, const double *beta, long T, int dk,
                          int dv, double scale, int l2norm, double eps,
                          double *S, double *o, double *snaps)
{
    double *qh = (double *)malloc(sizeof(double) * dk);
    double *kh = (double *)malloc(sizeof(double) * dk);
    double *u = (double *)malloc(sizeof(double) * dv);
    for (long t = 0; t < T; ++t) {
        if (l2norm) {
            oracle_l2norm(q + t * dk, 1, dk, eps, qh);
            oracle_l2norm(k + t * dk, 1, dk, eps, kh);
        } else {
            memcpy(qh, q + t * dk, sizeof(double) * dk);
            memcpy(kh, k + t * dk, sizeof(double) * dk);
        }
        double alpha = exp(g[t]);
        double bt = beta[t];
        for (int i = 0; i < dv; ++i) {
            double sk = 0.0;
            for (int j = 0; j < dk; ++j)
                sk += S[i * dk + j] * kh[j];
            u[i] = bt * (v[t * dv + i] - alpha * sk);
        }
        for (int i = 0; i < dv; ++i)
            for (int j = 0; j < dk; ++j)
                S[i * dk + j] = alpha * S[i * dk + j] + u[i] * kh[j];
        for (int i = 0; i < dv; ++i) {
            double acc = 0.0;
            for (int j = 0; j < dk; ++j)
                acc += S[i * dk + j] * qh[j];
            o[t * dv + i] = scale * acc;
        }
        if (snaps)
            memcpy(snaps + (size_t)t * dv * dk, S, sizeof(double) * dv * dk);
    }
    free(qh);
    free(kh);
    free(u);
}

/*
 * UT transform of one chunk of n tokens (the WY/UT form of the chunked gated
 * delta rule).  kn: [n][dk] normalised keys; beta, gcum: [n] with gcum the
 * within-chunk prefix sum of g.  Builds the strictly lower-triangular
 *   A[j][m] = beta_j * exp(gcum_j - gcum_m) * (k_j . k_m),   m < j,
 * and returns Tm = (I + A)^-1 ([n][n], row-major) by forward substitution,
 * row by row: Tm[i] = e_i - sum_{m<i} A[i][m] Tm[m].
 */
void oracle_ut_transform(const double *kn, const double *beta,
                         const double *gcum, int n, int dk, double *Tm)
{
    double *A = (double *)calloc((size_t)n * n, sizeof(double));
    for (int j = 0; j < n; ++j)
        for (int m = 0; m < j; ++m) {
            double kk = 0.0;
            for (int a = 0; a < dk; ++a)
                kk += kn[j * dk + a] * kn[m * dk + a];
            A[j * n + m] = beta[j] * exp(gcum[j] - gcum[m]) * kk;
        }
    for (int i = 0; i < n; ++i) {
        for (int c = 0; c < n; ++c)
            Tm[i * n + c] = (i == c) ? 1.0 : 0.0;
        for (int m = 0; m < i; ++m) {
            double aim = A[i * n + m];
            for (int c = 0; c < n; ++c)
                Tm[i * n + c] -= aim * Tm[m * n + c];
        }
    }
    free(A);
}

/*
 * Chunked (WY/UT) form of the same recurrence for one chain ("Flash Linear
 * Attention operations for efficient chunked computations", Qwen3next issue,
 * Highlights).  Same arguments as oracle_gdn_recurrent plus the chunk length.
 * Chunks restart at the sequence start; the last one may be partial.  Per
 * chunk of n tokens, with S0 the incoming state and gcum, Gam = exp(gcum)
 * within the chunk, D[i][j] = exp(gcum_i - gcum_j) for j <= i (else 0):
 *   Tm = (I + A)^-1                      (oracle_ut_transform)
 *   W  = Tm diag(beta Gam) K             [n][dk]
 *   U  = Tm diag(beta) V - W S0^T        [n][dv]
 *   O  = scale (diag(Gam) Q S0^T + (D .* Q K^T) U)
 *   S  = Gam_n S0 + U^T diag(D[n-1][.]) K
 * It exists only to be checked against the token form.
 */
void oracle_gdn_chunked(const double *q, const double *k, const double *v,
                        const double *g, const double *beta, long T, int dk,
                        int dv, double scale, int l2norm, double eps,
                        int chunk, double *S, double *o)
{
    double *Q = (double *)malloc(sizeof(double) * chunk * dk);
    double *K = (double *)malloc(sizeof(double) * chunk * dk);
    double *gc = (double *)malloc(sizeof(double) * chunk);
    double *Tm = (double *)malloc(sizeof(double) * chunk * chunk);
    double *Wm = (double *)malloc(sizeof(double) * chunk * dk);
    double *U = (double *)malloc(sizeof(double) * chunk * dv);
    double *Snew = (double *)malloc(sizeof(double) * dv * dk);

    for (long s = 0; s < T; s += chunk) {
        int n = (int)((T - s) < chunk ? (T - s) : chunk);
        if (l2norm) {
            oracle_l2norm(q + s * dk, n, dk, eps, Q);
            oracle_l2norm(k + s * dk, n, dk, eps, K);
        } else {
            memcpy(Q, q + s * dk, sizeof(double) * n * dk);
            memcpy(K, k + s * dk, sizeof(double) * n * dk);
        }
        const double *V = v + s * dv;
        const double *B = beta + s;
        double run = 0.0;
        for (int i = 0; i < n; ++i) {
            run += g[s + i];
            gc[i] = run;
        }
        oracle_ut_transform(K, B, gc, n, dk, Tm);

        /* W = Tm diag(beta Gam) K */
        for (int i = 0; i < n; ++i)
            for (int a = 0; a < dk; ++a) {
                double acc = 0.0;
                for (int j = 0; j < n; ++j)
                    acc += Tm[i * n + j] * B[j] * exp(gc[j]) * K[j * dk + a];
                Wm[i * dk + a] = acc;
            }
        /* U = Tm diag(beta) V - W S0^T */
        for (int i = 0; i < n; ++i)
            for (int c = 0; c < dv; ++c) {
                double acc = 0.0;
                for (int j = 0; j < n; ++j)
                    acc += Tm[i * n + j] * B[j] * V[j * dv + c];
                double ws = 0.0;
                for (int a = 0; a < dk; ++a)
                    ws += Wm[i * dk + a] * S[c * dk + a];
                U[i * dv + c] = acc - ws;
            }
        /* O = scale (diag(Gam) Q S0^T + (D .* Q K^T) U) */
        for (int i = 0; i < n; ++i)
            for (int c = 0; c < dv; ++c) {
                double qs = 0.0;
                for (int a = 0; a < dk; ++a)
                    qs += Q[i * dk + a] * S[c * dk + a];
                double acc = exp(gc[i]) * qs;
                for (int j = 0; j <= i; ++j) {
                    double qk = 0.0;
                    for (int a = 0; a < dk; ++a)
                        qk += Q[i * dk + a] * K[j * dk + a];
                    acc += exp(gc[i] - gc[j]) * qk * U[j * dv + c];
                }
                o[(s + i) * dv + c] = scale * acc;
            }
        /* S = Gam_n S0 + U^T diag(D[n-1][.]) K */
        for (int c = 0; c < dv; ++c)
            for (int a = 0; a < dk; ++a) {
                double acc = exp(gc[n - 1]) * S[c * dk + a];
                for (int j = 0; j < n; ++j)
                    acc += U[j * dv + c] * exp(gc[n - 1] - gc[j]) * K[j * dk + a];
                Snew[c * dk + a] = acc;
            }
        memcpy(S, Snew, sizeof(double) * dv * dk);
    }
    free(Q);
    free(K);
    free(gc);
    free(Tm);
    free(Wm);
    free(U);
    free(Snew);
}

/*
 * Gated RMSNorm of the layer output ("gated RMSNorm", "[model] Support
 * Qwen3next", LightLLM issue 1097, Highlights; the page names the kernel
 * without a formula).  Reading
 * taken: per (token, V head) row of dv values,
 *   y = o / sqrt(mean(o^2) + eps) * w * SiLU(z)
 * normalising first, then gating.  o, z, y: [n][d]; w: [d].
 */
void oracle_gated_rmsnorm(const double *o, const double *z, const double *w,
                          long n, int d, double eps, double *y)
{
    for (long i = 0; i < n; ++i) {
        double ss = 0.0;
        for (int j = 0; j < d; ++j)
            ss += o[i * d + j] * o[i * d + j];
        double inv = 1.0 / sqrt(ss / d + eps);
        for (int j = 0; j < d; ++j)
            y[i * d + j] = o[i * d + j] * inv * w[j] * silu(z[i * d + j]);
    }
}
