// Causal depthwise conv1d + SiLU over the q|k|v channel stream ("causal 1D
// convolutions", "[model] support Qwen3next", Highlights), for packed
// variable-length prefill and for decode / MTP updates against a slot pool.
//
// Each thread owns 16 bytes of channels (8 bf16 or 4 fp32) and walks a run of
// tokens, keeping the last width-1 inputs in registers, so every input row is
// read from HBM once (plus width-1 rows at the head of each run).
#include "common.cuh"

namespace gdn {

GDN_DECLARE_STATUS_WORD(g_status_conv)
GDN_STATUS_READER(read_status_conv, g_status_conv)

constexpr int kConvThreads = 128;
constexpr int kConvTokensPerThread = 8;

template <typename T, int W>
struct ConvTaps {
    static constexpr int V = Vec16<T>::N;
    float w[W][V];
    float bias[V];
    // The V x W taps of channels c0 .. c0+V-1 are 16 W contiguous bytes: W
    // 16-byte loads (weight and bias 16-byte aligned, checked on the host).
    __device__ __forceinline__ void load(const T *weight, const T *b, int c0) {
        float e[V * W];
        const uint4 *src = reinterpret_cast<const uint4 *>(weight + (int64_t)c0 * W);
#pragma unroll
        for (int u = 0; u < W; ++u) Vec16<T>::unpack(__ldg(src + u), e + u * V);
#pragma unroll
        for (int v = 0; v < V; ++v)
#pragma unroll
            for (int j = 0; j < W; ++j) w[j][v] = e[v * W + j];
        if (b) {
            Vec16<T>::load(b + c0, bias);
        } else {
#pragma unroll
            for (int v = 0; v < V; ++v) bias[v] = 0.0f;
        }
    }
    // out = act(bias + sum_j w[j] * e[t-(W-1)+j]); win holds e[t-(W-1) .. t-1].
    __device__ __forceinline__ void apply(const float (&win)[W - 1][V], const float *cur,
                                          int silu, float *out) const {
#pragma unroll
        for (int v = 0; v < V; ++v) {
            float acc = bias[v];
#pragma unroll
            for (int j = 0; j < W - 1; ++j) acc = fmaf(w[j][v], win[j][v], acc);
            acc = fmaf(w[W - 1][v], cur[v], acc);
            out[v] = silu ? silu_f(acc) : acc;
        }
    }
};

template <int W, int V>
__device__ __forceinline__ void shift_in(float (&win)[W - 1][V], const float *cur) {
#pragma unroll
    for (int j = 0; j + 1 < W - 1; ++j)
#pragma unroll
        for (int v = 0; v < V; ++v) win[j][v] = win[j + 1][v];
#pragma unroll
    for (int v = 0; v < V; ++v) win[W - 2][v] = cur[v];
}

// Slot of sequence i if it holds usable history, else -1 (flags bad slots).
__device__ __forceinline__ int64_t history_slot(const int32_t *idx, const uint8_t *has_init,
                                                int i, int64_t n_slots) {
    const int64_t s = idx[i];
    if (s < 0) return -1;
    if (s >= n_slots) {
        flag_status(GDN_DEVSTAT_BAD_INDEX);
        return -1;
    }
    if (has_init && has_init[i] == 0) return -1;
    return s;
}

// Prefill: blockIdx.x = token run, blockIdx.y * blockDim.x + tid = channel group.
template <typename T, int W>
__global__ void __launch_bounds__(kConvThreads)
conv_fwd_kernel(const T *__restrict__ x, int64_t x_stride, const T *__restrict__ weight,
                const T *__restrict__ bias, const int32_t *__restrict__ cu, int n_seqs,
                int64_t n_tokens, int C, const T *__restrict__ pool, int64_t n_slots,
                const int32_t *__restrict__ idx, const uint8_t *__restrict__ has_init,
                int silu, T *__restrict__ y) {
    constexpr int V = Vec16<T>::N;
    const int c0 = (blockIdx.y * blockDim.x + threadIdx.x) * V;
    if (c0 >= C) return;
    const int64_t t0 = (int64_t)blockIdx.x * kConvTokensPerThread;
    if (t0 >= n_tokens) return;
    const int64_t t1 = min(t0 + (int64_t)kConvTokensPerThread, n_tokens);

    // The token rows and taps do not depend on the sequence lookup: issue
    // their loads first, so the binary search below overlaps them.
    uint4 raw[kConvTokensPerThread];
#pragma unroll
    for (int tt = 0; tt < kConvTokensPerThread; ++tt)
        if (t0 + tt < t1) raw[tt] = *reinterpret_cast<const uint4 *>(x + (t0 + tt) * x_stride + c0);
    ConvTaps<T, W> taps;
    taps.load(weight, bias, c0);

    // first sequence i with cu[i+1] > t0
    int lo = 0, hi = n_seqs;
    while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if (cu[mid + 1] > t0) hi = mid; else lo = mid + 1;
    }
    int i = lo;
    float win[W - 1][V];
    // fast path: the whole run lies in one sequence, so every load is issued
    // before the first use (8 token rows + the history rows in flight)
    if (i < n_seqs) {
        const int64_t ss = cu[i], se = cu[i + 1];
        if (ss >= 0 && ss <= t0 && t1 <= se && se <= n_tokens) {
            const int64_t hs = (t0 - ss < W - 1) ? history_slot(idx, has_init, i, n_slots) : -1;
#pragma unroll
            for (int r = 0; r < W - 1; ++r) {
                const int64_t n = t0 - (W - 1) + r;
                if (n >= ss) {
                    Vec16<T>::load(x + n * x_stride + c0, win[r]);
                } else if (hs >= 0) {
                    Vec16<T>::load(pool + (hs * (W - 1) + (W - 1) + (n - ss)) * C + c0, win[r]);
                } else {
#pragma unroll
                    for (int v = 0; v < V; ++v) win[r][v] = 0.0f;
                }
            }
#pragma unroll
            for (int tt = 0; tt < kConvTokensPerThread; ++tt) {
                if (t0 + tt < t1) {
                    float cur[V], out[V];
                    Vec16<T>::unpack(raw[tt], cur);
                    taps.apply(win, cur, silu, out);
                    Vec16<T>::store(y + (t0 + tt) * C + c0, out);
                    shift_in<W, V>(win, cur);
                }
            }
            return;
        }
    }
    int64_t s_end = -1;
    for (int64_t t = t0; t < t1; ++t) {
        if (t >= s_end) {
            while (i < n_seqs && cu[i + 1] <= t) ++i;
            if (i >= n_seqs) {                 // cu_seqlens does not cover n_tokens
                flag_status(GDN_DEVSTAT_BAD_SEQLEN);
                return;
            }
            const int64_t s_start = cu[i];
            s_end = cu[i + 1];
            if (s_start < 0 || s_start > t || s_end > n_tokens) {
                flag_status(GDN_DEVSTAT_BAD_SEQLEN);
                return;
            }
            const int64_t hs = history_slot(idx, has_init, i, n_slots);
#pragma unroll
            for (int r = 0; r < W - 1; ++r) {
                const int64_t n = t - (W - 1) + r;
                if (n >= s_start) {
                    Vec16<T>::load(x + n * x_stride + c0, win[r]);
                } else if (hs >= 0) {
                    const int64_t hr = (W - 1) + (n - s_start);   // history row, oldest first
                    Vec16<T>::load(pool + (hs * (W - 1) + hr) * C + c0, win[r]);
                } else {
#pragma unroll
                    for (int v = 0; v < V; ++v) win[r][v] = 0.0f;
                }
            }
        }
        float cur[V], out[V];
        Vec16<T>::load(x + t * x_stride + c0, cur);
        taps.apply(win, cur, silu, out);
        Vec16<T>::store(y + t * C + c0, out);
        shift_in<W, V>(win, cur);
    }
}

// Final conv state of every sequence: the last W-1 inputs of history ++ x.
// Runs after conv_fwd_kernel so no block reads a slot this one rewrites.
template <typename T, int W>
__global__ void __launch_bounds__(kConvThreads)
conv_final_state_kernel(const T *__restrict__ x, int64_t x_stride, const int32_t *__restrict__ cu,
                        int64_t n_tokens, int C, T *__restrict__ pool, int64_t n_slots,
                        const int32_t *__restrict__ idx, const uint8_t *__restrict__ has_init) {
    constexpr int V = Vec16<T>::N;
    const int i = blockIdx.x;
    const int c0 = (blockIdx.y * blockDim.x + threadIdx.x) * V;
    if (c0 >= C) return;
    const int64_t slot = idx[i];
    if (slot < 0) return;
    if (slot >= n_slots) {
        flag_status(GDN_DEVSTAT_BAD_INDEX);
        return;
    }
    const int64_t s = cu[i], e = cu[i + 1];
    if (s < 0 || e < s || e > n_tokens) {
        flag_status(GDN_DEVSTAT_BAD_SEQLEN);
        return;
    }
    const bool hist = !(has_init && has_init[i] == 0);
    const int64_t len = e - s;
    float vals[W - 1][V];
#pragma unroll
    for (int r = 0; r < W - 1; ++r) {
        const int64_t n = len - (W - 1) + r;
        if (n >= 0) {
            Vec16<T>::load(x + (s + n) * x_stride + c0, vals[r]);
        } else if (hist) {
            Vec16<T>::load(pool + (slot * (W - 1) + (W - 1) + n) * C + c0, vals[r]);
        } else {
#pragma unroll
            for (int v = 0; v < V; ++v) vals[r][v] = 0.0f;
        }
    }
#pragma unroll
    for (int r = 0; r < W - 1; ++r) Vec16<T>::store(pool + (slot * (W - 1) + r) * C + c0, vals[r]);
}

// Decode / MTP update: blockIdx.x = sequence, blockIdx.y = channel block.
template <typename T, int W>
__global__ void __launch_bounds__(kConvThreads)
conv_update_kernel(const T *__restrict__ x, int tps, int C, const T *__restrict__ weight,
                   const T *__restrict__ bias, T *__restrict__ pool, int64_t n_slots,
                   const int32_t *__restrict__ idx, const int32_t *__restrict__ snap, int silu,
                   T *__restrict__ y) {
    constexpr int V = Vec16<T>::N;
    const int i = blockIdx.x;
    const int c0 = (blockIdx.y * blockDim.x + threadIdx.x) * V;
    if (c0 >= C) return;
    const int64_t slot = idx[i];
    if (slot < 0 || slot >= n_slots) {
        if (slot >= n_slots) flag_status(GDN_DEVSTAT_BAD_INDEX);
        float z[V];
#pragma unroll
        for (int v = 0; v < V; ++v) z[v] = 0.0f;
        for (int t = 0; t < tps; ++t) Vec16<T>::store(y + ((int64_t)i * tps + t) * C + c0, z);
        return;
    }
    ConvTaps<T, W> taps;
    taps.load(weight, bias, c0);
    float win[W - 1][V];
#pragma unroll
    for (int r = 0; r < W - 1; ++r)
        Vec16<T>::load(pool + (slot * (W - 1) + r) * C + c0, win[r]);
    for (int t = 0; t < tps; ++t) {
        const int64_t row = (int64_t)i * tps + t;
        float cur[V], out[V];
        Vec16<T>::load(x + row * C + c0, cur);
        taps.apply(win, cur, silu, out);
        Vec16<T>::store(y + row * C + c0, out);
        shift_in<W, V>(win, cur);
        if (snap) {
            const int64_t d = snap[row];
            if (d >= n_slots) flag_status(GDN_DEVSTAT_BAD_INDEX);
            else if (d >= 0)
#pragma unroll
                for (int r = 0; r < W - 1; ++r)
                    Vec16<T>::store(pool + (d * (W - 1) + r) * C + c0, win[r]);
        }
    }
    if (!snap)
#pragma unroll
        for (int r = 0; r < W - 1; ++r) Vec16<T>::store(pool + (slot * (W - 1) + r) * C + c0, win[r]);
}

template <typename T, int W>
static void launch_fwd(const void *x, int64_t xs, const void *w, const void *b, const int32_t *cu,
                       int n_seqs, int64_t n_tokens, int C, void *pool, int64_t n_slots,
                       const int32_t *idx, const uint8_t *has, int silu, void *y, cudaStream_t s) {
    constexpr int V = Vec16<T>::N;
    const int groups = C / V;
    dim3 block(kConvThreads);
    if (n_tokens > 0) {
        dim3 grid((unsigned)((n_tokens + kConvTokensPerThread - 1) / kConvTokensPerThread),
                  (unsigned)((groups + kConvThreads - 1) / kConvThreads));
        conv_fwd_kernel<T, W><<<grid, block, 0, s>>>(
            (const T *)x, xs, (const T *)w, (const T *)b, cu, n_seqs, n_tokens, C,
            (const T *)pool, n_slots, idx, has, silu, (T *)y);
    }
    if (pool) {
        dim3 grid2((unsigned)n_seqs, (unsigned)((groups + kConvThreads - 1) / kConvThreads));
        conv_final_state_kernel<T, W><<<grid2, block, 0, s>>>(
            (const T *)x, xs, cu, n_tokens, C, (T *)pool, n_slots, idx, has);
    }
}

template <typename T, int W>
static void launch_update(const void *x, int n_seqs, int tps, int C, const void *w, const void *b,
                          void *pool, int64_t n_slots, const int32_t *idx, const int32_t *snap,
                          int silu, void *y, cudaStream_t s) {
    constexpr int V = Vec16<T>::N;
    const int groups = C / V;
    dim3 grid((unsigned)n_seqs, (unsigned)((groups + kConvThreads - 1) / kConvThreads));
    conv_update_kernel<T, W><<<grid, kConvThreads, 0, s>>>(
        (const T *)x, tps, C, (const T *)w, (const T *)b, (T *)pool, n_slots, idx, snap, silu,
        (T *)y);
}

static bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace gdn

using namespace gdn;

extern "C" gdn_status causal_conv1d_fwd(const void *x, int64_t x_row_stride, const void *weight,
                                        const void *bias, const int32_t *cu_seqlens, int32_t n_seqs,
                                        int64_t n_tokens, int32_t channels, int32_t width,
                                        void *conv_state_pool, int64_t n_slots,
                                        const int32_t *state_indices,
                                        const uint8_t *has_initial_state, int32_t silu, void *y,
                                        int32_t dtype, void *stream) {
    GDN_REQUIRE(dtype == GDN_F32 || dtype == GDN_BF16, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(n_seqs >= 0 && n_tokens >= 0 && channels > 0 && n_slots >= 0, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(width >= 2 && width <= 4, GDN_ERR_UNSUPPORTED);
    GDN_REQUIRE(channels % 8 == 0, GDN_ERR_UNSUPPORTED);
    if (n_seqs == 0) return n_tokens == 0 ? GDN_OK : GDN_ERR_INVALID_ARG;
    GDN_REQUIRE(weight && cu_seqlens && state_indices && conv_state_pool, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(n_tokens == 0 || (x && y), GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(x_row_stride >= channels, GDN_ERR_INVALID_ARG);
    const int elem = dtype == GDN_F32 ? 4 : 2;
    GDN_REQUIRE((x_row_stride * elem) % 16 == 0, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(aligned16(x) && aligned16(y) && aligned16(conv_state_pool), GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(aligned16(weight) && aligned16(bias), GDN_ERR_INVALID_ARG);
    cudaStream_t s = (cudaStream_t)stream;
#define GDN_CONV_FWD(T, W)                                                                     \
    launch_fwd<T, W>(x, x_row_stride, weight, bias, cu_seqlens, n_seqs, n_tokens, channels,    \
                     conv_state_pool, n_slots, state_indices, has_initial_state, silu, y, s)
    if (dtype == GDN_F32) {
        if (width == 2) GDN_CONV_FWD(float, 2);
        else if (width == 3) GDN_CONV_FWD(float, 3);
        else GDN_CONV_FWD(float, 4);
    } else {
        if (width == 2) GDN_CONV_FWD(__nv_bfloat16, 2);
        else if (width == 3) GDN_CONV_FWD(__nv_bfloat16, 3);
        else GDN_CONV_FWD(__nv_bfloat16, 4);
    }
#undef GDN_CONV_FWD
    return launch_status();
}

extern "C" gdn_status causal_conv1d_update(const void *x, int32_t n_seqs, int32_t tokens_per_seq,
                                           int32_t channels, int32_t width, const void *weight,
                                           const void *bias, void *conv_state_pool,
                                           int64_t n_slots, const int32_t *state_indices,
                                           const int32_t *snap_indices, int32_t silu, void *y,
                                           int32_t dtype, void *stream) {
    GDN_REQUIRE(dtype == GDN_F32 || dtype == GDN_BF16, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(n_seqs >= 0 && channels > 0 && n_slots >= 0, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(tokens_per_seq >= 1 && tokens_per_seq <= 16, GDN_ERR_UNSUPPORTED);
    GDN_REQUIRE(width >= 2 && width <= 4, GDN_ERR_UNSUPPORTED);
    GDN_REQUIRE(channels % 8 == 0, GDN_ERR_UNSUPPORTED);
    if (n_seqs == 0) return GDN_OK;
    GDN_REQUIRE(x && y && weight && conv_state_pool && state_indices, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(aligned16(x) && aligned16(y) && aligned16(conv_state_pool), GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(aligned16(weight) && aligned16(bias), GDN_ERR_INVALID_ARG);
    cudaStream_t s = (cudaStream_t)stream;
#define GDN_CONV_UPD(T, W)                                                                     \
    launch_update<T, W>(x, n_seqs, tokens_per_seq, channels, weight, bias, conv_state_pool,    \
                        n_slots, state_indices, snap_indices, silu, y, s)
    if (dtype == GDN_F32) {
        if (width == 2) GDN_CONV_UPD(float, 2);
        else if (width == 3) GDN_CONV_UPD(float, 3);
        else GDN_CONV_UPD(float, 4);
    } else {
        if (width == 2) GDN_CONV_UPD(__nv_bfloat16, 2);
        else if (width == 3) GDN_CONV_UPD(__nv_bfloat16, 3);
        else GDN_CONV_UPD(__nv_bfloat16, 4);
    }
#undef GDN_CONV_UPD
    return launch_status();
}
