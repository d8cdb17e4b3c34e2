// Causal depthwise conv1d + SiLU over the q|k|v channel stream ("causal 1D
// convolutions", "[model] support Qwen3next", Highlights), for packed
// variable-length prefill and for decode / MTP updates against a slot pool.
//
// A thread owns a few channels and walks a run of tokens, keeping the last
// width-1 inputs in registers, so every input row is read from HBM once (plus
// width-1 rows at the head of each run):
//   - prefill, bf16 with channels a multiple of 512: tiles of 32 tokens x 512
//     channels staged in shared memory by TMA (conv_fwd_tma_kernel);
//   - prefill, other shapes: 4 channels x 8 tokens per thread, straight from
//     global memory (conv_fwd_kernel);
//   - decode / MTP update: 16 bytes of channels per thread over the few new
//     tokens of a sequence (conv_update_kernel).
#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "tc.cuh"

namespace gdn {

GDN_DECLARE_STATUS_WORD(g_status_conv)
GDN_STATUS_READER(read_status_conv, g_status_conv)

constexpr int kConvThreads = 128;
constexpr int kConvTokensPerThread = 8;   // token run of a thread in the forward kernel

// SiLU: silu_for<T> (common.cuh) -- the fast division for fp32 outputs, the
// one-instruction tanh form for bf16.  The forward conv is issue-bound on this
// arithmetic.

// Four channels of T as one vector access (8 bytes of bf16, 16 of fp32).
template <typename T> struct Vec4;
template <> struct Vec4<float> {
    using Raw = float4;
    static __device__ __forceinline__ Raw raw(const float *p) { return *reinterpret_cast<const float4 *>(p); }
    static __device__ __forceinline__ void unpack(const Raw &r, float *out) {
        out[0] = r.x; out[1] = r.y; out[2] = r.z; out[3] = r.w;
    }
    static __device__ __forceinline__ void load(const float *p, float *out) { unpack(raw(p), out); }
    static __device__ __forceinline__ void store(float *p, const float *in) {
        *reinterpret_cast<float4 *>(p) = make_float4(in[0], in[1], in[2], in[3]);
    }
};
template <> struct Vec4<__nv_bfloat16> {
    using Raw = uint2;
    static __device__ __forceinline__ Raw raw(const __nv_bfloat16 *p) { return *reinterpret_cast<const uint2 *>(p); }
    static __device__ __forceinline__ void unpack(const Raw &r, float *out) {
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.y));
        out[0] = a.x; out[1] = a.y; out[2] = b.x; out[3] = b.y;
    }
    static __device__ __forceinline__ void load(const __nv_bfloat16 *p, float *out) { unpack(raw(p), out); }
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, const float *in) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(in[0], in[1]), hi = __floats2bfloat162_rn(in[2], in[3]);
        uint2 u;
        u.x = *reinterpret_cast<const uint32_t *>(&lo);
        u.y = *reinterpret_cast<const uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(p) = u;
    }
};

// V channels' taps and bias in registers.
template <typename T, int W, int V = Vec16<T>::N>
struct ConvTaps {
    float w[W][V];
    float bias[V];
    // The V x W taps of channels c0 .. c0+V-1 are V W contiguous elements,
    // read as 8-byte pieces (V W sizeof(T) is a multiple of 8 and c0 W
    // sizeof(T) one of 8 for V >= 4; weight and bias are 16-byte aligned,
    // checked on the host).
    __device__ __forceinline__ void load(const T *weight, const T *b, int c0) {
        constexpr int kPer8 = 8 / (int)sizeof(T);
        constexpr int kPieces = V * W / kPer8;
        static_assert((V * W) % kPer8 == 0, "taps are whole 8-byte pieces");
        __align__(8) T e[V * W];
        const uint2 *src = reinterpret_cast<const uint2 *>(weight + (int64_t)c0 * W);
#pragma unroll
        for (int u = 0; u < kPieces; ++u) *reinterpret_cast<uint2 *>(e + u * kPer8) = __ldg(src + u);
#pragma unroll
        for (int v = 0; v < V; ++v)
#pragma unroll
            for (int j = 0; j < W; ++j) w[j][v] = to_f(e[v * W + j]);
        if (b) {
#pragma unroll
            for (int v = 0; v < V; ++v) bias[v] = to_f(b[c0 + v]);
        } else {
#pragma unroll
            for (int v = 0; v < V; ++v) bias[v] = 0.0f;
        }
    }
    static __device__ __forceinline__ float to_f(float a) { return a; }
    static __device__ __forceinline__ float to_f(__nv_bfloat16 a) { return __bfloat162float(a); }
    // out = act(bias + sum_j w[j] * e[t-(W-1)+j]); win holds e[t-(W-1) .. t-1].
    __device__ __forceinline__ void apply(const float (&win)[W - 1][V], const float *cur,
                                          int silu, float *out) const {
#pragma unroll
        for (int v = 0; v < V; ++v) {
            float acc = bias[v];
#pragma unroll
            for (int j = 0; j < W - 1; ++j) acc = fmaf(w[j][v], win[j][v], acc);
            acc = fmaf(w[W - 1][v], cur[v], acc);
            out[v] = silu ? silu_for<T>(acc) : acc;
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

// Prefill: blockIdx.x = token run of R tokens, blockIdx.y * blockDim.x + tid
// = group of 4 channels.  A thread keeps 4 channels' taps, its W-1 window
// and its R input rows in registers (about 70 at R = 8 in bf16), so 8 warps
// and more share an SM: the kernel is issue-bound on the conv + SiLU
// arithmetic, not on HBM, when fewer warps hide its latencies.
template <typename T, int W, int R>
__global__ void __launch_bounds__(kConvThreads)
conv_fwd_kernel(const T *__restrict__ x, int64_t x_stride, const T *__restrict__ weight,
                const T *__restrict__ bias, const int32_t *__restrict__ cu, int n_seqs,
                int64_t n_tokens, int C, const T *__restrict__ pool, int64_t n_slots,
                const int32_t *__restrict__ idx, const uint8_t *__restrict__ has_init,
                int silu, T *__restrict__ y) {
    constexpr int V = 4;
    using VT = Vec4<T>;
    const int c0 = (blockIdx.y * blockDim.x + threadIdx.x) * V;
    if (c0 >= C) return;
    const int64_t t0 = (int64_t)blockIdx.x * R;
    if (t0 >= n_tokens) return;
    const int64_t t1 = min(t0 + (int64_t)R, n_tokens);

    // The token rows, the W-1 rows before the run (the window when the run
    // does not start a sequence) and the taps do not depend on the sequence
    // lookup: issue their loads first, so the binary search overlaps them.
    typename VT::Raw raw[R], hraw[W - 1];
#pragma unroll
    for (int tt = 0; tt < R; ++tt)
        if (t0 + tt < t1) raw[tt] = VT::raw(x + (t0 + tt) * x_stride + c0);
#pragma unroll
    for (int r = 0; r < W - 1; ++r) {
        const int64_t n = t0 - (W - 1) + r;
        if (n >= 0) hraw[r] = VT::raw(x + n * x_stride + c0);
    }
    ConvTaps<T, W, V> taps;
    taps.load(weight, bias, c0);

    // first sequence i with cu[i+1] > t0
    int lo = 0, hi = n_seqs;
    while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if (cu[mid + 1] > t0) hi = mid; else lo = mid + 1;
    }
    int i = lo;
    float win[W - 1][V];
    // fast path: the whole run lies in one sequence
    if (i < n_seqs) {
        const int64_t ss = cu[i], se = cu[i + 1];
        if (ss >= 0 && ss <= t0 && t1 <= se && se <= n_tokens) {
            const int64_t hs = (t0 - ss < W - 1) ? history_slot(idx, has_init, i, n_slots) : -1;
#pragma unroll
            for (int r = 0; r < W - 1; ++r) {
                const int64_t n = t0 - (W - 1) + r;
                if (n >= ss) {
                    VT::unpack(hraw[r], win[r]);
                } else if (hs >= 0) {
                    VT::load(pool + (hs * (W - 1) + (W - 1) + (n - ss)) * C + c0, win[r]);
                } else {
#pragma unroll
                    for (int v = 0; v < V; ++v) win[r][v] = 0.0f;
                }
            }
#pragma unroll
            for (int tt = 0; tt < R; ++tt) {
                if (t0 + tt < t1) {
                    float cur[V], out[V];
                    VT::unpack(raw[tt], cur);
                    taps.apply(win, cur, silu, out);
                    VT::store(y + (t0 + tt) * C + c0, out);
                    shift_in<W, V>(win, cur);
                }
            }
            return;
        }
    }
    // the run crosses a sequence boundary (or cu_seqlens is malformed)
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
                    VT::load(x + n * x_stride + c0, win[r]);
                } else if (hs >= 0) {
                    const int64_t hr = (W - 1) + (n - s_start);   // history row, oldest first
                    VT::load(pool + (hs * (W - 1) + hr) * C + c0, win[r]);
                } else {
#pragma unroll
                    for (int v = 0; v < V; ++v) win[r][v] = 0.0f;
                }
            }
        }
        float cur[V], out[V];
        VT::load(x + t * x_stride + c0, cur);
        taps.apply(win, cur, silu, out);
        VT::store(y + t * C + c0, out);
        shift_in<W, V>(win, cur);
    }
}

// Prefill, TMA-staged (bf16, channels a multiple of 512): a persistent grid
// of CTAs walks tiles of 32 tokens x 512 channels.  A tile's 32 input rows
// and the 3 rows before them come into shared memory as two 2-D TMA boxes
// of 256 channels x 35 rows (zero-filled outside the tensor), through a ring
// of 2 stages on mbarriers (3 CTAs per SM), so the next tile is in flight
// while this one is computed, whatever the registers.  256 threads: thread t
// convolves channels 4 (t % 128) .. +3 over tokens 16 (t / 128) .. +15 of
// the tile from shared memory (its window is in the staged rows too) and
// stores y directly.
// The kernel is bound by the latency of its conv + SiLU chains more than by
// HBM: a tile that lies inside one sequence with its window staged (nearly
// all) runs a branch-free loop over its 16 tokens, so the compiler can
// interleave 64 independent chains per thread.  A CTA's tiles move forward
// in tokens, so its sequence index only ever advances.
constexpr int kTileTok = 32;
constexpr int kTileCh = 512;                        // 128 channel threads x 4 channels
constexpr int kTileHist = 3;                        // rows before the tile (W - 1 <= 3)
constexpr int kTileRows = kTileTok + kTileHist;
constexpr int kBoxCh = 256;                         // TMA box width (<= 256 elements)
constexpr uint32_t kBoxBytes = kTileRows * kBoxCh * 2;
constexpr uint32_t kTileBytes = 2 * kBoxBytes;
constexpr int kTileStages = 2;
constexpr int kTileCtasPerSm = 3;
constexpr int kTileParts = 2;                       // token halves of a tile
constexpr int kPartTok = kTileTok / kTileParts;
constexpr int kTmaThreads = (kTileCh / 4) * kTileParts;

template <int W>
__global__ void __launch_bounds__(kTmaThreads, kTileCtasPerSm)
conv_fwd_tma_kernel(const __grid_constant__ CUtensorMap tm_x, const __nv_bfloat16 *__restrict__ weight,
                    const __nv_bfloat16 *__restrict__ bias, const int32_t *__restrict__ cu,
                    int n_seqs, int n_tokens, int C, const __nv_bfloat16 *__restrict__ pool,
                    int64_t n_slots, const int32_t *__restrict__ idx,
                    const uint8_t *__restrict__ has_init, int silu, __nv_bfloat16 *__restrict__ y) {
    using namespace tc;
    using VT = Vec4<__nv_bfloat16>;
    constexpr int V = 4;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    __shared__ uint64_t full[kTileStages];
    __shared__ int abort_flag;
    const int tid = threadIdx.x;
    const int ct = tid % (kTileCh / V), part = tid / (kTileCh / V);
    const int n_cb = C / kTileCh;
    const int n_tiles = ((n_tokens + kTileTok - 1) / kTileTok) * n_cb;
    if (tid == 0) {
        for (int st = 0; st < kTileStages; ++st) mbar_init(&full[st], 1);
        abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&tm_x);
    }
    __syncthreads();
    volatile int *abort = &abort_flag;
    auto issue = [&](int tile, int st) {   // thread 0
        const int tb = tile / n_cb, cb = tile - tb * n_cb;
        uint8_t *dst = smem_raw + st * kTileBytes;
        mbar_arrive_expect_tx(&full[st], kTileBytes);
        tma_load_2d(dst, &tm_x, &full[st], cb * kTileCh, tb * kTileTok - kTileHist);
        tma_load_2d(dst + kBoxBytes, &tm_x, &full[st], cb * kTileCh + kBoxCh, tb * kTileTok - kTileHist);
    };
    if (tid == 0)
        for (int j = 0; j < kTileStages - 1; ++j) {
            const int tile = blockIdx.x + j * gridDim.x;
            if (tile < n_tiles) issue(tile, j);
        }
    // this thread's 4 channels within a staged row (row r = token tb*32 - 3 + r)
    const int box = ct / (kBoxCh / V), col = ct % (kBoxCh / V);
    auto row_raw = [&](const uint8_t *stage, int r) {
        return *reinterpret_cast<const VT::Raw *>(stage + box * kBoxBytes + r * (kBoxCh * 2) + col * 8);
    };
    int i = -1;                       // sequence of this thread's current token
    int64_t ss = 0, se = 0;           // its token range
    bool bad = false;                 // cu_seqlens does not describe the tokens
    int cb_taps = -1;
    ConvTaps<__nv_bfloat16, W, V> taps;
    for (int j = 0;; ++j) {
        const int tile = blockIdx.x + j * gridDim.x;
        if (tile >= n_tiles) break;
        const int st = j % kTileStages;
        if (tid == 0) {               // refill the stage the previous tile used
            const int tn = tile + (kTileStages - 1) * gridDim.x;
            if (tn < n_tiles) issue(tn, (j + kTileStages - 1) % kTileStages);
        }
        const int tb = tile / n_cb, cb = tile - tb * n_cb;
        const int c0 = cb * kTileCh + ct * V;
        if (cb != cb_taps) {
            taps.load(weight, bias, c0);
            cb_taps = cb;
        }
        const int64_t tbase = (int64_t)tb * kTileTok;             // staged row 3
        const int64_t t0 = tbase + part * kPartTok;                // this thread's tokens
        const int64_t t1 = min(t0 + (int64_t)kPartTok, (int64_t)n_tokens);
        const bool any = t0 < t1;
        // the sequence holding t0 (forward from the last one, else a search)
        if (any && (i < 0 || t0 < ss)) {
            int lo = 0, hi = n_seqs;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (cu[mid + 1] > t0) hi = mid; else lo = mid + 1;
            }
            i = lo;
            if (i < n_seqs) { ss = cu[i]; se = cu[i + 1]; }
        }
        while (any && i < n_seqs && se <= t0) {
            ++i;
            if (i < n_seqs) { ss = cu[i]; se = cu[i + 1]; }
        }
        if (any && (i >= n_seqs || ss < 0 || ss > t0 || se > n_tokens)) bad = true;
        const uint8_t *stage = smem_raw + st * kTileBytes;
        const int r0 = part * kPartTok + kTileHist;                // staged row of t0
        mbar_wait(&full[st], (j / kTileStages) & 1, abort);
        if (!bad && t1 - t0 == kPartTok && t0 - ss >= W - 1 && se >= t1) {
            // inside one sequence with the window staged: no branches
            float win[W - 1][V];
#pragma unroll
            for (int r = 0; r < W - 1; ++r) VT::unpack(row_raw(stage, r0 - (W - 1) + r), win[r]);
#pragma unroll
            for (int tt = 0; tt < kPartTok; ++tt) {
                float cur[V], out[V];
                VT::unpack(row_raw(stage, r0 + tt), cur);
                taps.apply(win, cur, silu, out);
                VT::store(y + (t0 + tt) * C + c0, out);
                shift_in<W, V>(win, cur);
            }
        } else if (!bad && any) {
            float win[W - 1][V];
            // history of the sequence from its slot (or zeros) for rows
            // before its start, else the staged rows
            auto fill_window = [&](int64_t t) {
                const int64_t hs = (t - ss < W - 1) ? history_slot(idx, has_init, i, n_slots) : -1;
#pragma unroll
                for (int r = 0; r < W - 1; ++r) {
                    const int64_t n = t - (W - 1) + r;
                    if (n >= ss) {
                        VT::unpack(row_raw(stage, (int)(n - tbase) + kTileHist), win[r]);
                    } else if (hs >= 0) {
                        VT::load(pool + (hs * (W - 1) + (W - 1) + (n - ss)) * C + c0, win[r]);
                    } else {
#pragma unroll
                        for (int v = 0; v < V; ++v) win[r][v] = 0.0f;
                    }
                }
            };
            fill_window(t0);
            for (int tt = 0; tt < kPartTok; ++tt) {
                const int64_t t = t0 + tt;
                if (t >= t1) break;
                if (t == se) {        // the next sequence starts here
                    do {              // (skipping empty ones)
                        ++i;
                        if (i < n_seqs) { ss = cu[i]; se = cu[i + 1]; }
                    } while (i < n_seqs && se == t && ss == t);
                    if (i >= n_seqs || ss != t || se < ss || se > n_tokens) { bad = true; break; }
                    fill_window(t);
                }
                float cur[V], out[V];
                VT::unpack(row_raw(stage, r0 + tt), cur);
                taps.apply(win, cur, silu, out);
                VT::store(y + t * C + c0, out);
                shift_in<W, V>(win, cur);
            }
        }
        __syncthreads();              // the stage is refilled next iteration
    }
    if (bad) flag_status(GDN_DEVSTAT_BAD_SEQLEN);
    if (tid == 0 && abort_flag) flag_status(GDN_DEVSTAT_TIMEOUT);
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
    constexpr int kAhead = 4;   // tokens whose x rows and snapshot slots are loaded up front
    const int i = blockIdx.x;
    const int c0 = (blockIdx.y * blockDim.x + threadIdx.x) * V;
    if (c0 >= C) return;
    const int64_t slot = idx[i];
    // what needs no slot id is requested while the slot id is on its way
    uint4 xr[kAhead];
    int64_t sn[kAhead];
#pragma unroll
    for (int t = 0; t < kAhead; ++t) {
        if (t < tps) {
            const int64_t row = (int64_t)i * tps + t;
            xr[t] = *reinterpret_cast<const uint4 *>(x + row * C + c0);
            sn[t] = snap ? (int64_t)snap[row] : -1;
        }
    }
    ConvTaps<T, W> taps;
    taps.load(weight, bias, c0);
    if (slot < 0 || slot >= n_slots) {
        if (slot >= n_slots) flag_status(GDN_DEVSTAT_BAD_INDEX);
        float z[V];
#pragma unroll
        for (int v = 0; v < V; ++v) z[v] = 0.0f;
        for (int t = 0; t < tps; ++t) Vec16<T>::store(y + ((int64_t)i * tps + t) * C + c0, z);
        return;
    }
    float win[W - 1][V];
#pragma unroll
    for (int r = 0; r < W - 1; ++r)
        Vec16<T>::load(pool + (slot * (W - 1) + r) * C + c0, win[r]);
    for (int t = 0; t < tps; ++t) {
        const int64_t row = (int64_t)i * tps + t;
        float cur[V], out[V];
        if (t < kAhead) {
#pragma unroll
            for (int u = 0; u < kAhead; ++u)
                if (u == t) Vec16<T>::unpack(xr[u], cur);
        } else {
            Vec16<T>::load(x + row * C + c0, cur);
        }
        taps.apply(win, cur, silu, out);
        Vec16<T>::store(y + row * C + c0, out);
        shift_in<W, V>(win, cur);
        if (snap) {
            int64_t d = 0;
            if (t < kAhead) {
#pragma unroll
                for (int u = 0; u < kAhead; ++u)
                    if (u == t) d = sn[u];
            } else {
                d = snap[row];
            }
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

// The TMA-staged kernel when the shape allows it (bf16, channels a multiple
// of 512, token coordinates in int32); false: use the register kernel.
template <int W>
static bool launch_fwd_tma(const void *x, int64_t xs, const void *w, const void *b,
                           const int32_t *cu, int n_seqs, int64_t n_tokens, int C, void *pool,
                           int64_t n_slots, const int32_t *idx, const uint8_t *has, int silu,
                           void *y, cudaStream_t s) {
    if (C % kTileCh != 0 || n_tokens + kTileTok >= (1ll << 31)) return false;
    CUtensorMap tm;
    if (!encode_tmap_2d_bf16(&tm, x, (uint64_t)C, (uint64_t)n_tokens, (uint64_t)xs, kBoxCh,
                             kTileRows, false))
        return false;
    const int smem = kTileStages * kTileBytes;
    if (cudaFuncSetAttribute(conv_fwd_tma_kernel<W>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
        return false;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t n_tiles = ((n_tokens + kTileTok - 1) / kTileTok) * (C / kTileCh);
    const int grid = (int)std::min<int64_t>(n_tiles, (int64_t)sms * kTileCtasPerSm);
    conv_fwd_tma_kernel<W><<<grid, kTmaThreads, smem, s>>>(
        tm, (const __nv_bfloat16 *)w, (const __nv_bfloat16 *)b, cu, n_seqs, (int)n_tokens, C,
        (const __nv_bfloat16 *)pool, n_slots, idx, has, silu, (__nv_bfloat16 *)y);
    return true;
}

template <typename T, int W>
static void launch_fwd(const void *x, int64_t xs, const void *w, const void *b, const int32_t *cu,
                       int n_seqs, int64_t n_tokens, int C, void *pool, int64_t n_slots,
                       const int32_t *idx, const uint8_t *has, int silu, void *y, cudaStream_t s) {
    dim3 block(kConvThreads);
    bool done = n_tokens == 0;
    if constexpr (std::is_same<T, __nv_bfloat16>::value)
        if (!done)
            done = launch_fwd_tma<W>(x, xs, w, b, cu, n_seqs, n_tokens, C, pool, n_slots, idx, has,
                                     silu, y, s);
    if (!done) {
        dim3 grid((unsigned)((n_tokens + kConvTokensPerThread - 1) / kConvTokensPerThread),
                  (unsigned)((C / 4 + kConvThreads - 1) / kConvThreads));
        conv_fwd_kernel<T, W, kConvTokensPerThread><<<grid, block, 0, s>>>(
            (const T *)x, xs, (const T *)w, (const T *)b, cu, n_seqs, n_tokens, C,
            (const T *)pool, n_slots, idx, has, silu, (T *)y);
    }
    if (pool) {
        constexpr int V = Vec16<T>::N;
        const int groups = C / V;
        dim3 grid2((unsigned)n_seqs, (unsigned)((groups + kConvThreads - 1) / kConvThreads));
        conv_final_state_kernel<T, W><<<grid2, block, 0, s>>>(
            (const T *)x, xs, cu, n_tokens, C, (T *)pool, n_slots, idx, has);
    }
}

// bf16, up to kUpd1MaxTps tokens per sequence (the decode step, the MTP
// step): one thread per 8 channels of one sequence, with the taps kept as
// the raw 16-byte vectors they load as and widened where they are used.  Few
// registers, so many warps in flight: the kernel is latency-bound (a slot id,
// then the slot's conv state).  Same arithmetic order as conv_update_kernel.
constexpr int kUpd1Threads = 256;
constexpr int kUpd1MaxTps = 4;
template <int W, int kMaxT>   // kMaxT: 1 for the decode step (fewer registers), else 4
__global__ void __launch_bounds__(kUpd1Threads)
conv_update1_kernel(const __nv_bfloat16 *__restrict__ x, int n_seqs, int tps, int C,
                    const __nv_bfloat16 *__restrict__ weight, const __nv_bfloat16 *__restrict__ bias,
                    __nv_bfloat16 *__restrict__ pool, int64_t n_slots,
                    const int32_t *__restrict__ idx, const int32_t *__restrict__ snap, int silu,
                    __nv_bfloat16 *__restrict__ y) {
    const int per_seq = C / 8;
    const int64_t gt = (int64_t)blockIdx.x * kUpd1Threads + threadIdx.x;
    const int i = (int)(gt / per_seq);
    if (i >= n_seqs) return;
    const int c0 = (int)(gt - (int64_t)i * per_seq) * 8;
    const int64_t slot = idx[i];
    // everything but the conv state is requested before the slot id is back
    uint4 xv[kMaxT];
    int64_t sn[kMaxT];
#pragma unroll
    for (int t = 0; t < kMaxT; ++t) {
        if (t < tps) {
            const int64_t row = (int64_t)i * tps + t;
            xv[t] = *reinterpret_cast<const uint4 *>(x + row * C + c0);
            sn[t] = snap ? (int64_t)snap[row] : -1;
        }
    }
    uint4 wv[W];                                   // taps of the 8 channels: 8 W bf16
    const uint4 *wsrc = reinterpret_cast<const uint4 *>(weight + (int64_t)c0 * W);
#pragma unroll
    for (int u = 0; u < W; ++u) wv[u] = __ldg(wsrc + u);
    const uint4 bv = bias ? __ldg(reinterpret_cast<const uint4 *>(bias + c0)) : make_uint4(0u, 0u, 0u, 0u);
    if (slot < 0 || slot >= n_slots) {
        if (slot >= n_slots && c0 == 0) flag_status(GDN_DEVSTAT_BAD_INDEX);
#pragma unroll
        for (int t = 0; t < kMaxT; ++t)
            if (t < tps)
                *reinterpret_cast<uint4 *>(y + ((int64_t)i * tps + t) * C + c0) =
                    make_uint4(0u, 0u, 0u, 0u);
        return;
    }
    __nv_bfloat16 *cs = pool + slot * (W - 1) * C + c0;
    uint4 hv[W];                                   // the window: W - 1 earlier inputs, then x_t
#pragma unroll
    for (int r = 0; r < W - 1; ++r) hv[r] = *reinterpret_cast<const uint4 *>(cs + (int64_t)r * C);
    auto elem = [](const uint4 *v, int e) {        // bf16 element e of a vector array
        const uint32_t w = reinterpret_cast<const uint32_t *>(v)[e >> 1];
        return __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
    };
#pragma unroll
    for (int t = 0; t < kMaxT; ++t) {
        if (t >= tps) break;
        hv[W - 1] = xv[t];
        uint32_t out[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            float r2[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int v = 2 * p + u;
                float acc = elem(&bv, v);
#pragma unroll
                for (int j = 0; j < W; ++j) acc = fmaf(elem(wv, v * W + j), elem(&hv[j], v), acc);
                r2[u] = silu ? silu_bf16out(acc) : acc;
            }
            __nv_bfloat162 h2 = __floats2bfloat162_rn(r2[0], r2[1]);
            out[p] = *reinterpret_cast<uint32_t *>(&h2);
        }
        *reinterpret_cast<uint4 *>(y + ((int64_t)i * tps + t) * C + c0) =
            make_uint4(out[0], out[1], out[2], out[3]);
        // the window shifts by one input: the raw bf16 values move as they are
#pragma unroll
        for (int r = 0; r < W - 1; ++r) hv[r] = hv[r + 1];
        if (snap) {   // the state after token t (the last W - 1 inputs) to slot sn[t]
            if (sn[t] >= n_slots) {
                flag_status(GDN_DEVSTAT_BAD_INDEX);
            } else if (sn[t] >= 0) {
                __nv_bfloat16 *ds = pool + sn[t] * (W - 1) * C + c0;
#pragma unroll
                for (int r = 0; r < W - 1; ++r) *reinterpret_cast<uint4 *>(ds + (int64_t)r * C) = hv[r];
            }
        }
    }
    if (!snap)
#pragma unroll
        for (int r = 0; r < W - 1; ++r) *reinterpret_cast<uint4 *>(cs + (int64_t)r * C) = hv[r];
}

template <typename T, int W>
static void launch_update(const void *x, int n_seqs, int tps, int C, const void *w, const void *b,
                          void *pool, int64_t n_slots, const int32_t *idx, const int32_t *snap,
                          int silu, void *y, cudaStream_t s) {
    if constexpr (std::is_same<T, __nv_bfloat16>::value) {
        if (tps <= kUpd1MaxTps) {
            const int64_t threads = (int64_t)n_seqs * (C / 8);
            const unsigned grid = (unsigned)((threads + kUpd1Threads - 1) / kUpd1Threads);
            if (tps == 1)
                conv_update1_kernel<W, 1><<<grid, kUpd1Threads, 0, s>>>(
                    (const __nv_bfloat16 *)x, n_seqs, tps, C, (const __nv_bfloat16 *)w,
                    (const __nv_bfloat16 *)b, (__nv_bfloat16 *)pool, n_slots, idx, snap, silu,
                    (__nv_bfloat16 *)y);
            else
                conv_update1_kernel<W, kUpd1MaxTps><<<grid, kUpd1Threads, 0, s>>>(
                    (const __nv_bfloat16 *)x, n_seqs, tps, C, (const __nv_bfloat16 *)w,
                    (const __nv_bfloat16 *)b, (__nv_bfloat16 *)pool, n_slots, idx, snap, silu,
                    (__nv_bfloat16 *)y);
            return;
        }
    }
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
