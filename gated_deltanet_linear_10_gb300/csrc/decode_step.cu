// One decode step of the layer in one kernel: causal conv update (width 4)
// + SiLU of the raw q|k|v stream, fused gating, q/k L2 norms and the
// recurrent update of the state ("[model] support Qwen3next" and "[model]
// Support Qwen3next", Highlights: causal 1D convolution, fused GDN gating,
// fused recurrent GDN).  bf16 activations, dk = dv = 128, one token per
// sequence; the conv state and the recurrent state of sequence i live in
// slot idx[i] of their pools.
//
// Persistent CTAs loop over (sequence, QK head) groups.  A group is the
// grp = hv / hqk V heads that read one QK head, as 2 * grp items of 64
// state rows.  Per group, thread t computes the conv of one q|k channel
// (t < 256) and of one of the group's v channels, writes both conv states,
// and the group's q, k are normalised once in shared memory (double-buffered:
// group G + 1's are computed after group G's first item, while its other
// items stream); the items stream their 32 KiB half-states through two
// shared-memory stages exactly as the streaming decode kernel does.  Doing the conv of the shared q|k
// channels in one CTA is what makes the in-place conv state update safe:
// no other CTA reads those channels.  The next group's raw inputs are loaded
// into registers one group ahead.
#include <algorithm>

#include "common.cuh"
#include "tc.cuh"

namespace gdn {

GDN_DECLARE_STATUS_WORD(g_status_decode_step)
GDN_STATUS_READER(read_status_decode_step, g_status_decode_step)

namespace dstep {
using namespace tc;

constexpr int kThreads = 256;
constexpr int kW = 4;                        // conv width
constexpr int kRows = 64;                    // state rows per item
constexpr uint32_t kStageBytes = kRows * 128 * 4;
constexpr int kCtasPerSm = 3;
constexpr int kMaxGrp = 2;                   // V heads per QK head (256 v channels)
constexpr float kL2Eps = 1e-6f;

__device__ __forceinline__ float bf(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ float softplus_f(float x) { return x > 20.f ? x : log1pf(__expf(x)); }

// One channel's raw conv inputs: the current token, 3 history values, 4 taps.
struct ConvIn {
    float x, h[kW - 1], w[kW], bias;
};

__device__ __forceinline__ void load_conv(ConvIn &c, const __nv_bfloat16 *x,
                                          const __nv_bfloat16 *cw, const __nv_bfloat16 *cb,
                                          const __nv_bfloat16 *cpool, int64_t cslot, int C,
                                          int ch) {
    c.x = bf(x + ch);
#pragma unroll
    for (int r = 0; r < kW - 1; ++r) c.h[r] = bf(cpool + (cslot * (kW - 1) + r) * C + ch);
    const uint2 wv = *reinterpret_cast<const uint2 *>(cw + (int64_t)ch * kW);   // 4 taps, 8 B
    const float2 w01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&wv.x));
    const float2 w23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&wv.y));
    c.w[0] = w01.x; c.w[1] = w01.y; c.w[2] = w23.x; c.w[3] = w23.y;
    c.bias = cb ? bf(cb + ch) : 0.f;
}

// SiLU(bias + sum_w W[w] x_{t-3+w}); tap 3 multiplies the current token.
__device__ __forceinline__ float conv_out(const ConvIn &c) {
    float acc = c.bias;
#pragma unroll
    for (int r = 0; r < kW - 1; ++r) acc = fmaf(c.w[r], c.h[r], acc);
    acc = fmaf(c.w[kW - 1], c.x, acc);
    return silu_bf16out(acc);
}

// Shifted history: the last W-1 pre-activation inputs, oldest first.
__device__ __forceinline__ void store_conv_state(const ConvIn &c, __nv_bfloat16 *cpool,
                                                 int64_t cslot, int C, int ch) {
#pragma unroll
    for (int r = 0; r < kW - 2; ++r)
        cpool[(cslot * (kW - 1) + r) * C + ch] = __float2bfloat16_rn(c.h[r + 1]);
    cpool[(cslot * (kW - 1) + kW - 2) * C + ch] = __float2bfloat16_rn(c.x);
}

template <int LPR>
__device__ __forceinline__ float wsum(float v) {
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float dot4(float4 a, float4 b) {
    return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}

struct GroupIn {          // one group's raw inputs, as this thread needs them
    ConvIn qk, vv;        // q|k channel t, v channel t
    float a, b;           // gate inputs of V head (t % grp) (threads < grp)
    int64_t slot;
};

__global__ void __launch_bounds__(kThreads, kCtasPerSm)
decode_step_kernel(const __nv_bfloat16 *__restrict__ x, int64_t xs,
                   const __nv_bfloat16 *__restrict__ cw, const __nv_bfloat16 *__restrict__ cb,
                   __nv_bfloat16 *__restrict__ cpool, const __nv_bfloat16 *__restrict__ a,
                   const __nv_bfloat16 *__restrict__ b, const float *__restrict__ A_log,
                   const float *__restrict__ dt_bias, int n_seqs, int hqk, int hv, int C,
                   float scale, float *__restrict__ pool, int64_t n_slots,
                   const int32_t *__restrict__ idx, __nv_bfloat16 *__restrict__ o) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    __shared__ uint64_t full[2];
    // per-group vectors, double-buffered: group G + 1's are computed while
    // group G's items stream
    __shared__ float q_s[2][128], k_s[2][128], v_s[2][128 * kMaxGrp], g_s[2][kMaxGrp],
        b_s[2][kMaxGrp];
    __shared__ float red_s[8], o_s[kRows];
    __shared__ int abort_flag;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int grp = hv / hqk;
    const int n_groups = n_seqs * hqk;
    const int nq = hqk * 128;                    // q channels; k follows, then v
    if (tid == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    volatile int *abort = &abort_flag;

    auto live_slot = [&](int64_t slot) { return slot >= 0 && slot < n_slots; };
    auto load_group = [&](int gi, GroupIn &in) {
        const int i = gi / hqk, hq = gi - i * hqk;
        in.slot = idx[i];
        const __nv_bfloat16 *xr = x + (int64_t)i * xs;
        const int qk_ch = tid < 128 ? hq * 128 + tid : nq + hq * 128 + (tid - 128);
        const int v_ch = 2 * nq + hq * grp * 128 + tid;          // grp * 128 <= 256 channels
        if (live_slot(in.slot)) {
            load_conv(in.qk, xr, cw, cb, cpool, in.slot, C, qk_ch);
            if (tid < grp * 128) load_conv(in.vv, xr, cw, cb, cpool, in.slot, C, v_ch);
        }
        if (tid < grp) {
            const int h = hq * grp + tid;
            in.a = bf(a + (int64_t)i * hv + h);
            in.b = bf(b + (int64_t)i * hv + h);
        }
    };
    // conv + SiLU of this thread's q|k and v channels, their conv states, the
    // gates and the q / k norms of group gi into buffer bb (all threads)
    auto prologue = [&](int gi, const GroupIn &in, int bb) {
        if (!live_slot(in.slot)) return;         // uniform over the CTA
        const int hq = gi % hqk;
        const float yq = conv_out(in.qk);
        store_conv_state(in.qk, cpool, in.slot, C,
                         tid < 128 ? hq * 128 + tid : nq + hq * 128 + (tid - 128));
        const float ss = wsum<32>(yq * yq);       // q rows: warps 0..3, k rows: 4..7
        if (lane == 0) red_s[warp] = ss;
        if (tid < grp * 128) {
            v_s[bb][tid] = conv_out(in.vv);
            store_conv_state(in.vv, cpool, in.slot, C, 2 * nq + hq * grp * 128 + tid);
        }
        if (tid < grp) {
            const int h = hq * grp + tid;
            g_s[bb][tid] = -__expf(A_log[h]) * softplus_f(in.a + dt_bias[h]);
            b_s[bb][tid] = 1.f / (1.f + __expf(-in.b));
        }
        __syncthreads();
        const float nrm = rsqrtf((tid < 128 ? red_s[0] + red_s[1] + red_s[2] + red_s[3]
                                            : red_s[4] + red_s[5] + red_s[6] + red_s[7]) +
                                 kL2Eps);
        if (tid < 128) q_s[bb][tid] = yq * nrm; else k_s[bb][tid - 128] = yq * nrm;
        __syncthreads();                          // red_s is reused, the vectors are read
    };
    auto state_ptr = [&](int64_t slot, int h, int part) {
        return pool + ((slot * hv + h) * (int64_t)128 + part * kRows) * 128;
    };
    // item k of group gi: V head hq * grp + k / 2, rows 64 (k % 2) ..
    auto issue_state = [&](int gi, int64_t slot, int kk, int s) {
        const int hq = gi % hqk;
        mbar_arrive_expect_tx(&full[s], kStageBytes);
        bulk_load(smem_raw + s * kStageBytes, state_ptr(slot, hq * grp + (kk >> 1), kk & 1),
                  kStageBytes, &full[s]);
    };
    int ph[2] = {0, 0};
    int n = 0;                                  // items processed by this CTA
    int gi = blockIdx.x;
    GroupIn cur, nxt;
    if (gi < n_groups) {
        load_group(gi, cur);
        if (live_slot(cur.slot)) {
            if (tid == 0) issue_state(gi, cur.slot, 0, 0);
            ++ph[0];
        }
        prologue(gi, cur, 0);
    }
    for (int it = 0; gi < n_groups; gi += gridDim.x, ++it) {
        const int i = gi / hqk, hq = gi - i * hqk;
        const int bb = it & 1;
        const bool live = live_slot(cur.slot);
        if (cur.slot >= n_slots && tid == 0) flag_status(GDN_DEVSTAT_BAD_INDEX);
        const int gn = gi + gridDim.x;
        if (gn < n_groups) load_group(gn, nxt);   // into registers; used after item 0
        const float4 q4 = *reinterpret_cast<const float4 *>(q_s[bb] + 4 * lane);
        const float4 k4 = *reinterpret_cast<const float4 *>(k_s[bb] + 4 * lane);
        const float kq = wsum<32>(dot4(k4, q4));
        for (int kk = 0; kk < 2 * grp; ++kk, ++n) {
            const int s = n & 1;
            const int h = hq * grp + (kk >> 1), part = kk & 1;
            {   // prefetch the next item's state (this group's next item, or the
                // next group's first) into the other stage; every thread keeps
                // the same count of loads per stage
                const bool in_group = kk + 1 < 2 * grp;
                const int64_t sn = in_group ? cur.slot : (gn < n_groups ? nxt.slot : -1);
                if (live_slot(sn)) {
                    if (tid == 0) {
                        bulk_wait_read_all();    // the stage's last store has read it
                        issue_state(in_group ? gi : gn, sn, in_group ? kk + 1 : 0, s ^ 1);
                    }
                    ++ph[s ^ 1];
                }
            }
            float *st = reinterpret_cast<float *>(smem_raw + s * kStageBytes);
            if (live) {
                mbar_wait(&full[s], (ph[s] - 1) & 1, abort);
                const float alpha = __expf(g_s[bb][kk >> 1]);
                const float beta_ = b_s[bb][kk >> 1];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int r = 8 * warp + j;
                    float4 *sp = reinterpret_cast<float4 *>(st + r * 128) + lane;
                    const float4 sv = *sp;
                    const float sk = wsum<32>(dot4(sv, k4));
                    const float sq = wsum<32>(dot4(sv, q4));
                    const float u = beta_ * (v_s[bb][(kk >> 1) * 128 + part * kRows + r] - alpha * sk);
                    *sp = make_float4(fmaf(alpha, sv.x, u * k4.x), fmaf(alpha, sv.y, u * k4.y),
                                      fmaf(alpha, sv.z, u * k4.z), fmaf(alpha, sv.w, u * k4.w));
                    if (lane == 0) o_s[r] = scale * fmaf(alpha, sq, u * kq);
                }
                fence_async_smem();
            } else if (lane == 0) {
#pragma unroll
                for (int j = 0; j < 8; ++j) o_s[8 * warp + j] = 0.f;
            }
            __syncthreads();
            if (live && tid == 0) {
                bulk_store(state_ptr(cur.slot, h, part), st, kStageBytes);
                bulk_commit();
            }
            if (tid < kRows)
                o[((int64_t)i * hv + h) * 128 + part * kRows + tid] = __float2bfloat16_rn(o_s[tid]);
            __syncthreads();
            if (kk == 0 && gn < n_groups) prologue(gn, nxt, bb ^ 1);   // overlaps the streaming
        }
        cur = nxt;
    }
    if (tid == 0) {
        bulk_wait_read_all();
        if (abort_flag) flag_status(GDN_DEVSTAT_TIMEOUT);
    }
}

// ------------------------------------------------- with a workspace --
// The same step as two kernels: this front kernel (conv update + SiLU of the
// raw stream into y, the gates into g / beta, all in the workspace), then the
// streaming decode kernel launched behind it (programmatic dependent launch),
// which L2-normalises q and k itself.  Every channel is convolved once, so
// the in-place conv state update needs no grouping, and the decode streams
// its state blocks in the pool's order.
constexpr int kFrontThreads = 256;
constexpr int kFrontVec = 8;                 // channels per thread: one 16-byte vector

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__global__ void __launch_bounds__(kFrontThreads)
decode_front_kernel(const __nv_bfloat16 *__restrict__ x, int64_t xs,
                    const __nv_bfloat16 *__restrict__ cw, const __nv_bfloat16 *__restrict__ cb,
                    __nv_bfloat16 *__restrict__ cpool, const __nv_bfloat16 *__restrict__ a,
                    const __nv_bfloat16 *__restrict__ b, const float *__restrict__ A_log,
                    const float *__restrict__ dt_bias, int n_seqs, int hv, int C,
                    int64_t n_slots, const int32_t *__restrict__ idx,
                    __nv_bfloat16 *__restrict__ y, float *__restrict__ g_out,
                    float *__restrict__ b_out) {
    // the decode kernel behind this one may start placing its CTAs (they
    // fetch their first state, then wait for this grid to complete)
    griddep_launch();
    const int per_seq = C / kFrontVec;
    const int64_t gt = (int64_t)blockIdx.x * kFrontThreads + threadIdx.x;
    const int i = (int)(gt / per_seq);
    const int v8 = (int)(gt - (int64_t)i * per_seq);
    if (i < n_seqs) {
        const int64_t slot = idx[i];
        // everything but the conv state is requested before the slot id is back
        const int ch = v8 * kFrontVec;
        const uint4 xv = *reinterpret_cast<const uint4 *>(x + (int64_t)i * xs + ch);
        const uint4 *wp = reinterpret_cast<const uint4 *>(cw + (int64_t)ch * kW);
        const uint4 wv[4] = {wp[0], wp[1], wp[2], wp[3]};   // 8 channels x 4 taps
        uint4 bv = make_uint4(0u, 0u, 0u, 0u);
        if (cb) bv = *reinterpret_cast<const uint4 *>(cb + ch);
        if (v8 < hv) {    // the gates of (i, head v8)
            const int64_t r = (int64_t)i * hv + v8;
            g_out[r] = -__expf(A_log[v8]) * softplus_f(bf(a + r) + dt_bias[v8]);
            b_out[r] = 1.f / (1.f + __expf(-bf(b + r)));
        }
        if (slot >= 0 && slot < n_slots) {
            __nv_bfloat16 *cs = cpool + slot * (kW - 1) * C + ch;
            const uint4 h0 = *reinterpret_cast<const uint4 *>(cs);
            const uint4 h1 = *reinterpret_cast<const uint4 *>(cs + C);
            const uint4 h2 = *reinterpret_cast<const uint4 *>(cs + 2 * C);
            const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, w0[4] = {h0.x, h0.y, h0.z, h0.w},
                           w1[4] = {h1.x, h1.y, h1.z, h1.w}, w2[4] = {h2.x, h2.y, h2.z, h2.w},
                           bw[4] = {bv.x, bv.y, bv.z, bv.w};
            const uint32_t *tw = reinterpret_cast<const uint32_t *>(wv);   // taps: 2 words per channel
            uint32_t out[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {          // channels 2e, 2e + 1
                float r2[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int c = 2 * e + u;
                    const uint32_t t01 = tw[2 * c], t23 = tw[2 * c + 1];
                    const float xin = u ? bf_hi(xw[e]) : bf_lo(xw[e]);
                    const float s0 = u ? bf_hi(w0[e]) : bf_lo(w0[e]);
                    const float s1 = u ? bf_hi(w1[e]) : bf_lo(w1[e]);
                    const float s2 = u ? bf_hi(w2[e]) : bf_lo(w2[e]);
                    float acc = u ? bf_hi(bw[e]) : bf_lo(bw[e]);
                    acc = fmaf(bf_lo(t01), s0, acc);
                    acc = fmaf(bf_hi(t01), s1, acc);
                    acc = fmaf(bf_lo(t23), s2, acc);
                    acc = fmaf(bf_hi(t23), xin, acc);
                    r2[u] = silu_bf16out(acc);
                }
                out[e] = pack_bf16(r2[0], r2[1]);
            }
            *reinterpret_cast<uint4 *>(y + (int64_t)i * C + ch) = make_uint4(out[0], out[1], out[2], out[3]);
            // the state shifts by one input: the raw bf16 values move as they are
            *reinterpret_cast<uint4 *>(cs) = h1;
            *reinterpret_cast<uint4 *>(cs + C) = h2;
            *reinterpret_cast<uint4 *>(cs + 2 * C) = xv;
        } else if (slot >= n_slots && v8 == 0) {
            flag_status(GDN_DEVSTAT_BAD_INDEX);
        }
    }
}

__host__ __device__ inline size_t align256(size_t n) { return (n + 255) / 256 * 256; }

}  // namespace dstep
}  // namespace gdn

using namespace gdn;

extern "C" size_t gdn_decode_step_workspace_size(int32_t n_seqs, int32_t hqk, int32_t hv) {
    if (n_seqs <= 0 || hqk <= 0 || hv <= 0) return 0;
    const size_t C = 2 * (size_t)hqk * 128 + (size_t)hv * 128;
    return dstep::align256((size_t)n_seqs * C * 2) + 2 * dstep::align256((size_t)n_seqs * hv * 4);
}

extern "C" gdn_status gdn_decode_step_fused(const void *x, int64_t x_row_stride,
                                            const void *conv_weight, const void *conv_bias,
                                            void *conv_state_pool, const void *a, const void *b,
                                            const float *A_log, const float *dt_bias,
                                            int32_t n_seqs, int32_t hqk, int32_t hv, float scale,
                                            float *state_pool, int64_t n_slots,
                                            const int32_t *state_indices, void *workspace,
                                            size_t workspace_bytes, void *o, void *stream) {
    GDN_REQUIRE(n_seqs >= 0 && hqk > 0 && hv > 0 && n_slots >= 0, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(hv % hqk == 0, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(hv / hqk <= dstep::kMaxGrp, GDN_ERR_UNSUPPORTED);
    if (n_seqs == 0) return GDN_OK;
    GDN_REQUIRE((int64_t)n_seqs * hqk < (1ll << 31), GDN_ERR_UNSUPPORTED);
    GDN_REQUIRE(x && conv_weight && conv_state_pool && a && b && A_log && dt_bias && state_pool &&
                    state_indices && o,
                GDN_ERR_INVALID_ARG);
    const int C = 2 * hqk * 128 + hv * 128;
    GDN_REQUIRE(x_row_stride >= C, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(((uintptr_t)conv_weight % 8) == 0 && ((uintptr_t)state_pool % 16) == 0,
                GDN_ERR_INVALID_ARG);
    cudaStream_t s = (cudaStream_t)stream;
    const size_t ws_need = gdn_decode_step_workspace_size(n_seqs, hqk, hv);
    const bool two_kernels =
        workspace && workspace_bytes >= ws_need && ((uintptr_t)workspace % 256) == 0 &&
        ((uintptr_t)x % 16) == 0 && (x_row_stride % 8) == 0 &&
        ((uintptr_t)conv_weight % 16) == 0 && ((uintptr_t)conv_state_pool % 16) == 0 &&
        (!conv_bias || ((uintptr_t)conv_bias % 16) == 0);
    if (two_kernels) {
        uint8_t *ws = (uint8_t *)workspace;
        __nv_bfloat16 *y = (__nv_bfloat16 *)ws;
        float *g = (float *)(ws + dstep::align256((size_t)n_seqs * C * 2));
        float *beta = g + dstep::align256((size_t)n_seqs * hv * 4) / 4;
        const int64_t threads = (int64_t)n_seqs * (C / dstep::kFrontVec);
        dstep::decode_front_kernel<<<(unsigned)((threads + dstep::kFrontThreads - 1) /
                                                dstep::kFrontThreads),
                                     dstep::kFrontThreads, 0, s>>>(
            (const __nv_bfloat16 *)x, x_row_stride, (const __nv_bfloat16 *)conv_weight,
            (const __nv_bfloat16 *)conv_bias, (__nv_bfloat16 *)conv_state_pool,
            (const __nv_bfloat16 *)a, (const __nv_bfloat16 *)b, A_log, dt_bias, n_seqs, hv, C,
            n_slots, state_indices, y, g, beta);
        gdn_status st = launch_status();
        if (st != GDN_OK) return st;
        const int nq = hqk * 128;
        cudaError_t e = launch_decode_stream_after(y, C, y + nq, C, y + 2 * nq, C, g, beta, n_seqs,
                                                   hqk, hv, scale, state_pool, n_slots,
                                                   state_indices, (__nv_bfloat16 *)o, s);
        if (e != cudaSuccess) {
            set_last_cuda_error(e);
            return GDN_ERR_LAUNCH;
        }
        return GDN_OK;
    }
    const int n_groups = n_seqs * hqk;
    const int grid = std::min(n_groups, sm_count() * dstep::kCtasPerSm);
    cudaError_t e = cudaFuncSetAttribute(dstep::decode_step_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(2 * dstep::kStageBytes));
    if (e != cudaSuccess) {
        set_last_cuda_error(e);
        return GDN_ERR_LAUNCH;
    }
    dstep::decode_step_kernel<<<grid, dstep::kThreads, 2 * dstep::kStageBytes, s>>>(
        (const __nv_bfloat16 *)x, x_row_stride, (const __nv_bfloat16 *)conv_weight,
        (const __nv_bfloat16 *)conv_bias, (__nv_bfloat16 *)conv_state_pool,
        (const __nv_bfloat16 *)a, (const __nv_bfloat16 *)b, A_log, dt_bias, n_seqs, hqk, hv, C,
        scale, state_pool, n_slots, state_indices, (__nv_bfloat16 *)o);
    return launch_status();
}
