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

}  // namespace dstep
}  // namespace gdn

using namespace gdn;

extern "C" gdn_status gdn_decode_step_fused(const void *x, int64_t x_row_stride,
                                            const void *conv_weight, const void *conv_bias,
                                            void *conv_state_pool, const void *a, const void *b,
                                            const float *A_log, const float *dt_bias,
                                            int32_t n_seqs, int32_t hqk, int32_t hv, float scale,
                                            float *state_pool, int64_t n_slots,
                                            const int32_t *state_indices, void *o, void *stream) {
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
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int n_groups = n_seqs * hqk;
    const int grid = std::min(n_groups, sms * dstep::kCtasPerSm);
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
