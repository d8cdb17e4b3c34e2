// One MTP step of the layer in one kernel (fusion of the "causal 1D
// convolution", "fused GDN gating" and "fused recurrent GDN" kernels the
// Qwen3next pages name, for the MTP draft step whose linear-attention states
// are copied per draft token, "[model] support Qwen3next", Highlights).  For
// sequence i with tps new tokens (row i * tps + t):
//   the causal conv update (width 4) + SiLU of the raw q|k|v stream, the
//     conv state after token t written to slot snap[i][t] of the conv pool;
//   the gates, the q / k L2 norms;
//   the gated delta rule over the tps tokens, the state after token t
//     written to slot snap[i][t] of the state pool.
// The source slot idx[i] of both pools is only read.  The result equals
// causal_conv1d_update (with snapshots) + gdn_gating + gdn_decode_recurrent
// (with snapshots).
//
// One CTA of 256 threads per (sequence, V head, row half), as the MTP decode
// kernel: the half-state (64 rows) stays in registers across the tokens.  A
// prologue convolves this CTA's channels for every token into shared memory:
// the 256 q|k channels of its QK head and its 64 v channels.  Every CTA of a
// QK head's group computes the q|k conv; the one with V head h % grp == 0 and
// row half 0 writes their conv snapshots, each CTA those of its v channels.
// With snapshots no conv state is updated in place, so CTAs that share the
// q|k channels never race.
#include "common.cuh"

namespace gdn {

GDN_DECLARE_STATUS_WORD(g_status_mtp_step)
GDN_STATUS_READER(read_status_mtp_step, g_status_mtp_step)

namespace mtp {

constexpr int kThreads = 256;
constexpr int kW = 4;                 // conv width
constexpr int kRows = 64;             // state rows per CTA
constexpr int kMaxTps = 16;
constexpr int kCh = 320;              // channels a CTA convolves: 128 q, 128 k, 64 v
constexpr int kPieces = kCh / 8;      // 16-byte pieces of one row of those channels
constexpr float kL2Eps = 1e-6f;

__device__ __forceinline__ float bf(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ float softplus_f(float x) { return x > 20.f ? x : log1pf(__expf(x)); }
__device__ __forceinline__ float dot4(float4 a, float4 b) {
    return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}
__device__ __forceinline__ float wsum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;\n" ::: "memory");
}

// The CTA's channel c (0..319: q of QK head hq, k of QK head hq, v rows r0..
// r0 + 63 of V head h) in the q|k|v stream.
__device__ __forceinline__ int stream_ch(int c, int hq, int nq, int h, int r0) {
    return c < 128 ? hq * 128 + c : c < 256 ? nq + hq * 128 + (c - 128) : 2 * nq + h * 128 + r0 + (c - 256);
}

// Rows [C] of the stream -> shared rows of the CTA's kCh channels: 16-byte
// async copies when the rows allow them, else element by element.
__device__ __forceinline__ void stage_rows(__nv_bfloat16 (*dst)[kCh], const __nv_bfloat16 *src,
                                           int64_t stride, int n_rows, bool vec, int hq, int nq,
                                           int h, int r0) {
    if (vec) {
        for (int e = threadIdx.x; e < n_rows * kPieces; e += kThreads) {
            const int r = e / kPieces, p = e - r * kPieces;
            cp_async16(&dst[r][p * 8], src + (int64_t)r * stride + stream_ch(p * 8, hq, nq, h, r0));
        }
    } else {
        for (int e = threadIdx.x; e < n_rows * kCh; e += kThreads) {
            const int r = e / kCh, c = e - r * kCh;
            dst[r][c] = src[(int64_t)r * stride + stream_ch(c, hq, nq, h, r0)];
        }
    }
}

// Channel c over the tokens: out[t] = SiLU(conv) from the staged history and
// inputs.
__device__ __forceinline__ void conv_channel(const __nv_bfloat16 (*hist)[kCh],
                                             const __nv_bfloat16 (*xin)[kCh], int c, uint2 wv,
                                             float bias, int tps, float *out, int out_stride) {
    float h0 = __bfloat162float(hist[0][c]);
    float h1 = __bfloat162float(hist[1][c]);
    float h2 = __bfloat162float(hist[2][c]);
    const float2 w01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&wv.x));
    const float2 w23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&wv.y));
    for (int t = 0; t < tps; ++t) {
        const float xt = __bfloat162float(xin[t][c]);
        float acc = fmaf(w01.x, h0, bias);
        acc = fmaf(w01.y, h1, acc);
        acc = fmaf(w23.x, h2, acc);
        acc = fmaf(w23.y, xt, acc);
        out[t * out_stride] = silu_bf16out(acc);
        h0 = h1;
        h1 = h2;
        h2 = xt;
    }
}

__global__ void __launch_bounds__(kThreads, 4)   // 64 registers: 4 CTAs per SM
mtp_step_kernel(const __nv_bfloat16 *__restrict__ x, int64_t xs, bool x_vec,
                const __nv_bfloat16 *__restrict__ cw, const __nv_bfloat16 *__restrict__ cb,
                __nv_bfloat16 *__restrict__ cpool, const __nv_bfloat16 *__restrict__ a,
                const __nv_bfloat16 *__restrict__ bg, const float *__restrict__ A_log,
                const float *__restrict__ dt_bias, int tps, int hqk, int hv, int C, float scale,
                float *__restrict__ pool, int64_t n_slots, const int32_t *__restrict__ idx,
                const int32_t *__restrict__ snap, __nv_bfloat16 *__restrict__ o) {
    __shared__ __align__(16) __nv_bfloat16 x_s[kMaxTps][kCh];
    __shared__ __align__(16) __nv_bfloat16 h_s[kW - 1][kCh];
    __shared__ float o_s[kMaxTps][kRows];
    __shared__ float v_s[kMaxTps][kRows];
    __shared__ __align__(16) float q_s[kMaxTps][128];
    __shared__ __align__(16) float k_s[kMaxTps][128];
    __shared__ float a_s[kMaxTps], b_s[kMaxTps];
    __shared__ int64_t sn_s[kMaxTps];

    griddep_launch();   // an accept copy behind this kernel may be set up meanwhile
    const int part = blockIdx.x & 1;
    const int ih = blockIdx.x >> 1;
    const int i = ih / hv;
    const int h = ih - i * hv;
    const int grp = hv / hqk;
    const int hq = h / grp;
    const int r0 = part * kRows;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int col = lane * 4;
    const int nq = hqk * 128;
    const int tid = threadIdx.x;

    // everything that does not depend on the slot is requested first
    const int64_t slot = idx[i];
    stage_rows(x_s, x + (int64_t)i * tps * xs, xs, tps, x_vec, hq, nq, h, r0);
    const int chq = stream_ch(tid, hq, nq, h, r0);              // q|k channel of this thread
    const int chv = stream_ch(256 + (tid & 63), hq, nq, h, r0);  // v channel (threads < 64)
    const uint2 wq = *reinterpret_cast<const uint2 *>(cw + (int64_t)chq * kW);
    const uint2 wv = *reinterpret_cast<const uint2 *>(cw + (int64_t)chv * kW);
    const float bq = cb ? bf(cb + chq) : 0.f;
    const float bv = cb ? bf(cb + chv) : 0.f;
    float ga = 0.f, gb = 0.f;
    int64_t snt = -1;
    if (tid < tps) {
        const int64_t row = (int64_t)i * tps + tid;
        ga = bf(a + row * hv + h);
        gb = bf(bg + row * hv + h);
        snt = snap[(int64_t)i * tps + tid];
    }

    const bool live = slot >= 0 && slot < n_slots;
    if (slot >= n_slots && tid == 0 && part == 0) flag_status(GDN_DEVSTAT_BAD_INDEX);
    if (!live) {   // padding: o rows zero, neither pool touched
        cp_async_wait_all();
        for (int e = tid; e < tps * kRows; e += kThreads) {
            const int t = e / kRows, r = e - t * kRows;
            o[(((int64_t)i * tps + t) * hv + h) * 128 + r0 + r] = __float2bfloat16_rn(0.f);
        }
        return;
    }

    // the half-state: row 8 p + warp of this CTA's rows, columns 4 lane ..
    float *src = pool + ((slot * hv + h) * (int64_t)128 + r0) * 128;
    float4 st[8];
#pragma unroll
    for (int p = 0; p < 8; ++p)
        st[p] = __ldcs(reinterpret_cast<const float4 *>(src + (int64_t)(8 * p + warp) * 128 + col));
    stage_rows(h_s, cpool + slot * (kW - 1) * C, C, kW - 1, true, hq, nq, h, r0);

    if (tid < tps) {
        const float g = -__expf(A_log[h]) * softplus_f(ga + dt_bias[h]);
        a_s[tid] = __expf(g);
        b_s[tid] = 1.f / (1.f + __expf(-gb));
        if (snt >= n_slots) {
            if (part == 0) flag_status(GDN_DEVSTAT_BAD_INDEX);
            snt = -1;
        }
        sn_s[tid] = snt;
    }
    cp_async_wait_all();
    __syncthreads();

    // The conv state after token t is window rows t + 1 .. t + 3 of
    // [history rows 0..2, x rows 0..tps-1], all staged: each snapshot row is a
    // copy of a staged row, 16 bytes at a time.  The q|k vectors of QK head hq
    // are split over the 2 grp CTAs that share it; each CTA writes those of
    // its own v channels.
    {
        const int j = (h - hq * grp) * 2 + part;
        const int n_units = tps * (kW - 1) * kPieces;
        for (int e = tid; e < n_units; e += kThreads) {
            const int t = e / ((kW - 1) * kPieces);
            const int rem = e - t * ((kW - 1) * kPieces);
            const int r = rem / kPieces, u = rem - r * kPieces;   // row, 16-byte piece
            const int64_t d = sn_s[t];
            if (d < 0 || (u < 32 && (u * 2 * grp) / 32 != j)) continue;
            const int w = t + 1 + r;                              // window row
            const uint4 val = w < kW - 1 ? *reinterpret_cast<const uint4 *>(&h_s[w][u * 8])
                                         : *reinterpret_cast<const uint4 *>(&x_s[w - (kW - 1)][u * 8]);
            *reinterpret_cast<uint4 *>(cpool + (d * (kW - 1) + r) * C +
                                       stream_ch(u * 8, hq, nq, h, r0)) = val;
        }
    }
    // conv + SiLU of the CTA's channels
    conv_channel(h_s, x_s, tid, wq, bq, tps, tid < 128 ? &q_s[0][tid] : &k_s[0][tid - 128], 128);
    if (tid < kRows) conv_channel(h_s, x_s, 256 + tid, wv, bv, tps, &v_s[0][tid], kRows);
    __syncthreads();

    for (int t = 0; t < tps; ++t) {
        float4 q4 = *reinterpret_cast<const float4 *>(&q_s[t][col]);
        float4 k4 = *reinterpret_cast<const float4 *>(&k_s[t][col]);
        const float qn = rsqrtf(wsum(dot4(q4, q4)) + kL2Eps);
        const float kn = rsqrtf(wsum(dot4(k4, k4)) + kL2Eps);
        q4 = make_float4(q4.x * qn, q4.y * qn, q4.z * qn, q4.w * qn);
        k4 = make_float4(k4.x * kn, k4.y * kn, k4.z * kn, k4.w * kn);
        const float kq = wsum(dot4(k4, q4));
        const float alpha = a_s[t];
        const float beta = b_s[t];
        // the dot products S k, S q of four of the warp's rows reduced
        // together (lane l ends with value l mod 8), then read back
#pragma unroll
        for (int p0 = 0; p0 < 8; p0 += 4) {
            float pv[8];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                pv[p] = dot4(st[p0 + p], k4);
                pv[4 + p] = dot4(st[p0 + p], q4);
            }
            reduce_scatter_step<8>(pv, lane);
            reduce_scatter_step<4>(pv, lane);
            reduce_scatter_step<2>(pv, lane);
            float tot = pv[0] + __shfl_xor_sync(0xffffffffu, pv[0], 8);
            tot += __shfl_xor_sync(0xffffffffu, tot, 16);
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const int r = 8 * (p0 + p) + warp;
                const float sk = __shfl_sync(0xffffffffu, tot, p);
                const float sq = __shfl_sync(0xffffffffu, tot, 4 + p);
                const float4 s = st[p0 + p];
                const float u = beta * (v_s[t][r] - alpha * sk);
                st[p0 + p] = make_float4(fmaf(alpha, s.x, u * k4.x), fmaf(alpha, s.y, u * k4.y),
                                         fmaf(alpha, s.z, u * k4.z), fmaf(alpha, s.w, u * k4.w));
                if (lane == 0) o_s[t][r] = scale * fmaf(alpha, sq, u * kq);
            }
        }
        const int64_t d = sn_s[t];
        if (d >= 0) {
            float *dst = pool + ((d * hv + h) * (int64_t)128 + r0) * 128;
#pragma unroll
            for (int p = 0; p < 8; ++p)
                __stcs(reinterpret_cast<float4 *>(dst + (int64_t)(8 * p + warp) * 128 + col), st[p]);
        }
    }
    __syncthreads();
    for (int e = tid; e < tps * kRows; e += kThreads) {
        const int t = e / kRows, r = e - t * kRows;
        o[(((int64_t)i * tps + t) * hv + h) * 128 + r0 + r] = __float2bfloat16_rn(o_s[t][r]);
    }
}

}  // namespace mtp
}  // namespace gdn

using namespace gdn;

extern "C" gdn_status gdn_mtp_step_fused(const void *x, int64_t x_row_stride,
                                         const void *conv_weight, const void *conv_bias,
                                         void *conv_state_pool, const void *a, const void *b,
                                         const float *A_log, const float *dt_bias,
                                         int32_t n_seqs, int32_t tokens_per_seq, int32_t hqk,
                                         int32_t hv, float scale, float *state_pool,
                                         int64_t n_slots, const int32_t *state_indices,
                                         const int32_t *snap_indices, void *o, void *stream) {
    GDN_REQUIRE(n_seqs >= 0 && hqk > 0 && hv > 0 && n_slots >= 0, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(hv % hqk == 0, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(tokens_per_seq >= 1 && tokens_per_seq <= mtp::kMaxTps, GDN_ERR_UNSUPPORTED);
    if (n_seqs == 0) return GDN_OK;
    GDN_REQUIRE((int64_t)n_seqs * hv * 2 < (1ll << 31), GDN_ERR_UNSUPPORTED);
    GDN_REQUIRE(x && conv_weight && conv_state_pool && a && b && A_log && dt_bias && state_pool &&
                    state_indices && snap_indices && o,
                GDN_ERR_INVALID_ARG);
    const int C = 2 * hqk * 128 + hv * 128;
    GDN_REQUIRE(x_row_stride >= C, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(((uintptr_t)conv_weight % 8) == 0 && ((uintptr_t)state_pool % 16) == 0 &&
                    ((uintptr_t)conv_state_pool % 16) == 0,
                GDN_ERR_INVALID_ARG);
    const bool x_vec = ((uintptr_t)x % 16) == 0 && (x_row_stride % 8) == 0;
    mtp::mtp_step_kernel<<<(unsigned)((int64_t)n_seqs * hv * 2), mtp::kThreads, 0,
                           (cudaStream_t)stream>>>(
        (const __nv_bfloat16 *)x, x_row_stride, x_vec, (const __nv_bfloat16 *)conv_weight,
        (const __nv_bfloat16 *)conv_bias, (__nv_bfloat16 *)conv_state_pool,
        (const __nv_bfloat16 *)a, (const __nv_bfloat16 *)b, A_log, dt_bias, tokens_per_seq, hqk,
        hv, C, scale, state_pool, n_slots, state_indices, snap_indices, (__nv_bfloat16 *)o);
    return launch_status();
}
