// Recurrent decode and MTP multi-token decode of the gated delta rule
// ("fused recurrent GDN", "[model] support Qwen3next", Highlights; the MTP
// linear-attention state copying of the same page's Highlights).
//
// One CTA per (sequence, V head).  The dv x dk fp32 state is streamed from
// its slot into registers with 16-byte loads (lane l of a row group owns
// columns [4l, 4l+4) of its rows), kept there across the tokens of the
// sequence, and written once per token that has a destination slot.  Per
// token and row the two dot products S k and S q are warp-shuffle
// reductions over the row's lanes:
//   u   = beta (v - alpha S k)
//   S  <- alpha S + u k^T
//   o   = scale (alpha S_old q + u (k . q))   (= scale S_new q)
// With GATED (one CTA per state only) the kernel writes
// y = o / sqrt(mean(o^2) + eps) * w * SiLU(z) ("gated RMSNorm", same pages)
// instead of o.
#include <algorithm>

#include "common.cuh"
#include "tc.cuh"

namespace gdn {

GDN_DECLARE_STATUS_WORD(g_status_decode)
GDN_STATUS_READER(read_status_decode, g_status_decode)

constexpr int kDecWarps = 8;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kMaxDv = 128;
constexpr int kMaxTps = 16;
constexpr float kL2Eps = 1e-6f;

template <int LPR>
__device__ __forceinline__ float row_sum(float v) {
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float dot4(float4 a, float4 b) {
    return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}

// SPLIT CTAs share one (sequence, V head): CTA `part` owns the state rows
// [part*rows, (part+1)*rows).  Fewer registers per thread, more resident CTAs.
template <int DK, int SPLIT, typename T, bool GATED>
__global__ void __launch_bounds__(kDecThreads, SPLIT == 2 ? 4 : 1)   // split: 64 registers
decode_kernel(const T *__restrict__ q, int64_t qs, const T *__restrict__ k, int64_t ks,
              const T *__restrict__ v, int64_t vs, const float *__restrict__ g,
              const float *__restrict__ beta, int tps, int hv, int grp, int dv, float scale,
              int l2norm, float *__restrict__ pool, int64_t n_slots,
              const int32_t *__restrict__ idx, const int32_t *__restrict__ snap,
              const T *__restrict__ z, int64_t zs, const float *__restrict__ nw, float neps,
              T *__restrict__ o) {
    constexpr int LPR = DK / 4;                     // lanes per state row
    constexpr int RPW = 32 / LPR;                   // rows per warp per pass
    constexpr int RPP = RPW * kDecWarps;            // rows per pass
    constexpr int kMaxRows = kMaxDv / SPLIT;
    constexpr int NP = (kMaxRows + RPP - 1) / RPP;  // passes covering this CTA's rows

    __shared__ float o_s[kMaxTps][kMaxRows];
    __shared__ float v_s[kMaxTps][kMaxRows];
    // every token's q, k (this QK head), exp(g) and beta, staged once with
    // the state load: no token waits on a global load
    __shared__ __align__(16) float q_s[kMaxTps][DK];
    __shared__ __align__(16) float k_s[kMaxTps][DK];
    __shared__ float a_s[kMaxTps], b_s[kMaxTps];

    const int part = blockIdx.x % SPLIT;
    const int ih = blockIdx.x / SPLIT;
    const int i = ih / hv;
    const int h = ih - i * hv;
    const int hq = h / grp;
    const int rows = (dv + SPLIT - 1) / SPLIT;
    const int r0 = part * rows;
    const int nr = max(0, min(dv, r0 + rows) - r0);   // rows of this CTA
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int col = (lane % LPR) * 4;
    const int sub = lane / LPR;

    const int64_t slot = idx[i];
    // the inputs need no slot id: they are staged while it is on its way
    for (int e = threadIdx.x; e < tps * nr; e += kDecThreads) {
        const int t = e / nr, r = e - t * nr;
        v_s[t][r] = Io<T>::load(v + ((int64_t)i * tps + t) * vs + (int64_t)h * dv + r0 + r);
    }
    for (int e = threadIdx.x; e < tps * DK; e += kDecThreads) {
        const int t = e / DK, c = e - t * DK;
        const int64_t row = (int64_t)i * tps + t;
        q_s[t][c] = Io<T>::load(q + row * qs + (int64_t)hq * DK + c);
        k_s[t][c] = Io<T>::load(k + row * ks + (int64_t)hq * DK + c);
    }
    if (threadIdx.x < tps) {
        const int64_t row = (int64_t)i * tps + threadIdx.x;
        a_s[threadIdx.x] = expf(g[row * hv + h]);
        b_s[threadIdx.x] = beta[row * hv + h];
    }
    const bool live = slot >= 0 && slot < n_slots;
    if (slot >= n_slots && threadIdx.x == 0 && part == 0) flag_status(GDN_DEVSTAT_BAD_INDEX);
    if (!live) {
        for (int e = threadIdx.x; e < tps * nr; e += kDecThreads) {
            const int t = e / nr, r = e - t * nr;
            Io<T>::store(o + (((int64_t)i * tps + t) * hv + h) * dv + r0 + r, 0.0f);
        }
        return;
    }

    float *src = pool + ((slot * hv + h) * (int64_t)dv + r0) * DK;
    float4 st[NP];
#pragma unroll
    for (int p = 0; p < NP; ++p) {
        const int r = p * RPP + warp * RPW + sub;
        st[p] = r < nr ? __ldcs(reinterpret_cast<const float4 *>(src + (int64_t)r * DK + col))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();

    for (int t = 0; t < tps; ++t) {
        const int64_t row = (int64_t)i * tps + t;
        float4 q4 = *reinterpret_cast<const float4 *>(&q_s[t][col]);
        float4 k4 = *reinterpret_cast<const float4 *>(&k_s[t][col]);
        if (l2norm) {
            const float qn = rsqrtf(row_sum<LPR>(dot4(q4, q4)) + kL2Eps);
            const float kn = rsqrtf(row_sum<LPR>(dot4(k4, k4)) + kL2Eps);
            q4 = make_float4(q4.x * qn, q4.y * qn, q4.z * qn, q4.w * qn);
            k4 = make_float4(k4.x * kn, k4.y * kn, k4.z * kn, k4.w * kn);
        }
        const float kq = row_sum<LPR>(dot4(k4, q4));
        const float alpha = a_s[t];
        const float b = b_s[t];
        if constexpr (LPR == 32 && NP == 8) {
            // a row per warp and pass: the dot products S k, S q of four of
            // the warp's rows reduced together (reduce-scatter: lane l ends
            // with value l mod 8), then read back -- 34 shuffles for the 8
            // rows instead of 80
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
                    const int r = (p0 + p) * RPP + warp;
                    const float sk = __shfl_sync(0xffffffffu, tot, p);
                    const float sq = __shfl_sync(0xffffffffu, tot, 4 + p);
                    if (r < nr) {
                        const float4 s = st[p0 + p];
                        const float u = b * (v_s[t][r] - alpha * sk);
                        st[p0 + p] = make_float4(fmaf(alpha, s.x, u * k4.x), fmaf(alpha, s.y, u * k4.y),
                                                 fmaf(alpha, s.z, u * k4.z), fmaf(alpha, s.w, u * k4.w));
                        if (lane == 0) o_s[t][r] = scale * fmaf(alpha, sq, u * kq);
                    }
                }
            }
        } else {
#pragma unroll
            for (int p = 0; p < NP; ++p) {
                const int r = p * RPP + warp * RPW + sub;
                if (p * RPP < nr) {                  // warp-uniform: shuffles stay converged
                    const float4 s = st[p];
                    const float sk = row_sum<LPR>(dot4(s, k4));
                    const float sq = row_sum<LPR>(dot4(s, q4));
                    if (r < nr) {
                        const float u = b * (v_s[t][r] - alpha * sk);
                        st[p] = make_float4(fmaf(alpha, s.x, u * k4.x), fmaf(alpha, s.y, u * k4.y),
                                            fmaf(alpha, s.z, u * k4.z), fmaf(alpha, s.w, u * k4.w));
                        if ((lane % LPR) == 0) o_s[t][r] = scale * fmaf(alpha, sq, u * kq);
                    }
                }
            }
        }
        if (snap) {
            const int64_t d = snap[row];
            if (d >= n_slots) {
                if (threadIdx.x == 0 && part == 0) flag_status(GDN_DEVSTAT_BAD_INDEX);
            } else if (d >= 0) {
                float *dst = pool + ((d * hv + h) * (int64_t)dv + r0) * DK;
#pragma unroll
                for (int p = 0; p < NP; ++p) {
                    const int r = p * RPP + warp * RPW + sub;
                    if (r < nr) __stcs(reinterpret_cast<float4 *>(dst + (int64_t)r * DK + col), st[p]);
                }
            }
        }
    }
    if (!snap) {
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            const int r = p * RPP + warp * RPW + sub;
            if (r < nr) __stcs(reinterpret_cast<float4 *>(src + (int64_t)r * DK + col), st[p]);
        }
    }
    __syncthreads();
    if constexpr (GATED) {
        static_assert(SPLIT == 1, "the norm needs every row of the state in this CTA");
        __shared__ float ss_s[kMaxTps];
        for (int t = warp; t < tps; t += kDecWarps) {
            float a = 0.f;
            for (int r = lane; r < nr; r += 32) a = fmaf(o_s[t][r], o_s[t][r], a);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
            if (lane == 0) ss_s[t] = a;
        }
        __syncthreads();
        for (int e = threadIdx.x; e < tps * nr; e += kDecThreads) {
            const int t = e / nr, r = e - t * nr;
            const int64_t row = (int64_t)i * tps + t;
            const float inv = rsqrtf(ss_s[t] / (float)dv + neps);
            const float zz = Io<T>::load(z + row * zs + (int64_t)h * dv + r0 + r);
            Io<T>::store(o + (row * hv + h) * dv + r0 + r, o_s[t][r] * inv * nw[r0 + r] * silu_for<T>(zz));
        }
    } else {
        for (int e = threadIdx.x; e < tps * nr; e += kDecThreads) {
            const int t = e / nr, r = e - t * nr;
            Io<T>::store(o + (((int64_t)i * tps + t) * hv + h) * dv + r0 + r, o_s[t][r]);
        }
    }
}


// ------------------------------------------------ streaming decode (T = 1)
using namespace tc;

// Persistent CTAs loop over (sequence, V head, row half) items of a 1-token
// decode with dk = dv = 128.  Each item's 64 x 128 fp32 half-state is one
// contiguous 32 KiB block of the pool: it is bulk-copied into one of two
// shared-memory stages while the CTA computes the previous item, updated in
// shared memory, and bulk-stored back, so a load and a store stay in flight
// through the compute.  The next item's q, k, v, g, beta are loaded into
// registers one item ahead.  Warp w updates rows 8w .. 8w + 7 of the item.
constexpr int kStrRows = 64;
constexpr uint32_t kStrBytes = kStrRows * 128 * 4;
constexpr int kStrCtasPerSm = 3;

template <typename T>
struct StrIn {            // one item's inputs, as this thread needs them
    float4 q4, k4;        // columns 4 lane .. 4 lane + 3
    float v;              // row 8 warp + lane (lanes 0..7)
    float g, b;
};

// kDyn: the items are handed out by a counter (atomicAdd on *ctr, zero at
// launch) instead of CTA b taking b, b + grid, ...; the kernel then reads
// nothing its primary grid writes and waits for that grid only at its end.
// Used when the decode runs beside the chain kernel of a mixed batch, on the
// SMs the chains leave free.
template <typename T, bool kDyn = false>
__global__ void __launch_bounds__(kDecThreads, kStrCtasPerSm)
decode_stream_kernel(const T *__restrict__ q, int64_t qs, const T *__restrict__ k, int64_t ks,
                     const T *__restrict__ v, int64_t vs, const float *__restrict__ g,
                     const float *__restrict__ beta, int n_items, int hv, int grp, float scale,
                     int l2norm, float *__restrict__ pool, int64_t n_slots,
                     const int32_t *__restrict__ idx, T *__restrict__ o, int *__restrict__ ctr) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    __shared__ uint64_t full[2];
    __shared__ float o_s[kStrRows];
    griddep_launch();   // a norm kernel behind this one may be set up meanwhile
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    volatile int *abort = &abort_flag;

    // item w: part = w % 2 (rows 64 part ..), (i, h) = w / 2
    auto slot_of = [&](int w, int &i, int &h, int &part) -> int64_t {
        part = w & 1;
        const int ih = w >> 1;
        i = ih / hv;
        h = ih - i * hv;
        return idx[i];
    };
    auto state_ptr = [&](int64_t slot, int h, int part) {
        return pool + ((slot * hv + h) * (int64_t)128 + part * kStrRows) * 128;
    };
    auto load_in = [&](int i, int h, int part, StrIn<T> &in) {
        const int hq = h / grp;
        in.q4 = load4(q + (int64_t)i * qs + (int64_t)hq * 128 + 4 * lane);
        in.k4 = load4(k + (int64_t)i * ks + (int64_t)hq * 128 + 4 * lane);
        in.v = lane < 8 ? Io<T>::load(v + (int64_t)i * vs + (int64_t)h * 128 + part * kStrRows + 8 * warp + lane)
                        : 0.f;
        in.g = g[(int64_t)i * hv + h];
        in.b = beta[(int64_t)i * hv + h];
    };
    int ph[2] = {0, 0};          // loads issued into each stage (same in every thread)
    __shared__ int w_sh[3];      // kDyn: a ring of item indices, published through barriers

    int w = blockIdx.x;
    if constexpr (kDyn) {
        if (threadIdx.x == 0) {
            w_sh[0] = atomicAdd(ctr, 1);
            w_sh[1] = atomicAdd(ctr, 1);
        }
        __syncthreads();
        w = w_sh[0];
    }
    StrIn<T> cur;
    if (w < n_items) {
        int i, h, part;
        const int64_t slot = slot_of(w, i, h, part);
        if (slot >= 0 && slot < n_slots) {
            if (threadIdx.x == 0) {
                mbar_arrive_expect_tx(&full[0], kStrBytes);
                bulk_load(smem_raw, state_ptr(slot, h, part), kStrBytes, &full[0]);
            }
            ++ph[0];
        }
        // launched behind the kernel that writes q, k, v, g and beta (the
        // fused decode step's front kernel): the first state is on its way,
        // the inputs are read only once that kernel has finished
        if constexpr (!kDyn) griddep_wait();
        load_in(i, h, part, cur);
    }
    for (int n = 0; w < n_items; ++n) {
        const int s = n & 1;
        int i, h, part;
        const int64_t slot = slot_of(w, i, h, part);
        const bool live = slot >= 0 && slot < n_slots;
        if (slot >= n_slots && threadIdx.x == 0) flag_status(GDN_DEVSTAT_BAD_INDEX);
        // prefetch the next item into the other stage (its previous store has
        // been read: the wait below), and its inputs into registers
        const int wn = kDyn ? w_sh[(n + 1) % 3] : w + (int)gridDim.x;
        // kDyn: the item after it, read by every thread at the top of the
        // next iteration; its slot was last read two iterations (or the
        // prologue) ago, with this CTA's barriers in between
        if (kDyn && threadIdx.x == 0) w_sh[(n + 2) % 3] = atomicAdd(ctr, 1);
        StrIn<T> nxt = cur;
        if (wn < n_items) {
            int in_, hn, pn;
            const int64_t sn = slot_of(wn, in_, hn, pn);
            if (sn >= 0 && sn < n_slots) {
                if (threadIdx.x == 0) {
                    bulk_wait_read_all();
                    mbar_arrive_expect_tx(&full[s ^ 1], kStrBytes);
                    bulk_load(smem_raw + (s ^ 1) * kStrBytes, state_ptr(sn, hn, pn), kStrBytes,
                              &full[s ^ 1]);
                }
                ++ph[s ^ 1];
            }
            load_in(in_, hn, pn, nxt);
        }
        float *st = reinterpret_cast<float *>(smem_raw + s * kStrBytes);
        if (live) {
            mbar_wait(&full[s], (ph[s] - 1) & 1, abort);
            float4 q4 = cur.q4, k4 = cur.k4;
            if (l2norm) {
                const float qn = rsqrtf(row_sum<32>(dot4(q4, q4)) + kL2Eps);
                const float kn = rsqrtf(row_sum<32>(dot4(k4, k4)) + kL2Eps);
                q4 = make_float4(q4.x * qn, q4.y * qn, q4.z * qn, q4.w * qn);
                k4 = make_float4(k4.x * kn, k4.y * kn, k4.z * kn, k4.w * kn);
            }
            const float kq = row_sum<32>(dot4(k4, q4));
            const float alpha = expf(cur.g);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float4 *sp = reinterpret_cast<float4 *>(st + (8 * warp + j) * 128) + lane;
                const float4 sv = *sp;
                const float sk = row_sum<32>(dot4(sv, k4));
                const float sq = row_sum<32>(dot4(sv, q4));
                const float vj = __shfl_sync(0xffffffffu, cur.v, j);
                const float u = cur.b * (vj - alpha * sk);
                *sp = make_float4(fmaf(alpha, sv.x, u * k4.x), fmaf(alpha, sv.y, u * k4.y),
                                  fmaf(alpha, sv.z, u * k4.z), fmaf(alpha, sv.w, u * k4.w));
                if (lane == 0) o_s[8 * warp + j] = scale * fmaf(alpha, sq, u * kq);
            }
            fence_async_smem();
        } else if (lane == 0) {
#pragma unroll
            for (int j = 0; j < 8; ++j) o_s[8 * warp + j] = 0.f;
        }
        __syncthreads();
        if (live && threadIdx.x == 0) {
            bulk_store(state_ptr(slot, h, part), st, kStrBytes);
            bulk_commit();
        }
        if (threadIdx.x < kStrRows)
            Io<T>::store(o + ((int64_t)i * hv + h) * 128 + part * kStrRows + threadIdx.x, o_s[threadIdx.x]);
        __syncthreads();                 // o_s is rewritten by the next item
        cur = nxt;
        w = wn;
    }
    if (threadIdx.x == 0) {
        bulk_wait_read_all();
        if (abort_flag) flag_status(GDN_DEVSTAT_TIMEOUT);
        if constexpr (kDyn) griddep_wait();   // this grid completes after its primary
    }
}

template <int DK, typename T, bool GATED>
static cudaError_t launch_decode(const void *q, int64_t qs, const void *k, int64_t ks,
                                 const void *v, int64_t vs, const float *g, const float *beta,
                                 int n_seqs, int tps, int hqk, int hv, int dv, float scale,
                                 int l2norm, float *pool, int64_t n_slots, const int32_t *idx,
                                 const int32_t *snap, const void *z, int64_t zs, const float *nw,
                                 float neps, void *o, cudaStream_t s) {
    const int64_t heads = (int64_t)n_seqs * hv;
    if (DK == 128 && dv == 128 && tps == 1 && !snap && !GATED &&
        ((uintptr_t)pool % 16) == 0) {   // the streaming kernel: state blocks through bulk copies
        int dev = 0, sms = 148;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        const int n_items = (int)(heads * 2);
        const int grid = (int)std::min<int64_t>(n_items, (int64_t)sms * kStrCtasPerSm);
        cudaError_t e = cudaFuncSetAttribute(decode_stream_kernel<T>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)(2 * kStrBytes));
        if (e != cudaSuccess) return e;
        decode_stream_kernel<T><<<grid, kDecThreads, 2 * kStrBytes, s>>>(
            (const T *)q, qs, (const T *)k, ks, (const T *)v, vs, g, beta, n_items, hv, hv / hqk,
            scale, l2norm, pool, n_slots, idx, (T *)o, nullptr);
        return cudaGetLastError();
    }
    if (dv > 64) {     // two CTAs per state: half the registers, twice the CTAs in flight
        decode_kernel<DK, 2, T, false><<<(unsigned)(heads * 2), kDecThreads, 0, s>>>(
            (const T *)q, qs, (const T *)k, ks, (const T *)v, vs, g, beta, tps, hv, hv / hqk, dv,
            scale, l2norm, pool, n_slots, idx, snap, nullptr, 0, nullptr, 0.f, (T *)o);
    } else {
        decode_kernel<DK, 1, T, GATED><<<(unsigned)heads, kDecThreads, 0, s>>>(
            (const T *)q, qs, (const T *)k, ks, (const T *)v, vs, g, beta, tps, hv, hv / hqk, dv,
            scale, l2norm, pool, n_slots, idx, snap, (const T *)z, zs, nw, neps, (T *)o);
    }
    return cudaGetLastError();
}

// The streaming decode (bf16, dk = dv = 128, one token, q / k L2-normalised)
// launched with programmatic stream serialization: its CTAs may start while
// the kernel before it in the stream (which writes q, k, v, g, beta) is still
// finishing, and fetch their first state meanwhile.
cudaError_t launch_decode_stream_after(const __nv_bfloat16 *q, int64_t qs,
                                       const __nv_bfloat16 *k, int64_t ks,
                                       const __nv_bfloat16 *v, int64_t vs, const float *g,
                                       const float *beta, int n_seqs, int hqk, int hv,
                                       float scale, float *pool, int64_t n_slots,
                                       const int32_t *idx, __nv_bfloat16 *o, cudaStream_t s) {
    const int n_items = (int)((int64_t)n_seqs * hv * 2);
    const int grid = (int)std::min<int64_t>(n_items, (int64_t)sm_count() * kStrCtasPerSm);
    cudaError_t e = cudaFuncSetAttribute(decode_stream_kernel<__nv_bfloat16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(2 * kStrBytes));
    if (e != cudaSuccess) return e;
    return launch_after(decode_stream_kernel<__nv_bfloat16>, dim3((unsigned)grid),
                        dim3(kDecThreads), 2 * kStrBytes, s, q, qs, k, ks, v, vs, g, beta,
                        n_items, hv, hv / hqk, scale, 1, pool, n_slots, idx, o, (int *)nullptr);
}

// The streaming decode with its items handed out by *ctr (zero before the
// launch), launched behind the kernel before it in the stream so that it runs
// on the SMs that kernel leaves free.  The caller guarantees that the kernel
// before it writes none of this decode's inputs, outputs or slots.
cudaError_t launch_decode_stream_beside(const __nv_bfloat16 *q, int64_t qs,
                                        const __nv_bfloat16 *k, int64_t ks,
                                        const __nv_bfloat16 *v, int64_t vs, const float *g,
                                        const float *beta, int n_seqs, int hqk, int hv,
                                        float scale, int l2norm, float *pool, int64_t n_slots,
                                        const int32_t *idx, __nv_bfloat16 *o, int *ctr,
                                        cudaStream_t s) {
    const int n_items = (int)((int64_t)n_seqs * hv * 2);
    const int grid = (int)std::min<int64_t>(n_items, (int64_t)sm_count() * kStrCtasPerSm);
    cudaError_t e = cudaFuncSetAttribute(decode_stream_kernel<__nv_bfloat16, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(2 * kStrBytes));
    if (e != cudaSuccess) return e;
    return launch_after(decode_stream_kernel<__nv_bfloat16, true>, dim3((unsigned)grid),
                        dim3(kDecThreads), 2 * kStrBytes, s, q, qs, k, ks, v, vs, g, beta,
                        n_items, hv, hv / hqk, scale, l2norm, pool, n_slots, idx, o, ctr);
}

}  // namespace gdn

using namespace gdn;

namespace gdn {
// The host-side checks of the decode entries, launching nothing: GDN_OK when
// the call would run (for n_seqs == 0: when it would return GDN_OK).
gdn_status decode_check(const void *q, int64_t q_row_stride, const void *k, int64_t k_row_stride,
                        const void *v, int64_t v_row_stride, const float *g, const float *beta,
                        int32_t n_seqs, int32_t tokens_per_seq, int32_t hqk, int32_t hv,
                        int32_t dk, int32_t dv, const float *state_pool, int64_t n_slots,
                        const int32_t *state_indices, const void *z, int64_t z_row_stride,
                        const float *norm_weight, float norm_eps, const void *o, int32_t dtype) {
    GDN_REQUIRE(dtype == GDN_F32 || dtype == GDN_BF16, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(n_seqs >= 0 && hqk > 0 && hv > 0 && n_slots >= 0, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(hv % hqk == 0, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(tokens_per_seq >= 1 && tokens_per_seq <= kMaxTps, GDN_ERR_UNSUPPORTED);
    GDN_REQUIRE(dk == 16 || dk == 32 || dk == 64 || dk == 128, GDN_ERR_UNSUPPORTED);
    GDN_REQUIRE(dv >= 1 && dv <= kMaxDv, GDN_ERR_UNSUPPORTED);
    if (n_seqs == 0) return GDN_OK;
    GDN_REQUIRE((int64_t)n_seqs * hv * 2 < (1ll << 31), GDN_ERR_UNSUPPORTED);
    GDN_REQUIRE(q && k && v && g && beta && state_pool && state_indices && o, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(q_row_stride >= (int64_t)hqk * dk && k_row_stride >= (int64_t)hqk * dk &&
                    v_row_stride >= (int64_t)hv * dv,
                GDN_ERR_INVALID_ARG);
    const bool gated = z != nullptr;
    GDN_REQUIRE(!gated || (norm_weight && norm_eps >= 0.f && z_row_stride >= (int64_t)hv * dv),
                GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(!gated || dv <= 64 || dv == 128, GDN_ERR_UNSUPPORTED);   // the norm pass's sizes
    GDN_REQUIRE(!gated || dv <= 64 ||
                    (((uintptr_t)z % 16) == 0 && ((uintptr_t)o % 16) == 0 && z_row_stride % 4 == 0),
                GDN_ERR_INVALID_ARG);                                      // and its alignment
    const int64_t align = dtype == GDN_F32 ? 16 : 8;      // load4 of q/k rows
    const int64_t elem = dtype == GDN_F32 ? 4 : 2;
    GDN_REQUIRE(((uintptr_t)q % align) == 0 && ((uintptr_t)k % align) == 0, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE((q_row_stride * elem) % align == 0 && (k_row_stride * elem) % align == 0,
                GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(((uintptr_t)state_pool % 16) == 0, GDN_ERR_INVALID_ARG);
    return GDN_OK;
}
}  // namespace gdn

static gdn_status decode_entry(const void *q, int64_t q_row_stride, const void *k,
                               int64_t k_row_stride, const void *v, int64_t v_row_stride,
                               const float *g, const float *beta, int32_t n_seqs,
                               int32_t tokens_per_seq, int32_t hqk, int32_t hv, int32_t dk,
                               int32_t dv, float scale, int32_t l2norm_qk, float *state_pool,
                               int64_t n_slots, const int32_t *state_indices,
                               const int32_t *snap_indices, const void *z, int64_t z_row_stride,
                               const float *norm_weight, float norm_eps, void *o, int32_t dtype,
                               void *stream) {
    const gdn_status st = decode_check(q, q_row_stride, k, k_row_stride, v, v_row_stride, g, beta,
                                       n_seqs, tokens_per_seq, hqk, hv, dk, dv, state_pool,
                                       n_slots, state_indices, z, z_row_stride, norm_weight,
                                       norm_eps, o, dtype);
    if (st != GDN_OK || n_seqs == 0) return st;
    const bool gated = z != nullptr;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaSuccess;
    // dv > 64: the norm is a separate pass, so the recurrence takes the plain
    // launch (and with it the streaming kernel)
    const bool fused_norm = gated && dv <= 64;
#define GDN_DEC(DK, T)                                                                          \
    e = fused_norm ? launch_decode<DK, T, true>(q, q_row_stride, k, k_row_stride, v, v_row_stride, g,  \
                                           beta, n_seqs, tokens_per_seq, hqk, hv, dv, scale,     \
                                           l2norm_qk, state_pool, n_slots, state_indices,        \
                                           snap_indices, z, z_row_stride, norm_weight, norm_eps, \
                                           o, s)                                                 \
              : launch_decode<DK, T, false>(q, q_row_stride, k, k_row_stride, v, v_row_stride,   \
                                            g, beta, n_seqs, tokens_per_seq, hqk, hv, dv, scale, \
                                            l2norm_qk, state_pool, n_slots, state_indices,       \
                                            snap_indices, nullptr, 0, nullptr, 0.f, o, s)
    if (dtype == GDN_BF16) {
        switch (dk) {
            case 16: GDN_DEC(16, __nv_bfloat16); break;
            case 32: GDN_DEC(32, __nv_bfloat16); break;
            case 64: GDN_DEC(64, __nv_bfloat16); break;
            default: GDN_DEC(128, __nv_bfloat16); break;
        }
    } else {
        switch (dk) {
            case 16: GDN_DEC(16, float); break;
            case 32: GDN_DEC(32, float); break;
            case 64: GDN_DEC(64, float); break;
            default: GDN_DEC(128, float); break;
        }
    }
#undef GDN_DEC
    if (e != cudaSuccess) {
        set_last_cuda_error(e);
        return GDN_ERR_LAUNCH;
    }
    if (gated && dv > 64) {
        // The state's rows are split over two CTAs.  Pairing them as a cluster
        // to add their halves of sum(o^2) cost more (the pair waits on each
        // other) than the separate norm pass below.
        gdn_status st = launch_status();
        if (st != GDN_OK) return st;
        return gdn_gated_rmsnorm(o, z, z_row_stride, norm_weight,
                                 (int64_t)n_seqs * tokens_per_seq, hv, dv, norm_eps, o, dtype,
                                 stream);
    }
    return launch_status();
}

extern "C" gdn_status gdn_decode_recurrent(const void *q, int64_t q_row_stride, const void *k,
                                           int64_t k_row_stride, const void *v,
                                           int64_t v_row_stride, const float *g,
                                           const float *beta, int32_t n_seqs,
                                           int32_t tokens_per_seq, int32_t hqk, int32_t hv,
                                           int32_t dk, int32_t dv, float scale, int32_t l2norm_qk,
                                           float *state_pool, int64_t n_slots,
                                           const int32_t *state_indices,
                                           const int32_t *snap_indices, void *o, int32_t dtype,
                                           void *stream) {
    return decode_entry(q, q_row_stride, k, k_row_stride, v, v_row_stride, g, beta, n_seqs,
                        tokens_per_seq, hqk, hv, dk, dv, scale, l2norm_qk, state_pool, n_slots,
                        state_indices, snap_indices, nullptr, 0, nullptr, 0.f, o, dtype, stream);
}

extern "C" gdn_status gdn_decode_recurrent_gated(
    const void *q, int64_t q_row_stride, const void *k, int64_t k_row_stride, const void *v,
    int64_t v_row_stride, const float *g, const float *beta, int32_t n_seqs,
    int32_t tokens_per_seq, int32_t hqk, int32_t hv, int32_t dk, int32_t dv, float scale,
    int32_t l2norm_qk, float *state_pool, int64_t n_slots, const int32_t *state_indices,
    const int32_t *snap_indices, const void *z, int64_t z_row_stride, const float *norm_weight,
    float norm_eps, void *y, int32_t dtype, void *stream) {
    GDN_REQUIRE(z != nullptr, GDN_ERR_INVALID_ARG);
    return decode_entry(q, q_row_stride, k, k_row_stride, v, v_row_stride, g, beta, n_seqs,
                        tokens_per_seq, hqk, hv, dk, dv, scale, l2norm_qk, state_pool, n_slots,
                        state_indices, snap_indices, z, z_row_stride, norm_weight, norm_eps, y,
                        dtype, stream);
}
