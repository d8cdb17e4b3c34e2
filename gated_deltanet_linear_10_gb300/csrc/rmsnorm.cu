// Gated RMSNorm of the layer output ("gated RMSNorm", "[model] Support
// Qwen3next", LightLLM issue 1097, Highlights; the page names the kernel
// without a formula):
//   y = o / sqrt(mean(o^2) + eps) * w * SiLU(z)
// per (token, V head) row of dv values, normalising first, then gating.
//
// One warp per row, kNormRows rows per warp at a time; lane l holds dv / 32
// consecutive elements (at least one), the mean square is a warp-shuffle
// reduction.  HBM-bound: o and z read once, y written once (y may be o).
// Grid-stride over rows, sized to the SMs.
#include <algorithm>

#include "common.cuh"
#include "tc.cuh"

namespace gdn {

GDN_DECLARE_STATUS_WORD(g_status_norm)
GDN_STATUS_READER(read_status_norm, g_status_norm)

constexpr int kNormWarps = 8;

__device__ __forceinline__ void store4(float *p, const float (&r)[4]) {
    *reinterpret_cast<float4 *>(p) = make_float4(r[0], r[1], r[2], r[3]);
}
__device__ __forceinline__ void store4(__nv_bfloat16 *p, const float (&r)[4]) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(r[0], r[1]), hi = __floats2bfloat162_rn(r[2], r[3]);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t *>(&lo);
    u.y = *reinterpret_cast<const uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(p) = u;
}

// Rows per warp and iteration: their loads are all issued before any
// reduction (two at dv = 256 to stay within 64 registers).
template <int DV> constexpr int norm_rows() { return DV >= 256 ? 2 : 4; }

template <int DV, typename T>
__global__ void __launch_bounds__(kNormWarps * 32, 4)   // 32 warps per SM: loads in flight
gated_rmsnorm_kernel(const T *__restrict__ o, const T *__restrict__ z, int64_t zs,
                     const float *__restrict__ w, uint32_t n_rows, uint32_t hv, float eps,
                     T *__restrict__ y) {
    constexpr int kNormRows = norm_rows<DV>();
    constexpr int EPL = DV >= 128 ? DV / 32 : 4;     // elements per lane, 4-wide vectors
    constexpr int LANES = DV / EPL;
    griddep_wait();   // launched behind the kernel that writes o: nothing is read before it
    const int lane = threadIdx.x & 31;
    const bool on = lane < LANES;
    const int j0 = lane * EPL;
    float wv[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) wv[e] = on ? w[j0 + e] : 0.f;
    const uint32_t stride = gridDim.x * kNormWarps * kNormRows;
    for (uint32_t base = (blockIdx.x * kNormWarps + (threadIdx.x >> 5)) * kNormRows;
         base < n_rows; base += stride) {
        float ov[kNormRows][EPL], zv[kNormRows][EPL];
#pragma unroll
        for (int u = 0; u < kNormRows; ++u) {
            const uint32_t row = base + u;
            const bool ok = on && row < n_rows;
            const uint32_t t = row / hv, h = row - t * hv;
            const T *orow = o + (int64_t)row * DV;
            const T *zrow = z + (int64_t)t * zs + (int64_t)h * DV;
#pragma unroll
            for (int e = 0; e < EPL; e += 4) {
                const float4 a = ok ? load4(orow + j0 + e) : make_float4(0.f, 0.f, 0.f, 0.f);
                const float4 b = ok ? load4(zrow + j0 + e) : make_float4(0.f, 0.f, 0.f, 0.f);
                ov[u][e] = a.x; ov[u][e + 1] = a.y; ov[u][e + 2] = a.z; ov[u][e + 3] = a.w;
                zv[u][e] = b.x; zv[u][e + 1] = b.y; zv[u][e + 2] = b.z; zv[u][e + 3] = b.w;
            }
        }
#pragma unroll
        for (int u = 0; u < kNormRows; ++u) {
            const uint32_t row = base + u;
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) ss = fmaf(ov[u][e], ov[u][e], ss);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            const float inv = rsqrtf(ss * (1.0f / DV) + eps);
            if (on && row < n_rows) {
                T *yrow = y + (int64_t)row * DV;
#pragma unroll
                for (int e = 0; e < EPL; e += 4) {
                    float r[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        r[c] = ov[u][e + c] * inv * wv[e + c] * silu_for<T>(zv[u][e + c]);
                    store4(yrow + j0 + e, r);
                }
            }
        }
    }
}

// Bulk-staged form: a persistent grid walks tiles of kTok whole tokens (all
// hv rows of each).  A tile's o rows (contiguous) and z rows (one copy per
// token, at its row stride) come into shared memory by 1-D bulk copies
// through a 2-stage mbarrier ring, so the next tile is in flight while warps
// normalise this one from shared memory and store y directly.  The register
// kernel above is bound by how many bytes its warps keep in flight
// (long-scoreboard stalls, an L2 that holds none of the rows); the ring
// keeps a tile per CTA in flight whatever the registers.
constexpr int kBulkStages = 2;
constexpr int kBulkCtasPerSm = 3;
constexpr uint32_t kBulkStageBytes = 32 * 1024;          // o and z halves of a stage

template <int DV, typename T>
__global__ void __launch_bounds__(kNormWarps * 32, kBulkCtasPerSm)
gated_rmsnorm_bulk_kernel(const T *__restrict__ o, const T *__restrict__ z, int64_t zs,
                          const float *__restrict__ w, int n_tokens, int hv, int tok_per_tile,
                          float eps, T *__restrict__ y) {
    using namespace tc;
    constexpr int EPL = DV >= 128 ? DV / 32 : 4;      // elements per lane, 4-wide vectors
    constexpr int LANES = DV / EPL;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    __shared__ uint64_t full[kBulkStages];
    __shared__ int abort_flag;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool on = lane < LANES;
    const int j0 = lane * EPL;
    const uint32_t row_bytes = DV * sizeof(T);
    const uint32_t half = kBulkStageBytes / 2;          // o rows, then z rows
    const int n_tiles = (n_tokens + tok_per_tile - 1) / tok_per_tile;
    griddep_wait();   // launched behind the kernel that writes o: nothing is read before it
    if (tid == 0) {
        for (int st = 0; st < kBulkStages; ++st) mbar_init(&full[st], 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    volatile int *abort = &abort_flag;
    float wv[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) wv[e] = on ? w[j0 + e] : 0.f;
    auto issue = [&](int tile, int st) {       // thread 0
        const int t0 = tile * tok_per_tile;
        const int nt = min(tok_per_tile, n_tokens - t0);
        const uint32_t tok_bytes = (uint32_t)hv * row_bytes;
        uint8_t *dst = smem_raw + st * kBulkStageBytes;
        mbar_arrive_expect_tx(&full[st], 2 * nt * tok_bytes);
        bulk_load(dst, o + (int64_t)t0 * hv * DV, nt * tok_bytes, &full[st]);
        for (int u = 0; u < nt; ++u)
            bulk_load(dst + half + u * tok_bytes, z + (int64_t)(t0 + u) * zs, tok_bytes, &full[st]);
    };
    if (tid == 0 && (int)blockIdx.x < n_tiles) issue(blockIdx.x, 0);
    for (int j = 0;; ++j) {
        const int tile = blockIdx.x + j * gridDim.x;
        if (tile >= n_tiles) break;
        const int st = j % kBulkStages;
        if (tid == 0) {                        // the other stage was freed by the last tile
            const int tn = tile + gridDim.x;
            if (tn < n_tiles) issue(tn, (j + 1) % kBulkStages);
        }
        const int t0 = tile * tok_per_tile;
        const int rows = min(tok_per_tile, n_tokens - t0) * hv;
        const uint8_t *stage = smem_raw + st * kBulkStageBytes;
        mbar_wait(&full[st], (j / kBulkStages) & 1, abort);
        constexpr int RB = 4;                  // rows per warp step: their reductions interleave
        for (int r0 = warp * RB; r0 < rows; r0 += kNormWarps * RB) {
            float ov[RB][EPL], zv[RB][EPL], inv[RB];
#pragma unroll
            for (int u = 0; u < RB; ++u) {
                const int r = min(r0 + u, rows - 1);   // past the tile: a valid row, not stored
#pragma unroll
                for (int e = 0; e < EPL; e += 4) {
                    const float4 a = on ? load4(reinterpret_cast<const T *>(stage + r * row_bytes) + j0 + e)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                    const float4 c = on ? load4(reinterpret_cast<const T *>(stage + half + r * row_bytes) + j0 + e)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                    ov[u][e] = a.x; ov[u][e + 1] = a.y; ov[u][e + 2] = a.z; ov[u][e + 3] = a.w;
                    zv[u][e] = c.x; zv[u][e + 1] = c.y; zv[u][e + 2] = c.z; zv[u][e + 3] = c.w;
                }
            }
#pragma unroll
            for (int u = 0; u < RB; ++u) {
                float ss = 0.f;
#pragma unroll
                for (int e = 0; e < EPL; ++e) ss = fmaf(ov[u][e], ov[u][e], ss);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                inv[u] = rsqrtf(ss * (1.0f / DV) + eps);
            }
#pragma unroll
            for (int u = 0; u < RB; ++u) {
                const int r = r0 + u;
                if (on && r < rows) {
                    T *yrow = y + ((int64_t)t0 * hv + r) * DV;
#pragma unroll
                    for (int e = 0; e < EPL; e += 4) {
                        float q[4];
#pragma unroll
                        for (int c = 0; c < 4; ++c) q[c] = ov[u][e + c] * inv[u] * wv[e + c] * silu_for<T>(zv[u][e + c]);
                        store4(yrow + j0 + e, q);
                    }
                }
            }
        }
        __syncthreads();                       // the stage is refilled next iteration
    }
    if (tid == 0 && abort_flag) flag_status(GDN_DEVSTAT_TIMEOUT);
}

// The bulk-staged kernel when every copy is whole 16-byte granules and a
// token's rows fit half a stage; false: use the register kernel.
template <int DV, typename T>
static bool launch_norm_bulk(const void *o, const void *z, int64_t zs, const float *w,
                             int64_t n_tokens, int hv, float eps, void *y, cudaStream_t s) {
    const int64_t tok_bytes = (int64_t)hv * DV * sizeof(T);
    if (tok_bytes % 16 != 0 || tok_bytes > (int64_t)kBulkStageBytes / 2) return false;
    if (((uintptr_t)o % 16) != 0 || ((uintptr_t)z % 16) != 0 || (zs * (int64_t)sizeof(T)) % 16 != 0)
        return false;
    if (n_tokens >= (1ll << 31) / hv) return false;
    const int tok_per_tile = (int)((kBulkStageBytes / 2) / tok_bytes);
    const int smem = kBulkStages * kBulkStageBytes;
    if (cudaFuncSetAttribute(gated_rmsnorm_bulk_kernel<DV, T>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return false;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t n_tiles = (n_tokens + tok_per_tile - 1) / tok_per_tile;
    const int grid = (int)std::min<int64_t>(n_tiles, (int64_t)sms * kBulkCtasPerSm);
    // programmatic launch: the grid is set up while the kernel before it ends
    return launch_after(gated_rmsnorm_bulk_kernel<DV, T>, dim3(grid), dim3(kNormWarps * 32),
                        (size_t)smem, s, (const T *)o, (const T *)z, zs, w, (int)n_tokens, hv,
                        tok_per_tile, eps, (T *)y) == cudaSuccess;
}

template <int DV, typename T>
static void launch_norm(const void *o, const void *z, int64_t zs, const float *w, int64_t rows,
                        int hv, float eps, void *y, cudaStream_t s) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t per = kNormWarps * norm_rows<DV>();
    const int64_t need = (rows + per - 1) / per;
    const unsigned blocks = (unsigned)std::min<int64_t>(need, (int64_t)sms * 8);
    launch_after(gated_rmsnorm_kernel<DV, T>, dim3(blocks), dim3(kNormWarps * 32), 0, s,
                 (const T *)o, (const T *)z, zs, w, (uint32_t)rows, (uint32_t)hv, eps, (T *)y);
}

// The host-side checks of gdn_gated_rmsnorm, launching nothing.
gdn_status norm_check(const void *o, const void *z, int64_t z_row_stride, const float *weight,
                      int64_t n_tokens, int32_t hv, int32_t dv, float eps, const void *y,
                      int32_t dtype) {
    GDN_REQUIRE(dtype == GDN_F32 || dtype == GDN_BF16, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(n_tokens >= 0 && hv > 0 && eps >= 0.f, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(dv == 16 || dv == 32 || dv == 64 || dv == 128 || dv == 256, GDN_ERR_UNSUPPORTED);
    if (n_tokens == 0) return GDN_OK;
    GDN_REQUIRE(o && z && weight && y, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(z_row_stride >= (int64_t)hv * dv, GDN_ERR_INVALID_ARG);
    const int64_t elem = dtype == GDN_F32 ? 4 : 2;           // 4-element vector accesses
    GDN_REQUIRE(((uintptr_t)o % (4 * elem)) == 0 && ((uintptr_t)z % (4 * elem)) == 0 &&
                    ((uintptr_t)y % (4 * elem)) == 0 && (z_row_stride % 4) == 0,
                GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(n_tokens * hv < (1ll << 31), GDN_ERR_UNSUPPORTED);
    return GDN_OK;
}

}  // namespace gdn

using namespace gdn;

extern "C" gdn_status gdn_gated_rmsnorm(const void *o, const void *z, int64_t z_row_stride,
                                        const float *weight, int64_t n_tokens, int32_t hv,
                                        int32_t dv, float eps, void *y, int32_t dtype,
                                        void *stream) {
    const gdn_status chk = norm_check(o, z, z_row_stride, weight, n_tokens, hv, dv, eps, y, dtype);
    if (chk != GDN_OK || n_tokens == 0) return chk;
    const int64_t rows = n_tokens * hv;
    cudaStream_t s = (cudaStream_t)stream;
#define GDN_NORM(DV, T)                                                                     \
    if (!launch_norm_bulk<DV, T>(o, z, z_row_stride, weight, n_tokens, hv, eps, y, s))     \
    launch_norm<DV, T>(o, z, z_row_stride, weight, rows, hv, eps, y, s)
#define GDN_NORM_DV(T)                          \
    switch (dv) {                               \
        case 16: GDN_NORM(16, T); break;        \
        case 32: GDN_NORM(32, T); break;        \
        case 64: GDN_NORM(64, T); break;        \
        case 128: GDN_NORM(128, T); break;      \
        default: GDN_NORM(256, T); break;       \
    }
    if (dtype == GDN_BF16) {
        GDN_NORM_DV(__nv_bfloat16)
    } else {
        GDN_NORM_DV(float)
    }
#undef GDN_NORM_DV
#undef GDN_NORM
    return launch_status();
}
