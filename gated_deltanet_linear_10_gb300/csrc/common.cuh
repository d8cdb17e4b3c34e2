// Shared device/host helpers of libgdn (internal header, not installed).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "gdn.h"

namespace gdn {

// ---------------------------------------------------------------- status --
// Each translation unit owns one device status word; gdn_get_device_status
// ORs them.  Kernels only ever set bits (atomicOr), never trap.
#define GDN_DECLARE_STATUS_WORD(name)                                          \
    __device__ unsigned int name = 0u;                                         \
    __device__ __forceinline__ void flag_status(unsigned int bits) {           \
        atomicOr(&name, bits);                                                 \
    }

// Host helpers implemented in api.cu.
void set_last_cuda_error(cudaError_t e);
gdn_status launch_status();  // cudaGetLastError() after a launch -> status
// decode.cu: the streaming decode launched behind the kernel producing its
// inputs (programmatic dependent launch); used by the fused decode step
cudaError_t launch_decode_stream_after(const __nv_bfloat16 *q, int64_t qs,
                                       const __nv_bfloat16 *k, int64_t ks,
                                       const __nv_bfloat16 *v, int64_t vs, const float *g,
                                       const float *beta, int n_seqs, int hqk, int hv,
                                       float scale, float *pool, int64_t n_slots,
                                       const int32_t *idx, __nv_bfloat16 *o, cudaStream_t s);
// decode.cu: the streaming decode with counter-assigned items, launched to run
// beside the kernel before it (the mixed batch's chain kernel)
cudaError_t launch_decode_stream_beside(const __nv_bfloat16 *q, int64_t qs,
                                        const __nv_bfloat16 *k, int64_t ks,
                                        const __nv_bfloat16 *v, int64_t vs, const float *g,
                                        const float *beta, int n_seqs, int hqk, int hv,
                                        float scale, int l2norm, float *pool, int64_t n_slots,
                                        const int32_t *idx, __nv_bfloat16 *o, int *ctr,
                                        cudaStream_t s);
int sm_count();              // multiprocessors of the current device

// Per-TU readers of the status word (defined next to each word).
gdn_status read_status_gating(uint32_t *out, int clear, cudaStream_t s);
gdn_status read_status_conv(uint32_t *out, int clear, cudaStream_t s);
gdn_status read_status_decode(uint32_t *out, int clear, cudaStream_t s);
gdn_status read_status_prefill_simt(uint32_t *out, int clear, cudaStream_t s);
gdn_status read_status_prefill_tc(uint32_t *out, int clear, cudaStream_t s);
gdn_status read_status_prefill_split(uint32_t *out, int clear, cudaStream_t s);
gdn_status read_status_decode_step(uint32_t *out, int clear, cudaStream_t s);
gdn_status read_status_api(uint32_t *out, int clear, cudaStream_t s);
gdn_status read_status_mixed(uint32_t *out, int clear, cudaStream_t s);
gdn_status read_status_prefill_scan(uint32_t *out, int clear, cudaStream_t s);
gdn_status read_status_mtp_step(uint32_t *out, int clear, cudaStream_t s);

#define GDN_STATUS_READER(fn, word)                                             \
    gdn_status fn(uint32_t *out, int clear, cudaStream_t s) {                  \
        unsigned int v = 0;                                                    \
        cudaError_t e = cudaMemcpyFromSymbolAsync(&v, word, sizeof(v), 0,      \
                                                  cudaMemcpyDeviceToHost, s);  \
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);                    \
        if (e == cudaSuccess && clear) {                                       \
            unsigned int z = 0;                                                \
            e = cudaMemcpyToSymbolAsync(word, &z, sizeof(z), 0,                \
                                        cudaMemcpyHostToDevice, s);            \
            if (e == cudaSuccess) e = cudaStreamSynchronize(s);                \
        }                                                                      \
        if (e != cudaSuccess) {                                                \
            set_last_cuda_error(e);                                            \
            return GDN_ERR_CUDA;                                               \
        }                                                                      \
        *out |= v;                                                             \
        return GDN_OK;                                                         \
    }

// ------------------------------------------------------------ element io --
template <typename T> struct Io;

template <> struct Io<float> {
    static __device__ __forceinline__ float load(const float *p) { return *p; }
    static __device__ __forceinline__ void store(float *p, float v) { *p = v; }
};

template <> struct Io<__nv_bfloat16> {
    static __device__ __forceinline__ float load(const __nv_bfloat16 *p) {
        return __bfloat162float(*p);
    }
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, float v) {
        *p = __float2bfloat16_rn(v);
    }
};

// Load 4 consecutive elements as fp32 (8-byte aligned for bf16, 16 for fp32).
__device__ __forceinline__ float4 load4(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16 *p) {
    uint2 r = *reinterpret_cast<const uint2 *>(p);
    __nv_bfloat162 lo = *reinterpret_cast<__nv_bfloat162 *>(&r.x);
    __nv_bfloat162 hi = *reinterpret_cast<__nv_bfloat162 *>(&r.y);
    float2 a = __bfloat1622float2(lo), b = __bfloat1622float2(hi);
    return make_float4(a.x, a.y, b.x, b.y);
}

// Vector of N elements moved as 16 bytes: 8 bf16 or 4 fp32.
template <typename T> struct Vec16;
template <> struct Vec16<float> {
    static constexpr int N = 4;
    static __device__ __forceinline__ void load(const float *p, float *out) {
        float4 v = *reinterpret_cast<const float4 *>(p);
        out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
    }
    static __device__ __forceinline__ void store(float *p, const float *in) {
        *reinterpret_cast<float4 *>(p) = make_float4(in[0], in[1], in[2], in[3]);
    }
    static __device__ __forceinline__ void unpack(const uint4 &r, float *out) {
        out[0] = __uint_as_float(r.x); out[1] = __uint_as_float(r.y);
        out[2] = __uint_as_float(r.z); out[3] = __uint_as_float(r.w);
    }
};
template <> struct Vec16<__nv_bfloat16> {
    static constexpr int N = 8;
    static __device__ __forceinline__ void unpack(const uint4 &r, float *out) {
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&r);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 f = __bfloat1622float2(h[i]);
            out[2 * i] = f.x;
            out[2 * i + 1] = f.y;
        }
    }
    static __device__ __forceinline__ void load(const __nv_bfloat16 *p, float *out) {
        uint4 r = *reinterpret_cast<const uint4 *>(p);
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&r);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 f = __bfloat1622float2(h[i]);
            out[2 * i] = f.x;
            out[2 * i + 1] = f.y;
        }
    }
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, const float *in) {
        uint4 r;
        __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&r);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(in[2 * i], in[2 * i + 1]);
        *reinterpret_cast<uint4 *>(p) = r;
    }
};

// Reduce-scatter step over a warp of N per-lane values: lanes whose bit N/2
// is set keep the upper half of the values, the others the lower half, each
// adding its partner's (lane ^ N/2) copy of the half it keeps.  Steps N, N/2,
// ..., 2 leave in lane l the sum, over the lanes that differ from l only in
// bits below N, of value (l mod N).
template <int N, int M>
__device__ __forceinline__ void reduce_scatter_step(float (&v)[M], int lane) {
    static_assert(N <= M && N >= 2, "step size");
    constexpr int H = N / 2;
    const bool up = (lane & H) != 0;
#pragma unroll
    for (int j = 0; j < H; ++j) {
        const float send = up ? v[j] : v[H + j];
        const float keep = up ? v[H + j] : v[j];
        v[j] = keep + __shfl_xor_sync(0xffffffffu, send, H);
    }
}

// SiLU(z) = z / (1 + e^-z) with the fast exponential and the fast division:
// relative error a few fp32 ulp, below the bf16 rounding of the outputs; for
// z << 0 the denominator overflows and the quotient goes to 0.  (The
// correctly rounded reciprocal costs several times the instructions, and the
// kernels that take SiLU per element are issue-bound.)
__device__ __forceinline__ float silu_f(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// SiLU for a bf16 result: z sigmoid(z) = h + h tanh(h) with h = z / 2 and the
// hardware tanh (tanh.approx.f32, one instruction; relative error about
// 2^-11, a quarter of the bf16 rounding of the result).
__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float silu_bf16out(float z) {
    const float h = 0.5f * z;
    return fmaf(h, tanh_approx(h), h);
}
// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may start while the kernel before it in the stream is still
// running; griddep_wait() returns once that kernel has completed and its
// writes are visible (immediately when there is none), and griddep_launch()
// lets the next such kernel start before this CTA exits.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch with programmatic stream serialization: the kernel may start once
// every CTA of the kernel before it in the stream has called griddep_launch()
// or exited.  It must call griddep_wait() before it reads what that kernel
// writes (and at least one of its threads must call it, so that its own
// completion still implies the earlier kernel's).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_after(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                cudaStream_t s, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// The SiLU a kernel with outputs of type T takes: the fast division for fp32
// outputs, the tanh form for bf16.
template <typename T> __device__ __forceinline__ float silu_for(float z);
template <> __device__ __forceinline__ float silu_for<float>(float z) { return silu_f(z); }
template <> __device__ __forceinline__ float silu_for<__nv_bfloat16>(float z) {
    return silu_bf16out(z);
}

}  // namespace gdn

// Host-side argument check helper.
#define GDN_REQUIRE(cond, code)                                                \
    do {                                                                       \
        if (!(cond)) return (code);                                            \
    } while (0)
