// Fused gating: g = -exp(A_log[h]) * softplus(a + dt_bias[h]), beta = sigmoid(b)
// ("fused gating", "[model] support Qwen3next", Highlights; "fused GDN gating",
// "[model] Support Qwen3next", Highlights).  One elementwise pass, fp32 out.
#include "common.cuh"

namespace gdn {

GDN_DECLARE_STATUS_WORD(g_status_gating)
GDN_STATUS_READER(read_status_gating, g_status_gating)

// softplus without overflow: for x > 20, log1p(e^x) = x to within 2e-9 rel.
__device__ __forceinline__ float softplus_f(float x) {
    return x > 20.0f ? x : log1pf(expf(x));
}

template <typename T>
__global__ void gating_kernel(const T *__restrict__ a, const T *__restrict__ b,
                              const float *__restrict__ A_log,
                              const float *__restrict__ dt_bias, int64_t n, int hv,
                              float *__restrict__ g, float *__restrict__ beta) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const int h = (int)(i % hv);
        const float x = Io<T>::load(a + i) + __ldg(dt_bias + h);
        g[i] = -expf(__ldg(A_log + h)) * softplus_f(x);
        beta[i] = 1.0f / (1.0f + expf(-Io<T>::load(b + i)));
    }
}

}  // namespace gdn

using namespace gdn;

extern "C" gdn_status gdn_gating(const void *a, const void *b, const float *A_log,
                                 const float *dt_bias, int64_t n_tokens, int32_t hv,
                                 int32_t in_dtype, float *g, float *beta, void *stream) {
    GDN_REQUIRE(n_tokens >= 0 && hv > 0, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(in_dtype == GDN_F32 || in_dtype == GDN_BF16, GDN_ERR_INVALID_ARG);
    if (n_tokens == 0) return GDN_OK;
    GDN_REQUIRE(a && b && A_log && dt_bias && g && beta, GDN_ERR_INVALID_ARG);
    const int64_t n = n_tokens * hv;
    const int threads = 256;
    int64_t blocks = (n + threads - 1) / threads;
    const int64_t max_blocks = (int64_t)sm_count() * 16;   // 16 CTAs of 256 per SM
    if (blocks > max_blocks) blocks = max_blocks;
    cudaStream_t s = (cudaStream_t)stream;
    if (in_dtype == GDN_F32)
        gating_kernel<float><<<(unsigned)blocks, threads, 0, s>>>(
            (const float *)a, (const float *)b, A_log, dt_bias, n, hv, g, beta);
    else
        gating_kernel<__nv_bfloat16><<<(unsigned)blocks, threads, 0, s>>>(
            (const __nv_bfloat16 *)a, (const __nv_bfloat16 *)b, A_log, dt_bias, n, hv, g, beta);
    return launch_status();
}
