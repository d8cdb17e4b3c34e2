// gdn_prefill_chunked_static: the two-kernel tensor-core prefill (prep kernel
// + chain kernel) with its scratch in a fixed device array inside the
// library instead of a caller workspace.  It allocates nothing.
#include <mutex>

#include "common.cuh"

namespace gdn {
size_t prefill_split_workspace(int n_seqs, int64_t n_tokens, int hv);
bool prefill_tc_supported(int dtype, int dk, int dv, int chunk, const void *q, int64_t qs,
                          const void *k, int64_t ks, const void *v, int64_t vs);
gdn_status prefill_split(const void *q, int64_t qs, const void *k, int64_t ks, const void *v,
                         int64_t vs, const float *g, const float *beta, const int32_t *cu,
                         int n_seqs, int64_t n_tokens, int hqk, int hv, float scale, int l2norm,
                         float *pool, int64_t n_slots, const int32_t *ii, const int32_t *fi,
                         void *o, void *ws, cudaStream_t s, const void *z = nullptr,
                         int64_t zs = 0, const float *norm_w = nullptr, float norm_eps = 0.f,
                         const void *ga = nullptr, const void *gb = nullptr,
                         const float *A_log = nullptr, const float *dt_bias = nullptr);

// One copy per device (a __device__ variable lives in every device's
// instance of the module).
static __device__ __align__(256) uint8_t g_prefill_static_scratch[GDN_PREFILL_STATIC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Address of this device's scratch array, looked up once per device with
// that device current.
gdn_status static_scratch(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        set_last_cuda_error(e);
        return GDN_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return GDN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_prefill_static_scratch);
        if (e != cudaSuccess) {
            set_last_cuda_error(e);
            return GDN_ERR_CUDA;
        }
        if (!p) return GDN_ERR_LAUNCH;   // no CUDA error to report: the lookup gave no address
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return GDN_OK;
}
}  // namespace

}  // namespace gdn

using namespace gdn;

extern "C" gdn_status gdn_prefill_chunked_static(
    const void *q, int64_t q_row_stride, const void *k, int64_t k_row_stride, const void *v,
    int64_t v_row_stride, const float *g, const float *beta, const int32_t *cu_seqlens,
    int32_t n_seqs, int64_t n_tokens, int32_t hqk, int32_t hv, float scale, int32_t l2norm_qk,
    float *state_pool, int64_t n_slots, const int32_t *initial_state_indices,
    const int32_t *final_state_indices, void *o, void *stream) {
    GDN_REQUIRE(n_seqs >= 0 && n_tokens >= 0 && hqk > 0 && hv > 0 && n_slots >= 0,
                GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(hv % hqk == 0, GDN_ERR_INVALID_ARG);
    if (n_seqs == 0) return n_tokens == 0 ? GDN_OK : GDN_ERR_INVALID_ARG;
    GDN_REQUIRE(cu_seqlens != nullptr, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(q && k && v && o && g && beta, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(state_pool || (!initial_state_indices && !final_state_indices),
                GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(q_row_stride >= (int64_t)hqk * 128 && k_row_stride >= (int64_t)hqk * 128 &&
                    v_row_stride >= (int64_t)hv * 128,
                GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(n_tokens > 0, GDN_ERR_UNSUPPORTED);
    GDN_REQUIRE(prefill_tc_supported(GDN_BF16, 128, 128, 64, q, q_row_stride, k, k_row_stride, v,
                                     v_row_stride) &&
                    ((uintptr_t)o & 15u) == 0,
                GDN_ERR_UNSUPPORTED);
    GDN_REQUIRE(prefill_split_workspace(n_seqs, n_tokens, hv) <= GDN_PREFILL_STATIC_SCRATCH_BYTES,
                GDN_ERR_TOO_LARGE);
    void *ws = nullptr;
    gdn_status st = static_scratch(&ws);
    if (st != GDN_OK) return st;
    return prefill_split(q, q_row_stride, k, k_row_stride, v, v_row_stride, g, beta, cu_seqlens,
                         n_seqs, n_tokens, hqk, hv, scale, l2norm_qk, state_pool, n_slots,
                         initial_state_indices, final_state_indices, o, ws,
                         (cudaStream_t)stream);
}
