// gdn_prefill_chunked entry point: argument checks and kernel choice.
#include "common.cuh"

namespace gdn {
gdn_status prefill_simt(int dtype, int dk, int chunk, const void *q, int64_t qs, const void *k,
                        int64_t ks, const void *v, int64_t vs, const float *g, const float *beta,
                        const int32_t *cu, int n_seqs, int64_t n_tokens, int hqk, int hv,
                        float scale, int l2norm, float *pool, int64_t n_slots, const int32_t *ii,
                        const int32_t *fi, void *o, cudaStream_t s);
bool prefill_tc_supported(int dtype, int dk, int dv, int chunk, const void *q, int64_t qs,
                          const void *k, int64_t ks, const void *v, int64_t vs);
gdn_status prefill_tc(const void *q, int64_t qs, const void *k, int64_t ks, const void *v,
                      int64_t vs, const float *g, const float *beta, const int32_t *cu,
                      int n_seqs, int64_t n_tokens, int hqk, int hv, float scale, int l2norm,
                      float *pool, int64_t n_slots, const int32_t *ii, const int32_t *fi,
                      void *o, cudaStream_t s);
size_t prefill_split_workspace(int n_seqs, int64_t n_tokens, int hv);
bool prefill_scan_sized(int n_seqs, int64_t n_tokens);
bool prefill_scan_fits(int hv);
size_t prefill_scan_workspace(int64_t n_tokens, int hv);
gdn_status prefill_scan(const void *q, int64_t qs, const void *k, int64_t ks, const void *v,
                        int64_t vs, const float *g, const float *beta, const int32_t *cu,
                        int64_t n_tokens, int hqk, int hv, float scale, int l2norm, float *pool,
                        int64_t n_slots, const int32_t *ii, const int32_t *fi, void *o, void *ws,
                        cudaStream_t s, const void *ga = nullptr, const void *gb = nullptr,
                        const float *A_log = nullptr, const float *dt_bias = nullptr);
gdn_status prefill_split(const void *q, int64_t qs, const void *k, int64_t ks, const void *v,
                         int64_t vs, const float *g, const float *beta, const int32_t *cu,
                         int n_seqs, int64_t n_tokens, int hqk, int hv, float scale, int l2norm,
                         float *pool, int64_t n_slots, const int32_t *ii, const int32_t *fi,
                         void *o, void *ws, cudaStream_t s, const void *z = nullptr,
                         int64_t zs = 0, const float *norm_w = nullptr, float norm_eps = 0.f,
                         const void *ga = nullptr, const void *gb = nullptr,
                         const float *A_log = nullptr, const float *dt_bias = nullptr);
gdn_status prefill_check(const void *q, int64_t q_row_stride, const void *k, int64_t k_row_stride,
                         const void *v, int64_t v_row_stride, const float *g, const float *beta,
                         const int32_t *cu_seqlens, int32_t n_seqs, int64_t n_tokens, int32_t hqk,
                         int32_t hv, int32_t dk, int32_t dv, int32_t chunk, const float *state_pool,
                         int64_t n_slots, const int32_t *initial_state_indices,
                         const int32_t *final_state_indices, const void *o, int32_t dtype);
gdn_status norm_check(const void *o, const void *z, int64_t z_row_stride, const float *weight,
                      int64_t n_tokens, int32_t hv, int32_t dv, float eps, const void *y,
                      int32_t dtype);
}  // namespace gdn

using namespace gdn;

// Only the tensor-core path (bf16, dk = dv = 128, chunk 64) uses scratch: the
// chunk-parallel prep kernel writes each (chunk, head) item's operands there.
extern "C" size_t gdn_prefill_workspace_size(int32_t n_seqs, int64_t n_tokens, int32_t hv,
                                             int32_t dk, int32_t dv, int32_t chunk,
                                             int32_t dtype) {
    if (n_seqs <= 0 || n_tokens <= 0 || hv <= 0) return 0;
    if (dtype != GDN_BF16 || dk != 128 || dv != 128 || chunk != 64) return 0;
    const size_t split = prefill_split_workspace(n_seqs, n_tokens, hv);
    if (!prefill_scan_sized(n_seqs, n_tokens)) return split;
    const size_t scan = prefill_scan_workspace(n_tokens, hv);
    return scan > split ? scan : split;
}

namespace gdn {
// The host-side checks of gdn_prefill_chunked, launching nothing: GDN_OK when
// the call would run (for n_seqs == 0: when it would return GDN_OK).
gdn_status prefill_check(const void *q, int64_t q_row_stride, const void *k, int64_t k_row_stride,
                         const void *v, int64_t v_row_stride, const float *g, const float *beta,
                         const int32_t *cu_seqlens, int32_t n_seqs, int64_t n_tokens, int32_t hqk,
                         int32_t hv, int32_t dk, int32_t dv, int32_t chunk, const float *state_pool,
                         int64_t n_slots, const int32_t *initial_state_indices,
                         const int32_t *final_state_indices, const void *o, int32_t dtype) {
    GDN_REQUIRE(dtype == GDN_F32 || dtype == GDN_BF16, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(n_seqs >= 0 && n_tokens >= 0 && hqk > 0 && hv > 0 && n_slots >= 0,
                GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(hv % hqk == 0, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(dk == dv && (dk == 16 || dk == 32 || dk == 64 || dk == 128), GDN_ERR_UNSUPPORTED);
    GDN_REQUIRE(chunk == 16 || chunk == 32 || chunk == 64, GDN_ERR_UNSUPPORTED);
    if (n_seqs == 0) return n_tokens == 0 ? GDN_OK : GDN_ERR_INVALID_ARG;
    GDN_REQUIRE((int64_t)n_seqs * hv * (dv / (dv < 32 ? dv : 32)) < (1ll << 31),
                GDN_ERR_UNSUPPORTED);
    GDN_REQUIRE(cu_seqlens != nullptr, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(n_tokens == 0 || (q && k && v && o && g && beta), GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(state_pool || (!initial_state_indices && !final_state_indices),
                GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(q_row_stride >= (int64_t)hqk * dk && k_row_stride >= (int64_t)hqk * dk &&
                    v_row_stride >= (int64_t)hv * dv,
                GDN_ERR_INVALID_ARG);
    return GDN_OK;
}
}  // namespace gdn

extern "C" gdn_status gdn_prefill_chunked(const void *q, int64_t q_row_stride, const void *k,
                                          int64_t k_row_stride, const void *v, int64_t v_row_stride,
                                          const float *g, const float *beta,
                                          const int32_t *cu_seqlens, int32_t n_seqs,
                                          int64_t n_tokens, int32_t hqk, int32_t hv, int32_t dk,
                                          int32_t dv, float scale, int32_t l2norm_qk,
                                          int32_t chunk, float *state_pool, int64_t n_slots,
                                          const int32_t *initial_state_indices,
                                          const int32_t *final_state_indices, void *o,
                                          int32_t dtype, void *workspace, size_t workspace_bytes,
                                          void *stream) {
    const gdn_status st = prefill_check(q, q_row_stride, k, k_row_stride, v, v_row_stride, g, beta,
                                        cu_seqlens, n_seqs, n_tokens, hqk, hv, dk, dv, chunk,
                                        state_pool, n_slots, initial_state_indices,
                                        final_state_indices, o, dtype);
    if (st != GDN_OK || n_seqs == 0) return st;
    cudaStream_t s = (cudaStream_t)stream;
    if (n_tokens > 0 && prefill_tc_supported(dtype, dk, dv, chunk, q, q_row_stride, k,
                                             k_row_stride, v, v_row_stride)) {
        const bool ws_ok = workspace && ((uintptr_t)workspace & 15u) == 0 &&
                           ((uintptr_t)o & 15u) == 0;
        if (ws_ok && prefill_scan_sized(n_seqs, n_tokens) && prefill_scan_fits(hv) &&
            workspace_bytes >= prefill_scan_workspace(n_tokens, hv))
            return prefill_scan(q, q_row_stride, k, k_row_stride, v, v_row_stride, g, beta,
                                cu_seqlens, n_tokens, hqk, hv, scale, l2norm_qk, state_pool,
                                n_slots, initial_state_indices, final_state_indices, o,
                                workspace, s);
        if (ws_ok && workspace_bytes >= prefill_split_workspace(n_seqs, n_tokens, hv))
            return prefill_split(q, q_row_stride, k, k_row_stride, v, v_row_stride, g, beta,
                                 cu_seqlens, n_seqs, n_tokens, hqk, hv, scale, l2norm_qk,
                                 state_pool, n_slots, initial_state_indices,
                                 final_state_indices, o, workspace, s);
        return prefill_tc(q, q_row_stride, k, k_row_stride, v, v_row_stride, g, beta, cu_seqlens,
                          n_seqs, n_tokens, hqk, hv, scale, l2norm_qk, state_pool, n_slots,
                          initial_state_indices, final_state_indices, o, s);
    }
    return prefill_simt(dtype, dk, chunk, q, q_row_stride, k, k_row_stride, v, v_row_stride, g,
                        beta, cu_seqlens, n_seqs, n_tokens, hqk, hv, scale, l2norm_qk,
                        state_pool, n_slots, initial_state_indices, final_state_indices, o, s);
}

// The prefill with the gated RMSNorm written instead of o.  On the two-kernel
// tensor-core path (a workspace, one chain per (sequence, V head)) the norm
// runs in the chain kernel's output epilogue; every other path is the prefill
// into y followed by gdn_gated_rmsnorm in place.
extern "C" gdn_status gdn_prefill_chunked_gated(
    const void *q, int64_t q_row_stride, const void *k, int64_t k_row_stride, const void *v,
    int64_t v_row_stride, const float *g, const float *beta, const int32_t *cu_seqlens,
    int32_t n_seqs, int64_t n_tokens, int32_t hqk, int32_t hv, int32_t dk, int32_t dv,
    float scale, int32_t l2norm_qk, int32_t chunk, float *state_pool, int64_t n_slots,
    const int32_t *initial_state_indices, const int32_t *final_state_indices, const void *z,
    int64_t z_row_stride, const float *norm_weight, float norm_eps, void *y, int32_t dtype,
    void *workspace, size_t workspace_bytes, void *stream) {
    gdn_status st = prefill_check(q, q_row_stride, k, k_row_stride, v, v_row_stride, g, beta,
                                  cu_seqlens, n_seqs, n_tokens, hqk, hv, dk, dv, chunk,
                                  state_pool, n_slots, initial_state_indices,
                                  final_state_indices, y, dtype);
    if (st != GDN_OK || n_seqs == 0) return st;
    st = norm_check(y, z, z_row_stride, norm_weight, n_tokens, hv, dv, norm_eps, y, dtype);
    if (st != GDN_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    const bool ws_ok = workspace && ((uintptr_t)workspace & 15u) == 0 && ((uintptr_t)y & 15u) == 0;
    const bool scan = prefill_scan_sized(n_seqs, n_tokens) && prefill_scan_fits(hv) &&
                      workspace_bytes >= prefill_scan_workspace(n_tokens, hv);
    if (n_tokens > 0 && ws_ok && !scan &&
        prefill_tc_supported(dtype, dk, dv, chunk, q, q_row_stride, k, k_row_stride, v,
                             v_row_stride) &&
        ((uintptr_t)z & 15u) == 0 && (z_row_stride % 8) == 0 &&
        workspace_bytes >= prefill_split_workspace(n_seqs, n_tokens, hv))
        return prefill_split(q, q_row_stride, k, k_row_stride, v, v_row_stride, g, beta,
                             cu_seqlens, n_seqs, n_tokens, hqk, hv, scale, l2norm_qk, state_pool,
                             n_slots, initial_state_indices, final_state_indices, y, workspace, s,
                             z, z_row_stride, norm_weight, norm_eps);
    st = gdn_prefill_chunked(q, q_row_stride, k, k_row_stride, v, v_row_stride, g, beta,
                             cu_seqlens, n_seqs, n_tokens, hqk, hv, dk, dv, scale, l2norm_qk,
                             chunk, state_pool, n_slots, initial_state_indices,
                             final_state_indices, y, dtype, workspace, workspace_bytes, stream);
    if (st != GDN_OK) return st;
    return gdn_gated_rmsnorm(y, z, z_row_stride, norm_weight, n_tokens, hv, dv, norm_eps, y,
                             dtype, stream);
}

// The prefill layer in one call: the conv of the raw q|k|v stream into the
// workspace, then the chunked prefill on its q, k, v views with the gates
// formed in the prep kernel from the raw a, b (no gating launch, no g / beta
// round trip).  Built for the tensor-core path: bf16, dk = dv = 128, chunk 64,
// conv width 4.
extern "C" size_t gdn_prefill_layer_workspace_size(int32_t n_seqs, int64_t n_tokens, int32_t hqk,
                                                   int32_t hv) {
    if (n_seqs <= 0 || n_tokens <= 0 || hqk <= 0 || hv <= 0) return 0;
    const size_t C = 2 * (size_t)hqk * 128 + (size_t)hv * 128;
    const size_t y = ((size_t)n_tokens * C * 2 + 1023) / 1024 * 1024;
    return y + gdn_prefill_workspace_size(n_seqs, n_tokens, hv, 128, 128, 64, GDN_BF16);
}

namespace {
// The layer's prefill in one call; with z, the gated RMSNorm output y is
// written instead of o (in the chain kernel's epilogue on the two-kernel
// path, by the norm kernel in place after the chunk-state scan).
gdn_status prefill_layer(const void *x, int64_t x_row_stride, const void *conv_weight,
                         const void *conv_bias, void *conv_state_pool, int64_t n_conv_slots,
                         const int32_t *conv_state_indices, const uint8_t *has_initial_state,
                         const void *a, const void *b, const float *A_log, const float *dt_bias,
                         const int32_t *cu_seqlens, int32_t n_seqs, int64_t n_tokens, int32_t hqk,
                         int32_t hv, float scale, float *state_pool, int64_t n_slots,
                         const int32_t *initial_state_indices, const int32_t *final_state_indices,
                         const void *z, int64_t z_row_stride, const float *norm_weight,
                         float norm_eps, void *out, void *workspace, size_t workspace_bytes,
                         void *stream) {
    GDN_REQUIRE(n_seqs >= 0 && n_tokens >= 0 && hqk > 0 && hv > 0, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(hv % hqk == 0, GDN_ERR_INVALID_ARG);
    if (n_seqs == 0) return n_tokens == 0 ? GDN_OK : GDN_ERR_INVALID_ARG;
    GDN_REQUIRE(a && b && A_log && dt_bias && x, GDN_ERR_INVALID_ARG);
    const int64_t C = 2 * (int64_t)hqk * 128 + (int64_t)hv * 128;
    const int64_t nq = (int64_t)hqk * 128;
    // the prefill's checks on the views of y (g, beta: stand-ins, never read)
    gdn_status st = prefill_check(x, C, x, C, x, C, A_log, dt_bias, cu_seqlens, n_seqs, n_tokens,
                                  hqk, hv, 128, 128, 64, state_pool, n_slots,
                                  initial_state_indices, final_state_indices, out, GDN_BF16);
    if (st != GDN_OK) return st;
    if (z) {
        st = norm_check(out, z, z_row_stride, norm_weight, n_tokens, hv, 128, norm_eps, out,
                        GDN_BF16);
        if (st != GDN_OK) return st;
    }
    if (n_tokens == 0) return GDN_OK;
    const size_t need = gdn_prefill_layer_workspace_size(n_seqs, n_tokens, hqk, hv);
    GDN_REQUIRE(workspace && workspace_bytes >= need && ((uintptr_t)workspace % 1024) == 0,
                GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(((uintptr_t)out % 16) == 0, GDN_ERR_INVALID_ARG);
    const size_t y_bytes = ((size_t)n_tokens * C * 2 + 1023) / 1024 * 1024;
    __nv_bfloat16 *y = (__nv_bfloat16 *)workspace;
    void *pws = (uint8_t *)workspace + y_bytes;
    const size_t pws_bytes = workspace_bytes - y_bytes;
    st = causal_conv1d_fwd(x, x_row_stride, conv_weight, conv_bias, cu_seqlens, n_seqs, n_tokens,
                           (int32_t)C, 4, conv_state_pool, n_conv_slots, conv_state_indices,
                           has_initial_state, 1, y, GDN_BF16, stream);
    if (st != GDN_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    if (prefill_scan_sized(n_seqs, n_tokens) && prefill_scan_fits(hv) &&
        pws_bytes >= prefill_scan_workspace(n_tokens, hv)) {
        st = prefill_scan(y, C, y + nq, C, y + 2 * nq, C, nullptr, nullptr, cu_seqlens, n_tokens,
                          hqk, hv, scale, 1, state_pool, n_slots, initial_state_indices,
                          final_state_indices, out, pws, s, a, b, A_log, dt_bias);
        if (st != GDN_OK || !z) return st;
        return gdn_gated_rmsnorm(out, z, z_row_stride, norm_weight, n_tokens, hv, 128, norm_eps,
                                 out, GDN_BF16, stream);
    }
    // the chain kernel's gated epilogue loads z by TMA: 16-byte rows
    const bool z_tma = z && ((uintptr_t)z % 16) == 0 && (z_row_stride % 8) == 0;
    st = prefill_split(y, C, y + nq, C, y + 2 * nq, C, nullptr, nullptr, cu_seqlens, n_seqs,
                       n_tokens, hqk, hv, scale, 1, state_pool, n_slots, initial_state_indices,
                       final_state_indices, out, pws, s, z_tma ? z : nullptr, z_row_stride,
                       norm_weight, norm_eps, a, b, A_log, dt_bias);
    if (st != GDN_OK || !z || z_tma) return st;
    return gdn_gated_rmsnorm(out, z, z_row_stride, norm_weight, n_tokens, hv, 128, norm_eps, out,
                             GDN_BF16, stream);
}
}  // namespace

extern "C" gdn_status gdn_prefill_layer(
    const void *x, int64_t x_row_stride, const void *conv_weight, const void *conv_bias,
    void *conv_state_pool, int64_t n_conv_slots, const int32_t *conv_state_indices,
    const uint8_t *has_initial_state, const void *a, const void *b, const float *A_log,
    const float *dt_bias, const int32_t *cu_seqlens, int32_t n_seqs, int64_t n_tokens,
    int32_t hqk, int32_t hv, float scale, float *state_pool, int64_t n_slots,
    const int32_t *initial_state_indices, const int32_t *final_state_indices, void *o,
    void *workspace, size_t workspace_bytes, void *stream) {
    return prefill_layer(x, x_row_stride, conv_weight, conv_bias, conv_state_pool, n_conv_slots,
                         conv_state_indices, has_initial_state, a, b, A_log, dt_bias, cu_seqlens,
                         n_seqs, n_tokens, hqk, hv, scale, state_pool, n_slots,
                         initial_state_indices, final_state_indices, nullptr, 0, nullptr, 0.f, o,
                         workspace, workspace_bytes, stream);
}

extern "C" gdn_status gdn_prefill_layer_gated(
    const void *x, int64_t x_row_stride, const void *conv_weight, const void *conv_bias,
    void *conv_state_pool, int64_t n_conv_slots, const int32_t *conv_state_indices,
    const uint8_t *has_initial_state, const void *a, const void *b, const float *A_log,
    const float *dt_bias, const int32_t *cu_seqlens, int32_t n_seqs, int64_t n_tokens,
    int32_t hqk, int32_t hv, float scale, float *state_pool, int64_t n_slots,
    const int32_t *initial_state_indices, const int32_t *final_state_indices, const void *z,
    int64_t z_row_stride, const float *norm_weight, float norm_eps, void *y, void *workspace,
    size_t workspace_bytes, void *stream) {
    GDN_REQUIRE(z || n_tokens == 0, GDN_ERR_INVALID_ARG);
    return prefill_layer(x, x_row_stride, conv_weight, conv_bias, conv_state_pool, n_conv_slots,
                         conv_state_indices, has_initial_state, a, b, A_log, dt_bias, cu_seqlens,
                         n_seqs, n_tokens, hqk, hv, scale, state_pool, n_slots,
                         initial_state_indices, final_state_indices, z, z_row_stride, norm_weight,
                         norm_eps, y, workspace, workspace_bytes, stream);
}
