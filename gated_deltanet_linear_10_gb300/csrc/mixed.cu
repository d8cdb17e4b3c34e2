// A serving step's mixed batch in one call: decode continuations and prefill
// (or chunked-prefill continuation) sequences of one packed varlen batch
// (the mixed batches and chunked prefill of "[model] support Qwen3next",
// which runs decode and prefill requests of one step through the layer).
//
// The first n_decode sequences are one token each, rows 0 .. n_decode-1;
// they go to the recurrent decode kernels, which stream each state once.
// The rest go to the chunked prefill on the same stream.  No kernel of its
// own: the two halves are the library's decode and prefill paths, with the
// prefill half given the tail of cu_seqlens (its token rows are absolute).
#include "common.cuh"

namespace gdn {

GDN_DECLARE_STATUS_WORD(g_status_mixed)
GDN_STATUS_READER(read_status_mixed, g_status_mixed)

// The decode rows must be one token each at rows 0 .. n_decode-1:
// cu_seqlens[i] == i for i <= n_decode.  A batch that breaks this is still
// run (the decode kernels read rows 0 .. n_decode-1) but is reported.
__global__ void mixed_check_kernel(const int32_t *__restrict__ cu, int n_decode) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i <= n_decode;
         i += gridDim.x * blockDim.x)
        if (cu[i] != i) flag_status(GDN_DEVSTAT_BAD_SEQLEN);
}

gdn_status prefill_check(const void *q, int64_t q_row_stride, const void *k, int64_t k_row_stride,
                         const void *v, int64_t v_row_stride, const float *g, const float *beta,
                         const int32_t *cu_seqlens, int32_t n_seqs, int64_t n_tokens, int32_t hqk,
                         int32_t hv, int32_t dk, int32_t dv, int32_t chunk, const float *state_pool,
                         int64_t n_slots, const int32_t *initial_state_indices,
                         const int32_t *final_state_indices, const void *o, int32_t dtype);
gdn_status decode_check(const void *q, int64_t q_row_stride, const void *k, int64_t k_row_stride,
                        const void *v, int64_t v_row_stride, const float *g, const float *beta,
                        int32_t n_seqs, int32_t tokens_per_seq, int32_t hqk, int32_t hv,
                        int32_t dk, int32_t dv, const float *state_pool, int64_t n_slots,
                        const int32_t *state_indices, const void *z, int64_t z_row_stride,
                        const float *norm_weight, float norm_eps, const void *o, int32_t dtype);
}  // namespace gdn

extern "C" gdn_status gdn_mixed_batch(
    const void *q, int64_t q_row_stride, const void *k, int64_t k_row_stride, const void *v,
    int64_t v_row_stride, const float *g, const float *beta, const int32_t *cu_seqlens,
    int32_t n_seqs, int32_t n_decode, int64_t n_tokens, int32_t hqk, int32_t hv, int32_t dk,
    int32_t dv, float scale, int32_t l2norm_qk, int32_t chunk, float *state_pool,
    int64_t n_slots, const int32_t *initial_state_indices, const int32_t *final_state_indices,
    int32_t decode_in_place, void *o, int32_t dtype, void *workspace, size_t workspace_bytes,
    void *stream) {
    GDN_REQUIRE(n_seqs >= 0 && n_decode >= 0 && n_decode <= n_seqs && n_tokens >= n_decode,
                GDN_ERR_INVALID_ARG);
    // in place: the streaming kernel; otherwise the state after the token
    // goes to the final slot and the initial one is only read
    const bool in_place = decode_in_place != 0;
    // both halves' host checks before either launches
    if (n_decode > 0) {
        // a decode row continues a state: it needs its initial slot
        GDN_REQUIRE(initial_state_indices != nullptr, GDN_ERR_INVALID_ARG);
        GDN_REQUIRE(in_place || final_state_indices != nullptr, GDN_ERR_INVALID_ARG);
        const gdn_status st = gdn::decode_check(
            q, q_row_stride, k, k_row_stride, v, v_row_stride, g, beta, n_decode, 1, hqk, hv, dk,
            dv, state_pool, n_slots, initial_state_indices, nullptr, 0, nullptr, 0.f, o, dtype);
        if (st != GDN_OK) return st;
    }
    if (n_seqs > n_decode) {
        GDN_REQUIRE(cu_seqlens != nullptr, GDN_ERR_INVALID_ARG);
        const gdn_status st = gdn::prefill_check(
            q, q_row_stride, k, k_row_stride, v, v_row_stride, g, beta, cu_seqlens + n_decode,
            n_seqs - n_decode, n_tokens, hqk, hv, dk, dv, chunk, state_pool, n_slots,
            initial_state_indices ? initial_state_indices + n_decode : nullptr,
            final_state_indices ? final_state_indices + n_decode : nullptr, o, dtype);
        if (st != GDN_OK) return st;
    }
    if (n_decode > 0) {
        if (cu_seqlens) {
            gdn::mixed_check_kernel<<<(n_decode + 256) / 256, 256, 0, (cudaStream_t)stream>>>(
                cu_seqlens, n_decode);
            const gdn_status st = gdn::launch_status();
            if (st != GDN_OK) return st;
        }
        const gdn_status st = gdn_decode_recurrent(
            q, q_row_stride, k, k_row_stride, v, v_row_stride, g, beta, n_decode, 1, hqk, hv, dk,
            dv, scale, l2norm_qk, state_pool, n_slots, initial_state_indices,
            in_place ? nullptr : final_state_indices, o, dtype, stream);
        if (st != GDN_OK) return st;
    }
    if (n_seqs == n_decode) return GDN_OK;
    return gdn_prefill_chunked(
        q, q_row_stride, k, k_row_stride, v, v_row_stride, g, beta, cu_seqlens + n_decode,
        n_seqs - n_decode, n_tokens, hqk, hv, dk, dv, scale, l2norm_qk, chunk, state_pool, n_slots,
        initial_state_indices ? initial_state_indices + n_decode : nullptr,
        final_state_indices ? final_state_indices + n_decode : nullptr, o, dtype, workspace,
        workspace_bytes, stream);
}
