// A serving step's mixed batch in one call: decode continuations and prefill
// (or chunked-prefill continuation) sequences of one packed varlen batch
// (the mixed batches and chunked prefill of "[model] support Qwen3next",
// which runs decode and prefill requests of one step through the layer).
//
// The first n_decode sequences are one token each, rows 0 .. n_decode-1;
// they go to the recurrent decode kernels, which stream each state once.
// The rest go to the chunked prefill on the same stream, with the prefill
// half given the tail of cu_seqlens (its token rows are absolute).
//
// When the decode rows take the streaming kernel in place and the workspace
// has room for a work counter past the prefill's part, the prefill runs
// first and the streaming decode is launched behind its chain kernel
// (programmatic dependent launch) with its items handed out by the counter:
// its CTAs start on the SMs the chains leave free (the chains are one per
// (prompt, V head), often fewer than the SMs) and take over the rest as the
// chains end.  The halves touch disjoint rows and slots, so the decode needs
// nothing from the prefill.
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
    cudaStream_t s = (cudaStream_t)stream;
    if (n_decode > 0 && cu_seqlens) {
        gdn::mixed_check_kernel<<<(n_decode + 256) / 256, 256, 0, s>>>(cu_seqlens, n_decode);
        const gdn_status st = gdn::launch_status();
        if (st != GDN_OK) return st;
    }
    // the decode beside the prefill's chains: the streaming kernel's case,
    // and a work counter past the prefill's part of the workspace
    if (n_decode > 0 && n_seqs > n_decode && in_place && dtype == GDN_BF16 && dk == 128 &&
        dv == 128 && ((uintptr_t)state_pool % 16) == 0 && workspace) {
        const size_t need = gdn_prefill_workspace_size(n_seqs - n_decode, n_tokens, hv, dk, dv,
                                                       chunk, dtype);
        const size_t at = (need + 255) / 256 * 256;
        if (need > 0 && workspace_bytes >= at + 256) {
            int *ctr = reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(workspace) + at);
            cudaError_t e = cudaMemsetAsync(ctr, 0, sizeof(int), s);
            if (e != cudaSuccess) {
                gdn::set_last_cuda_error(e);
                return GDN_ERR_CUDA;
            }
            const gdn_status st = gdn_prefill_chunked(
                q, q_row_stride, k, k_row_stride, v, v_row_stride, g, beta,
                cu_seqlens + n_decode, n_seqs - n_decode, n_tokens, hqk, hv, dk, dv, scale,
                l2norm_qk, chunk, state_pool, n_slots,
                initial_state_indices ? initial_state_indices + n_decode : nullptr,
                final_state_indices ? final_state_indices + n_decode : nullptr, o, dtype,
                workspace, need, stream);
            if (st != GDN_OK) return st;
            e = gdn::launch_decode_stream_beside(
                (const __nv_bfloat16 *)q, q_row_stride, (const __nv_bfloat16 *)k, k_row_stride,
                (const __nv_bfloat16 *)v, v_row_stride, g, beta, n_decode, hqk, hv, scale,
                l2norm_qk, state_pool, n_slots, initial_state_indices, (__nv_bfloat16 *)o, ctr,
                s);
            if (e != cudaSuccess) {
                gdn::set_last_cuda_error(e);
                return GDN_ERR_LAUNCH;
            }
            return GDN_OK;
        }
    }
    if (n_decode > 0) {
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
