/*
 * gdn.h — C ABI of libgdn, the GB300 (sm_103a) Gated DeltaNet layer.
 *
 * The layer is the linear-attention block of the Qwen3-Next hybrid model as
 * the LightLLM pull request "[model] support Qwen3next" (Highlights: causal 1D
 * convolutions, fused recurrent GDN, fused gating; linear-attention state
 * copying for MTP; a cache manager for linear-attention states), the LightLLM
 * issue "[model] Support Qwen3next" (Highlights: causal conv1d, fused GDN
 * gating, chunked and recurrent linear-attention operations) and the lmdeploy
 * issue "[Feature] Qwen3-Next-80B-A3B Support" (New attention kernels: 16 QK
 * heads, 32 V heads, head_dim 128) describe it.  The pages print no formula;
 * this library computes the standard gated delta rule:
 *
 *   g_t    = -exp(A_log[h]) * softplus(a_t + dt_bias[h]),  beta_t = sigmoid(b_t)
 *   S_t    = exp(g_t) * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *   o_t    = scale * S_t q_t,   q, k L2-normalised per head (eps 1e-6)
 *
 * preceded by a causal depthwise conv1d + SiLU over the channel stream
 * [q (hqk*dk) | k (hqk*dk) | v (hv*dv)].  V head h uses QK head
 * h / (hv / hqk).  S is dv x dk, row-major (row = value index).
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is a DEVICE pointer (cudaMalloc'd or torch
 *     storage) unless its comment says otherwise; the caller owns all memory.
 *     The library allocates no device memory.
 *   - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *     stream.  Every call is asynchronous on that stream and performs no host
 *     synchronisation (so it may be captured in a CUDA graph), except
 *     gdn_get_device_status, which synchronises `stream`.
 *   - Host-side argument checks return GDN_ERR_INVALID_ARG (bad pointer or
 *     size) or GDN_ERR_UNSUPPORTED (valid but not built, e.g. a head size);
 *     in both cases nothing is launched.  A failed launch returns
 *     GDN_ERR_LAUNCH.  Nothing throws across this boundary.
 *   - Values that live on the device (slot indices, cu_seqlens) are checked
 *     by the kernels: an index outside [0, n_slots) is skipped (as if < 0)
 *     and sets GDN_DEVSTAT_BAD_INDEX in the device status word.
 *   - Element counts and strides are in ELEMENTS, not bytes.
 *   - dtype: GDN_F32 = fp32 activations, GDN_BF16 = bf16 activations.
 *     g, beta, A_log, dt_bias and the recurrent state pool are always fp32.
 *   - Two entries of one call naming the same slot (twice as a destination,
 *     or as the source of one and the destination of another) give an
 *     undefined result.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,  /* a host-side argument check failed; nothing ran */
    GDN_ERR_UNSUPPORTED = 2,  /* shape/dtype combination not built; nothing ran */
    GDN_ERR_LAUNCH = 3,       /* a kernel launch failed (CUDA error recorded)   */
    GDN_ERR_CUDA = 4,         /* another CUDA runtime call failed               */
    GDN_ERR_TOO_LARGE = 5     /* beyond a fixed built-in capacity; nothing ran  */
} gdn_status;

typedef enum gdn_dtype {
    GDN_F32 = 0,
    GDN_BF16 = 1
} gdn_dtype;

/* Bits of the device status word (gdn_get_device_status). */
#define GDN_DEVSTAT_BAD_INDEX 0x1u  /* a slot index >= n_slots was skipped      */
#define GDN_DEVSTAT_BAD_SEQLEN 0x2u /* cu_seqlens not non-decreasing / > n_tokens */
#define GDN_DEVSTAT_TIMEOUT 0x4u    /* a bounded wait inside a kernel gave up     */

/* Human-readable name of a status code (static string, never NULL). */
const char *gdn_status_string(gdn_status s);

/* Library version string, e.g. "gdn 0.1.0 sm_103a" (static, never NULL). */
const char *gdn_version(void);

/* Text of the last CUDA error seen by this thread's calls ("" if none). */
const char *gdn_last_cuda_error(void);

/*
 * Fused gating ("fused gating", "[model] support Qwen3next", Highlights;
 * "fused GDN gating", "[model] Support Qwen3next", Highlights):
 *   g[t][h]    = -exp(A_log[h]) * softplus(a[t][h] + dt_bias[h])
 *   beta[t][h] = sigmoid(b[t][h])
 * a, b: [n_tokens][hv] in `in_dtype`, contiguous.  A_log, dt_bias: [hv] fp32.
 * g, beta: [n_tokens][hv] fp32 outputs.  n_tokens may be 0 (no launch).
 */
gdn_status gdn_gating(const void *a, const void *b, const float *A_log,
                      const float *dt_bias, int64_t n_tokens, int32_t hv,
                      int32_t in_dtype, float *g, float *beta, void *stream);

/*
 * Causal depthwise conv1d + optional SiLU over packed variable-length
 * sequences ("causal 1D convolutions", "[model] support Qwen3next",
 * Highlights).  For token t of a sequence and channel c:
 *   y[t][c] = act(bias[c] + sum_{w<width} weight[c][w] * e[t-(width-1)+w][c])
 * where e is the sequence's inputs preceded by its width-1 history rows.
 *   x: [n_tokens] rows, row r at x + r*x_row_stride, `channels` elements
 *      each (x_row_stride >= channels).
 *   weight: [channels][width], bias: [channels] or NULL (both in `dtype`,
 *      16-byte aligned).
 *   cu_seqlens: [n_seqs+1] int32, cu_seqlens[0] = 0, non-decreasing,
 *      cu_seqlens[n_seqs] = n_tokens.  Zero-length sequences are allowed.
 *   conv_state_pool: [n_slots][width-1][channels] in `dtype`; slot s holds the
 *      last width-1 pre-activation inputs, oldest first.
 *   state_indices: [n_seqs] int32.  < 0: zero history, final state not
 *      written.  Otherwise the final state is written to that slot, and the
 *      history is read from it unless has_initial_state[i] == 0.
 *   has_initial_state: [n_seqs] uint8, or NULL (= every slot holds history).
 *   y: [n_tokens][channels] contiguous, `dtype`; y must not alias x.
 * width in [2, 4]; channels a multiple of 8.
 */
gdn_status causal_conv1d_fwd(const void *x, int64_t x_row_stride,
                             const void *weight, const void *bias,
                             const int32_t *cu_seqlens, int32_t n_seqs,
                             int64_t n_tokens, int32_t channels, int32_t width,
                             void *conv_state_pool, int64_t n_slots,
                             const int32_t *state_indices,
                             const uint8_t *has_initial_state, int32_t silu,
                             void *y, int32_t dtype, void *stream);

/*
 * Conv1d decode update for tokens_per_seq new tokens per sequence (1 =
 * decode, mtp_step+1 = MTP; token t of sequence i is row i*tokens_per_seq+t,
 * the layout of "Qwen3 mtp dense", LightLLM pull request 1159, review of the
 * per-request b_seq_len slicing).  Same arithmetic as causal_conv1d_fwd with
 * the slot's state as history.
 *   x, y: [n_seqs*tokens_per_seq][channels] contiguous.
 *   state_indices: [n_seqs]; < 0 = padding row: y rows zero, nothing read
 *      or written.
 *   snap_indices: NULL -> the slot is updated in place.  Otherwise
 *      [n_seqs][tokens_per_seq] int32: the slot is only read and the state
 *      after token t is written to slot snap_indices[i][t] (< 0: skipped).
 * weight / bias as for causal_conv1d_fwd (16-byte aligned).
 * width in [2, 4]; channels a multiple of 8; tokens_per_seq in [1, 16].
 */
gdn_status causal_conv1d_update(const void *x, int32_t n_seqs,
                                int32_t tokens_per_seq, int32_t channels,
                                int32_t width, const void *weight,
                                const void *bias, void *conv_state_pool,
                                int64_t n_slots, const int32_t *state_indices,
                                const int32_t *snap_indices, int32_t silu,
                                void *y, int32_t dtype, void *stream);

/*
 * Chunked varlen prefill of the gated delta rule in WY/UT form ("a suite of
 * Flash Linear Attention operations for efficient chunked ... computations",
 * "[model] Support Qwen3next", Highlights).  Per sequence i and V head h the
 * tokens are taken in chunks of `chunk` from the sequence start; the result
 * equals the token-by-token recurrence up to rounding.
 *   q: token t, QK head j at q + t*q_row_stride + j*dk (same for k);
 *   v: token t, V head h at v + t*v_row_stride + h*dv.  (Views into the
 *      conv output [T][channels] have row stride = channels.)
 *   g, beta: [n_tokens][hv] fp32 (gdn_gating output).
 *   cu_seqlens: as for causal_conv1d_fwd.
 *   state_pool: [n_slots][hv][dv][dk] fp32.
 *   initial_state_indices: [n_seqs]; < 0 = zero initial state.
 *   final_state_indices: [n_seqs]; < 0 = final state not written.  It may
 *      equal the initial index of the same sequence (in-place carry).
 *   o: [n_tokens][hv][dv] contiguous, `dtype`.
 *   scale: multiplies o (usually dk^-1/2).  l2norm_qk: normalise q, k.
 *   workspace / workspace_bytes: device scratch, 16-byte aligned, owned by
 *      the caller and not kept after the call's work on `stream` ends.
 *      gdn_prefill_workspace_size(...) gives the size the two-kernel
 *      tensor-core path needs (bf16, dk = dv = 128, chunk 64): a chunk-
 *      parallel prep kernel writes every (chunk, V head) item's operands
 *      there and a chain kernel streams them back.  With less (or NULL) that
 *      path runs as one fused kernel instead; other shapes need none.
 *      Calls sharing one workspace on different streams race.
 * Built: dk = dv in {16, 32, 64, 128}, chunk in {16, 32, 64} (any dtype);
 * hv a multiple of hqk.
 */
gdn_status gdn_prefill_chunked(const void *q, int64_t q_row_stride,
                               const void *k, int64_t k_row_stride,
                               const void *v, int64_t v_row_stride,
                               const float *g, const float *beta,
                               const int32_t *cu_seqlens, int32_t n_seqs,
                               int64_t n_tokens, int32_t hqk, int32_t hv,
                               int32_t dk, int32_t dv, float scale,
                               int32_t l2norm_qk, int32_t chunk,
                               float *state_pool, int64_t n_slots,
                               const int32_t *initial_state_indices,
                               const int32_t *final_state_indices, void *o,
                               int32_t dtype, void *workspace,
                               size_t workspace_bytes, void *stream);

/* Bytes of scratch gdn_prefill_chunked uses for these sizes (0: none).
 * The two-kernel path takes a 1 KiB-rounded header of n_seqs + 1 chunk
 * offsets, then (ceil(n_tokens / 64) + n_seqs) * hv blocks of 33 KiB.  One
 * sequence of at least 64 chunks (4096 tokens) is given more: room for the
 * chunk-state scan, which cuts the sequence at a chunk boundary into two
 * segments whose chains run at the same time -- segment 0 from the initial
 * state, segment 1 from zero and from the identity (its state transition A
 * and output map Phi) -- then combines them: final state = S_1 A + B, and
 * segment 1's outputs += S_1 Phi^T (S_1: the state at the cut).  It halves
 * the serial chain of a long sequence.  The scan runs when the workspace
 * holds this size and the device has at least 3 * hv SMs; a workspace of
 * the two-kernel size above keeps the serial chain. */
size_t gdn_prefill_workspace_size(int32_t n_seqs, int64_t n_tokens,
                                  int32_t hv, int32_t dk, int32_t dv,
                                  int32_t chunk, int32_t dtype);

/*
 * gdn_prefill_chunked with the gated RMSNorm of gdn_gated_rmsnorm written
 * instead of o:  y = o / sqrt(mean(o^2) + norm_eps) * norm_weight * SiLU(z)
 * per (token, V head) row ("gated RMSNorm", "[model] Support Qwen3next",
 * LightLLM issue 1097, Highlights).  Arguments as gdn_prefill_chunked, plus
 * z (n_tokens rows of [hv][dv], row stride z_row_stride elements, `dtype`),
 * norm_weight [dv] fp32 and norm_eps >= 0; y: [n_tokens][hv][dv] contiguous.
 * On the two-kernel tensor-core path (bf16, dk = dv = 128, chunk 64, a
 * workspace, z 16-byte aligned with z_row_stride a multiple of 8) the norm
 * is computed in the chain kernel's output epilogue from the fp32 o, and o
 * never reaches memory; otherwise (other shapes, or the chunk-state scan) the
 * call is the prefill into y followed by gdn_gated_rmsnorm in place.  The
 * host checks of both (including those of gdn_gated_rmsnorm on y and z) run
 * before anything launches.
 */
gdn_status gdn_prefill_chunked_gated(const void *q, int64_t q_row_stride,
                                     const void *k, int64_t k_row_stride,
                                     const void *v, int64_t v_row_stride,
                                     const float *g, const float *beta,
                                     const int32_t *cu_seqlens, int32_t n_seqs,
                                     int64_t n_tokens, int32_t hqk, int32_t hv,
                                     int32_t dk, int32_t dv, float scale,
                                     int32_t l2norm_qk, int32_t chunk,
                                     float *state_pool, int64_t n_slots,
                                     const int32_t *initial_state_indices,
                                     const int32_t *final_state_indices,
                                     const void *z, int64_t z_row_stride,
                                     const float *norm_weight, float norm_eps,
                                     void *y, int32_t dtype, void *workspace,
                                     size_t workspace_bytes, void *stream);

/*
 * Bytes of the workspace gdn_prefill_layer takes: the conv output y
 * [n_tokens][2*hqk*128 + hv*128] bf16 (rounded up to 1 KiB), then
 * gdn_prefill_workspace_size(n_seqs, n_tokens, hv, 128, 128, 64, GDN_BF16).
 * 0 for an empty batch.
 */
size_t gdn_prefill_layer_workspace_size(int32_t n_seqs, int64_t n_tokens,
                                        int32_t hqk, int32_t hv);

/*
 * The prefill side of the layer in one call (the "causal 1D convolution",
 * "fused GDN gating" and chunked GDN kernels of the Qwen3next pages, over a
 * packed varlen batch):
 *   y = causal_conv1d_fwd(x) (width 4, SiLU; the conv states of
 *       conv_state_indices read for sequences with has_initial_state and the
 *       final ones written, as causal_conv1d_fwd), into the workspace;
 *   the chunked prefill of gdn_prefill_chunked on the q | k | v views of y,
 *       q and k L2-normalised, with g = -exp(A_log) softplus(a + dt_bias) and
 *       beta = sigmoid(b) formed by its prep kernel from the raw a, b (the
 *       same values gdn_gating writes; no gating launch).
 *   x: [n_tokens] rows of 2*hqk*128 + hv*128 channels, row stride
 *      x_row_stride elements (a multiple of 8), bf16, 16-byte aligned.
 *   conv_weight [channels][4], conv_bias [channels] or NULL, conv_state_pool
 *      [n_conv_slots][3][channels]: bf16, as causal_conv1d_fwd.
 *   a, b: [n_tokens][hv] bf16; A_log, dt_bias: [hv] fp32.
 *   state_pool, the index arrays, o [n_tokens][hv][128] bf16 (16-byte
 *      aligned): as gdn_prefill_chunked.
 *   workspace: at least gdn_prefill_layer_workspace_size bytes, 1 KiB
 *      aligned, owned by the caller.
 * Built: bf16, dk = dv = 128, chunk 64, conv width 4.  Every host check runs
 * before the first launch.
 */
gdn_status gdn_prefill_layer(const void *x, int64_t x_row_stride,
                             const void *conv_weight, const void *conv_bias,
                             void *conv_state_pool, int64_t n_conv_slots,
                             const int32_t *conv_state_indices,
                             const uint8_t *has_initial_state, const void *a,
                             const void *b, const float *A_log,
                             const float *dt_bias, const int32_t *cu_seqlens,
                             int32_t n_seqs, int64_t n_tokens, int32_t hqk,
                             int32_t hv, float scale, float *state_pool,
                             int64_t n_slots,
                             const int32_t *initial_state_indices,
                             const int32_t *final_state_indices, void *o,
                             void *workspace, size_t workspace_bytes,
                             void *stream);

/*
 * gdn_prefill_layer writing the layer's gated output instead of o ("gated
 * RMSNorm", Highlights of "[model] Support Qwen3next"):
 *   y = o / sqrt(mean over each (token, V head) row of o^2 + norm_eps)
 *       * norm_weight * SiLU(z),
 * the values gdn_gated_rmsnorm gives on gdn_prefill_layer's o.  On the
 * two-kernel path the norm runs in the prefill chain kernel's output
 * epilogue (o never reaches memory); after the chunk-state scan, or with a z
 * that a TMA tile cannot read (not 16-byte aligned, or a row stride not a
 * multiple of 8), the norm kernel runs on y in place.
 *   z: [n_tokens][hv][128] bf16, row stride z_row_stride elements (>= hv*128,
 *      a multiple of 4), 8-byte aligned; norm_weight: [128] fp32;
 *      norm_eps >= 0.
 *   y: [n_tokens][hv][128] bf16, 16-byte aligned.
 * Every other argument, the workspace and the errors: as gdn_prefill_layer;
 * z == NULL with n_tokens > 0 is GDN_ERR_INVALID_ARG.
 */
gdn_status gdn_prefill_layer_gated(const void *x, int64_t x_row_stride,
                                   const void *conv_weight,
                                   const void *conv_bias, void *conv_state_pool,
                                   int64_t n_conv_slots,
                                   const int32_t *conv_state_indices,
                                   const uint8_t *has_initial_state,
                                   const void *a, const void *b,
                                   const float *A_log, const float *dt_bias,
                                   const int32_t *cu_seqlens, int32_t n_seqs,
                                   int64_t n_tokens, int32_t hqk, int32_t hv,
                                   float scale, float *state_pool,
                                   int64_t n_slots,
                                   const int32_t *initial_state_indices,
                                   const int32_t *final_state_indices,
                                   const void *z, int64_t z_row_stride,
                                   const float *norm_weight, float norm_eps,
                                   void *y, void *workspace,
                                   size_t workspace_bytes, void *stream);

/*
 * gdn_prefill_chunked on its bf16, dk = dv = 128, chunk-64 two-kernel path,
 * with the scratch in a fixed device array built into the library instead of
 * a caller workspace.  The pages describe no such variant: it exists for
 * callers that cannot allocate device memory per call -- a C or C++ runtime
 * with no device allocator of its own in its step loop, where a cudaMalloc /
 * cudaFree pair per call would add synchronising calls mid-step.  It
 * allocates nothing.
 *
 * Arguments are those of gdn_prefill_chunked with dk = dv = 128, chunk = 64,
 * dtype = GDN_BF16 fixed (and no workspace); q, k, v and o must be 16-byte
 * aligned, the q, k, v row strides multiples of 8 elements.
 * Capacity: gdn_prefill_workspace_size(n_seqs, n_tokens, hv, 128, 128, 64,
 * GDN_BF16) <= GDN_PREFILL_STATIC_SCRATCH_BYTES (16 MiB: 496 (chunk, V head)
 * items, i.e. ceil(n_tokens / 64) + n_seqs <= 15 at hv = 32),
 * else GDN_ERR_TOO_LARGE and nothing runs.  n_tokens = 0 returns
 * GDN_ERR_UNSUPPORTED (use gdn_prefill_chunked).
 * The array's address is looked up once per device (cudaGetSymbolAddress
 * with the current device, the one `stream` must belong to); make the first
 * call on each device before any stream capture.  Nothing in the array needs
 * clearing: each call writes every byte it reads before reading it.  There
 * is one array per device, so calls that overlap in time on one device (on
 * different streams or host threads) race and give wrong results.
 */
#define GDN_PREFILL_STATIC_SCRATCH_BYTES (16u << 20)
gdn_status gdn_prefill_chunked_static(const void *q, int64_t q_row_stride,
                                      const void *k, int64_t k_row_stride,
                                      const void *v, int64_t v_row_stride,
                                      const float *g, const float *beta,
                                      const int32_t *cu_seqlens, int32_t n_seqs,
                                      int64_t n_tokens, int32_t hqk, int32_t hv,
                                      float scale, int32_t l2norm_qk,
                                      float *state_pool, int64_t n_slots,
                                      const int32_t *initial_state_indices,
                                      const int32_t *final_state_indices,
                                      void *o, void *stream);

/*
 * Recurrent decode ("fused recurrent GDN", "[model] support Qwen3next",
 * Highlights) for tokens_per_seq tokens per sequence (1 = decode, 4 = MTP
 * with mtp_step 3; row i*tokens_per_seq + t).  Each (sequence, V head) state
 * is read once, kept on chip across the tokens and written once per token
 * that has a destination.
 *   q, k, v: as for gdn_prefill_chunked (rows are tokens).
 *   g, beta: [n_seqs*tokens_per_seq][hv] fp32.
 *   state_pool: [n_slots][hv][dv][dk] fp32.
 *   state_indices: [n_seqs]; < 0 = padding: o rows zero, no state touched.
 *   snap_indices: NULL -> the state after the last token is written back
 *      to state_indices[i] (in place).  Otherwise [n_seqs][tokens_per_seq]:
 *      state_indices[i] is only read, and the state after token t is written
 *      to slot snap_indices[i][t] (< 0: skipped) — the per-draft-token
 *      snapshots MTP accept/rollback needs.
 *   o: [n_seqs*tokens_per_seq][hv][dv] contiguous, `dtype`.
 * Built: dk in {16, 32, 64, 128}, dv <= 128 multiple of 8,
 * tokens_per_seq in [1, 16].
 */
gdn_status gdn_decode_recurrent(const void *q, int64_t q_row_stride,
                                const void *k, int64_t k_row_stride,
                                const void *v, int64_t v_row_stride,
                                const float *g, const float *beta,
                                int32_t n_seqs, int32_t tokens_per_seq,
                                int32_t hqk, int32_t hv, int32_t dk, int32_t dv,
                                float scale, int32_t l2norm_qk,
                                float *state_pool, int64_t n_slots,
                                const int32_t *state_indices,
                                const int32_t *snap_indices, void *o,
                                int32_t dtype, void *stream);

/*
 * Gated RMSNorm of the layer output ("gated RMSNorm", "[model] Support
 * Qwen3next", LightLLM issue 1097, Highlights; the page names the kernel
 * without a formula).  Reading
 * taken: per (token, V head) row of dv values
 *   y = o / sqrt(mean(o^2) + eps) * weight * SiLU(z)     (normalise, then gate)
 *   o, y: [n_tokens][hv][dv] contiguous, `dtype`; y may be o (in place).
 *   z: n_tokens rows of [hv][dv], row stride z_row_stride elements (>= hv*dv),
 *      `dtype`.  weight: [dv] fp32.  eps >= 0.
 * o, z, y aligned to 4 elements and z_row_stride a multiple of 4 (vector
 * accesses), else GDN_ERR_INVALID_ARG.
 * Built: dv in {16, 32, 64, 128, 256}.  All pointers device, caller-owned.
 */
gdn_status gdn_gated_rmsnorm(const void *o, const void *z, int64_t z_row_stride,
                             const float *weight, int64_t n_tokens, int32_t hv,
                             int32_t dv, float eps, void *y, int32_t dtype,
                             void *stream);

/*
 * gdn_decode_recurrent with the gated RMSNorm above fused into its output:
 * writes y = RMSNorm(o) * norm_weight * SiLU(z) instead of o.  Arguments as
 * gdn_decode_recurrent, plus z (rows i * tokens_per_seq + t, stride
 * z_row_stride elements, `dtype`), norm_weight [dv] fp32 and norm_eps.
 * Rows of sequences with no slot are written as zeros.  With dv <= 64 the
 * norm runs inside the decode kernel (one CTA holds a whole state); with
 * dv > 64 the state's rows are split over two CTAs and the call is decode
 * followed by gdn_gated_rmsnorm in place (two launches, same result).
 * Built: dv <= 64 or dv = 128.
 */
gdn_status gdn_decode_recurrent_gated(const void *q, int64_t q_row_stride,
                                      const void *k, int64_t k_row_stride,
                                      const void *v, int64_t v_row_stride,
                                      const float *g, const float *beta,
                                      int32_t n_seqs, int32_t tokens_per_seq,
                                      int32_t hqk, int32_t hv, int32_t dk,
                                      int32_t dv, float scale, int32_t l2norm_qk,
                                      float *state_pool, int64_t n_slots,
                                      const int32_t *state_indices,
                                      const int32_t *snap_indices, const void *z,
                                      int64_t z_row_stride,
                                      const float *norm_weight, float norm_eps,
                                      void *y, int32_t dtype, void *stream);

/*
 * Bytes of the workspace gdn_decode_step_fused takes: the conv output y
 * [n_seqs][channels] bf16 and the gates g, beta [n_seqs][hv] fp32, each
 * rounded up to 256 bytes.  0 for an empty batch.
 */
size_t gdn_decode_step_workspace_size(int32_t n_seqs, int32_t hqk, int32_t hv);

/*
 * One decode step of the layer (fusion of the "causal 1D convolution",
 * "fused GDN gating" and "fused recurrent GDN" kernels the Qwen3next pages
 * name): for each sequence i with one new token,
 *   y   = SiLU(conv_bias + sum_w conv_weight[c][w] * [state; x_i][w])   (width 4)
 *   q|k|v = split(y), q and k L2-normalised per head (eps 1e-6)
 *   g = -exp(A_log[h]) softplus(a_ih + dt_bias[h]), beta = sigmoid(b_ih)
 *   the gated delta rule update of slot state_indices[i], o = scale S q.
 * Equal to causal_conv1d_update + gdn_gating + gdn_decode_recurrent.
 *   x: [n_seqs] rows of the raw q|k|v stream, 2*hqk*128 + hv*128 channels,
 *      row stride x_row_stride elements, bf16.
 *   conv_weight: [channels][4] bf16 (8-byte aligned); conv_bias: [channels]
 *      bf16 or NULL; conv_state_pool: [slots][3][channels] bf16, updated in
 *      place in slot state_indices[i] (the same slot id as the state pool).
 *   a, b: [n_seqs][hv] bf16; A_log, dt_bias: [hv] fp32.
 *   state_pool: [n_slots][hv][128][128] fp32 (16-byte aligned).
 *   workspace: NULL, or device scratch of workspace_bytes >=
 *      gdn_decode_step_workspace_size(n_seqs, hqk, hv), 256-byte aligned,
 *      owned by the caller and not shared with a call in flight on another
 *      stream.  With it (and x, x_row_stride, conv_weight, conv_bias and
 *      conv_state_pool 16-byte aligned) the step runs as two kernels: the
 *      conv update and gates into the workspace, then the streaming decode
 *      launched behind it (programmatic dependent launch).  Without it, or
 *      when it is too small, one kernel does the whole step.
 *   o: [n_seqs][hv][128] bf16.
 * A slot < 0 skips the sequence (o rows zero, neither pool touched); a slot
 * >= n_slots is skipped the same way and sets GDN_DEVSTAT_BAD_INDEX.
 * Built: bf16, dk = dv = 128, hv / hqk <= 2, conv width 4, SiLU on.
 */
gdn_status gdn_decode_step_fused(const void *x, int64_t x_row_stride,
                                 const void *conv_weight, const void *conv_bias,
                                 void *conv_state_pool, const void *a,
                                 const void *b, const float *A_log,
                                 const float *dt_bias, int32_t n_seqs,
                                 int32_t hqk, int32_t hv, float scale,
                                 float *state_pool, int64_t n_slots,
                                 const int32_t *state_indices, void *workspace,
                                 size_t workspace_bytes, void *o, void *stream);

/*
 * One MTP draft step of the layer in one kernel: gdn_decode_step_fused for
 * tokens_per_seq tokens per sequence (row i * tokens_per_seq + t) with the
 * per-token snapshots MTP accept / rollback needs (the state copying of
 * linear-attention states during MTP decode, "[model] support Qwen3next",
 * Highlights).  For each sequence i with a slot:
 *   the conv update + SiLU of the raw q|k|v stream, the conv state after
 *     token t written to slot snap_indices[i][t] of the conv pool;
 *   the gates, the q / k L2 norms;
 *   the gated delta rule over the tokens, the state after token t written to
 *     slot snap_indices[i][t] of the state pool (o as gdn_decode_recurrent).
 * Slot state_indices[i] of both pools is only read.  Equal to
 * causal_conv1d_update + gdn_gating + gdn_decode_recurrent, each with the
 * same snapshots.  snap_indices is required ([n_seqs][tokens_per_seq]; an
 * entry < 0 is skipped, >= n_slots skipped and flagged); snapshot slots
 * must differ from one another and from every source slot (a shared slot is
 * a race).  conv_state_pool must be 16-byte aligned.  Arguments as
 * gdn_decode_step_fused otherwise: x [n_seqs * tokens_per_seq] rows of the
 * raw stream, a, b [n_seqs * tokens_per_seq][hv] bf16, o
 * [n_seqs * tokens_per_seq][hv][128] bf16.
 * Built: bf16, dk = dv = 128, conv width 4, SiLU on, tokens_per_seq in [1, 16].
 */
gdn_status gdn_mtp_step_fused(const void *x, int64_t x_row_stride,
                              const void *conv_weight, const void *conv_bias,
                              void *conv_state_pool, const void *a, const void *b,
                              const float *A_log, const float *dt_bias, int32_t n_seqs,
                              int32_t tokens_per_seq, int32_t hqk, int32_t hv,
                              float scale, float *state_pool, int64_t n_slots,
                              const int32_t *state_indices,
                              const int32_t *snap_indices, void *o, void *stream);

/*
 * A serving step's mixed batch in one call: decode continuations and prefill
 * sequences packed in one varlen batch (the mixed decode / prefill batches
 * and chunked prefill of "[model] support Qwen3next").
 *   Sequences 0 .. n_decode-1 are decode rows: one token each, at rows
 *   0 .. n_decode-1 (cu_seqlens[i] = i for i <= n_decode).  Each continues
 *   the state in slot initial_state_indices[i] (< 0: the row is skipped and
 *   its o is zero; a new sequence, even of one token, belongs to the prefill
 *   part).  decode_in_place != 0 updates those slots in place (the
 *   streaming decode kernel; final_state_indices[i] is ignored for decode
 *   rows); decode_in_place == 0 writes the state after the token to
 *   final_state_indices[i] (< 0: dropped) and only reads the initial slot.
 *   Sequences n_decode .. n_seqs-1 run through gdn_prefill_chunked with
 *   cu_seqlens + n_decode (absolute token rows), the tail of both index
 *   arrays, and the workspace: size it with
 *   gdn_prefill_workspace_size(n_seqs - n_decode, n_tokens, ...).
 *   With 512 bytes more (and decode rows in place, bf16, dk = dv = 128), the
 *   decode rows run beside the prefill: the prefill goes first, and the
 *   streaming decode is launched behind its last kernel to take the SMs its
 *   chains leave free, with its items handed out by a counter kept in those
 *   extra bytes.  Decode rows and prompts must then use distinct slots (as
 *   slots within one call always must).
 * Other arguments, layouts and errors as gdn_prefill_chunked and
 * gdn_decode_recurrent (the decode rows need dk = dv <= 128 as those do).
 * Both halves' host-side checks run before either half launches, so a
 * failed check launches nothing, as for every entry point.  A batch whose
 * cu_seqlens[i] != i for some i <= n_decode breaks the decode-row layout:
 * it still runs (the decode half reads rows 0 .. n_decode-1) and sets
 * GDN_DEVSTAT_BAD_SEQLEN.
 */
gdn_status gdn_mixed_batch(const void *q, int64_t q_row_stride, const void *k,
                           int64_t k_row_stride, const void *v,
                           int64_t v_row_stride, const float *g,
                           const float *beta, const int32_t *cu_seqlens,
                           int32_t n_seqs, int32_t n_decode, int64_t n_tokens,
                           int32_t hqk, int32_t hv, int32_t dk, int32_t dv,
                           float scale, int32_t l2norm_qk, int32_t chunk,
                           float *state_pool, int64_t n_slots,
                           const int32_t *initial_state_indices,
                           const int32_t *final_state_indices,
                           int32_t decode_in_place, void *o, int32_t dtype,
                           void *workspace, size_t workspace_bytes,
                           void *stream);

/*
 * Whole-slot copy pool[dst[i]] <- pool[src[i]], bit for bit (the buffer copy
 * from source to destination indices of "[model] support Qwen3next", review
 * of the MTP buffer copy).  Used for the recurrent pool (slot_bytes =
 * hv*dv*dk*4) and the conv pool (slot_bytes = (width-1)*channels*elem).
 *   pool: base of [n_slots] slots of slot_bytes bytes each; 16-byte aligned,
 *      slot_bytes a multiple of 16.
 *   src, dst: [n] int32 device arrays; an entry < 0 on either side is
 *      skipped.  A slot used as a destination must not be a source in the
 *      same call.
 */
gdn_status gdn_state_snapshot(void *pool, int64_t n_slots, int64_t slot_bytes,
                              const int32_t *src, const int32_t *dst,
                              int32_t n, void *stream);

/*
 * Test control of the failure path (not for production use).  Sets the limit
 * of every bounded wait inside the two-kernel tensor-core prefill (the prep
 * and chain kernels of gdn_prefill_chunked with a workspace) to limit_ns
 * nanoseconds on the current device; 0 restores the default of one second.
 * With drop_prep_loads != 0 the prep kernel issues none of its K|Q tile
 * loads, so the waits for them run out after the limit: the kernel then
 * skips its stores, drains, frees its tensor memory, returns and sets
 * GDN_DEVSTAT_TIMEOUT, and the results of that call are undefined (every
 * index stays in bounds; the context stays usable).  Synchronises `stream`.
 * Restore both (0, 0) before production calls.
 */
gdn_status gdn_debug_set_wait_limit(uint64_t limit_ns, int32_t drop_prep_loads,
                                    void *stream);

/*
 * Reads the device status word (bits GDN_DEVSTAT_*) of the current device
 * into *out (a HOST pointer), synchronising `stream` first.  If clear != 0
 * the word is reset to 0 afterwards.
 */
gdn_status gdn_get_device_status(uint32_t *out, int32_t clear, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
