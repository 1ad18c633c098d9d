/*
 * gdn.h -- C ABI of the Gated Delta Net prefill in libgemm_f16.so (GB300, sm_103a).
 *
 * The operation (page "TIRx" (zixuwang.me), section "用状态递推解释 GDN"): every sequence and
 * value head carries a state H of shape [dv, dk].  Token by token:
 *
 *     H_decay    = alpha_t * H
 *     prediction = H_decay k_t
 *     update     = beta_t * (v_t - prediction)
 *     H          = H_decay + update k_t^T
 *     o_t        = scale * H q_t
 *
 * The kernels evaluate this recurrence in 64-token chunks (the page's GPU form): per chunk the
 * decays' running products, the chunk's K K^T and Q K^T, and the triangular solve that turns the
 * chunk's updates into matrix products; then a scan over each sequence's chunks carries the state
 * and writes the outputs.  Arithmetic is fp32 throughout; the result differs from the
 * token-by-token order only by rounding.
 *
 * Packed input (same page): the tokens of n_seqs independent sequences lie back to back;
 * sequence i owns tokens cu_seqlens[i] .. cu_seqlens[i+1]-1 and its own state, and a sequence's
 * replay never crosses its boundary.  The host never reads cu_seqlens: it is a device array, and
 * the call's first kernel checks it on the device before any token is touched.  Offsets that
 * break the contract below (a first offset other than 0, a last one other than total_tokens, or
 * a decreasing pair) are refused there: every sequence is then taken as empty, no token of q, k,
 * v, alpha, beta or o is read or written, the final states (if asked for) equal the initial
 * ones, and gdn_check_status returns GDN_ERR_INVALID_ARG for the call.  A one-sequence call,
 * which numbers its chunks from total_tokens, requires cu_seqlens = [0, total_tokens] the same
 * way.
 *
 * Heads (the page's three relations: MHA, GQA, GVA).  q has h_q heads, k h_k, and v, alpha,
 * beta and the states h_v, a multiple of h_k; state head j reads key head j / (h_v / h_k).
 *   h_q == h_k            o has h_v heads; state j reads query head j / (h_v / h_k) and writes
 *                         output head j (h_v == h_k: multi-head attention; larger: grouped
 *                         values, GVA)
 *   h_q a multiple of h_v o has h_q heads; query head m reads state m / (h_q / h_v) and writes
 *                         output head m (grouped queries, GQA; at most 8 query heads per state).
 *                         The state recurrence does not read q: the call runs the pipeline once
 *                         per query head of a group, each pass reproducing the same states.
 * gdn_prefill is gdn_prefill_heads with h_q == h_k == h_qk.
 *
 * Layouts (row-major, device memory of the current device):
 *   q              bfloat16 [total_tokens][h_q][head_dim]
 *   k              bfloat16 [total_tokens][h_k][head_dim]
 *   v              bfloat16 [total_tokens][h_v][head_dim]
 *   alpha, beta    float    [total_tokens][h_v]     alpha in (0, 1]; beta any real
 *   cu_seqlens     int32    [n_seqs + 1], non-decreasing, cu_seqlens[0] = 0,
 *                                     cu_seqlens[n_seqs] = total_tokens
 *   initial_state  float    [n_seqs][h_v][head_dim (dv)][head_dim (dk)], or NULL for zeros
 *   o              bfloat16 [total_tokens][h_o][head_dim]   (written; h_o as above)
 *   final_state    float    [n_seqs][h_v][dv][dk], or NULL   (written; may be the
 *                                     initial_state buffer itself, updated in place)
 *   workspace      gdn_prefill_workspace_bytes() bytes, 16-byte aligned
 *
 * The chunked form divides running products of alpha within a chunk, so every alpha must be
 * positive and the product of 64 consecutive alphas of a sequence must stay a normal fp32 number
 * (above 1e-37); alpha = 0, a full reset, is outside this routine's domain.
 *
 * Ownership: the caller owns every buffer; nothing is retained after a call.  Apart from the
 * state pair above, no written buffer may overlap another buffer of the call.  Asynchronous on
 * `stream`, in stream order: every kernel of a call is launched with programmatic dependent
 * launch, so it may be placed while the kernel before it finishes; the call's first kernel waits
 * for all earlier work on the stream before it reads or writes anything, the later ones before
 * they touch what an earlier kernel of the call writes.  A call enqueues kernel launches
 * only (no allocation, copy or synchronisation), so it may be recorded into a CUDA graph; the
 * first call on each device also sets the kernels' shared-memory attributes, so make that one
 * outside a capture.  Errors: GDN_ERR_INVALID_ARG (null pointer, negative size, heads in none of the
 * layouts above, workspace too small), GDN_ERR_UNSUPPORTED (head_dim other than 128, misaligned
 * q/k/v/o, more than 8 query heads per state head, more than 2^31 / 192 chunks x value heads),
 * GDN_ERR_CUDA (a launch failed;
 * gdn_last_error() says why).  Nothing is enqueued on an error.  n_seqs == 0 does nothing.
 *
 * Device-side failure: every wait of the scan kernel for a chunk's loads is bounded (default
 * 2000 ms, gdn_set_wait_timeout_ms).  A wait that runs out makes the kernel stop cleanly and set
 * a status word in the workspace, which gdn_check_status reads (GDN_ERR_TIMEOUT); the outputs of
 * that call are then undefined.  Each gdn_prefill call clears the word when it starts.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GDN_OK 0
#define GDN_ERR_INVALID_ARG 1
#define GDN_ERR_UNSUPPORTED 2
#define GDN_ERR_CUDA 3
#define GDN_ERR_TIMEOUT 4

/* Workspace bytes gdn_prefill needs for these sizes (an upper bound over all packings). */
int gdn_prefill_workspace_bytes(int64_t total_tokens, int64_t n_seqs, int64_t h_v,
                                size_t* bytes);

/* The gated delta rule over packed sequences, as above, q and k sharing h_qk heads. */
int gdn_prefill(const void* q, const void* k, const void* v, const float* alpha,
                const float* beta, const int32_t* cu_seqlens, int64_t n_seqs,
                int64_t total_tokens, int64_t h_qk, int64_t h_v, int64_t head_dim, float scale,
                const float* initial_state, void* o, float* final_state, void* workspace,
                size_t workspace_bytes, cudaStream_t stream);

/* The same with separate query, key and value head counts (MHA, GVA and GQA, as above). */
int gdn_prefill_heads(const void* q, const void* k, const void* v, const float* alpha,
                      const float* beta, const int32_t* cu_seqlens, int64_t n_seqs,
                      int64_t total_tokens, int64_t h_q, int64_t h_k, int64_t h_v,
                      int64_t head_dim, float scale, const float* initial_state, void* o,
                      float* final_state, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream);

/* The message of the calling thread's last failed gdn_* call ("" if none). */
const char* gdn_last_error(void);

/* Waits for `stream`, then reads the status word of the last gdn_prefill (or
 * gdn_check_offsets) call that used `workspace`: GDN_OK; GDN_ERR_INVALID_ARG if that call's
 * cu_seqlens broke its contract (nothing was processed); GDN_ERR_TIMEOUT if a scan CTA gave up a
 * bounded wait; GDN_ERR_CUDA if the stream reported an error. */
int gdn_check_status(const void* workspace, cudaStream_t stream);

/* Checks cu_seqlens [n_seqs + 1] (device memory) against the contract above on the device, with
 * the one small kernel a packed gdn_prefill call starts with, and nothing after it: it reads the
 * n_seqs + 1 offsets and writes only the workspace (sized by gdn_prefill_workspace_bytes for
 * total_tokens, n_seqs, h_v).  Asynchronous on `stream`; gdn_check_status then returns
 * GDN_ERR_INVALID_ARG for offsets that break the contract, else GDN_OK.  Errors as for
 * gdn_prefill (argument checks on the host; nothing is enqueued on an error). */
int gdn_check_offsets(const int32_t* cu_seqlens, int64_t n_seqs, int64_t total_tokens,
                      int64_t h_v, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* The same rule on a host copy of the offsets (1: valid, 0: not); the device check and this
 * function share one definition of the rule.  Host-only. */
int gdn_offsets_valid_host(const int32_t* cu_seqlens, int64_t n_seqs, int64_t total_tokens);

/* Limit of one wait of the scan kernel for a chunk's loads, for later calls of this process
 * (ms >= 1; default 2000). */
int gdn_set_wait_timeout_ms(uint32_t ms);

/* Which kernel runs the scan over each sequence's chunks, for later calls of this process:
 * GDN_SCAN_AUTO (default) and GDN_SCAN_TENSOR_CORE run its chunk products as tcgen05.mma streams
 * from shared memory into tensor memory, with 32 state rows per work item when 16-row items
 * would give every SM at least two, else 16; GDN_SCAN_TENSOR_CORE_16 / _32 fix the row count;
 * GDN_SCAN_MMA_SYNC runs the products as register-tile mma.sync.  All compute the same
 * recurrence at the same precision (fp32 operands as three bfloat16 pieces); the switch exists
 * for comparison and measurement. */
#define GDN_SCAN_AUTO 0
#define GDN_SCAN_TENSOR_CORE 1
#define GDN_SCAN_MMA_SYNC 2
#define GDN_SCAN_TENSOR_CORE_16 3
#define GDN_SCAN_TENSOR_CORE_32 4
int gdn_set_scan_kernel(int kernel);

/* Testing hook, 0 = off (default).  1: the scan kernels never issue the loads of each sequence's
 * second chunk, so the wait for them runs out (nothing is in flight) and the call reports
 * GDN_ERR_TIMEOUT through gdn_check_status.  For failure-detection tests only. */
int gdn_set_fault_injection(int mode);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
