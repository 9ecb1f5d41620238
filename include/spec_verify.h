/*
 * spec_verify.h -- C ABI of the GB300 (sm_103a) batched speculative-decoding verifier.
 *
 * The library implements draft verification by modified rejection sampling as these sources
 * define it:
 *  - "Speculative Decoding in Custom LLM Servicing: Implementing Draft Models in Rust",
 *    sections "The Memory Bandwidth Wall and Speculative Math" (accept x_i with probability
 *    min(1, p(x_i)/q(x_i)); at the first rejection draw from max(0, p - q) normalised),
 *    "The Verification Algorithm" (the target's K+1 logit rows become softmax(logits / T);
 *    the loop stops at the first rejection; with every draft accepted the extra token is drawn
 *    from row K; only the accepted count and the correction token go back to the host) and
 *    "Orchestrating the Inference Loop" (the target KV cache keeps 1 + accepted of the K+1 rows).
 *  - "Adding Speculative Decoding", section "Verification and sampling": one batched verify
 *    over k+1 rows per request, requests with different k, greedy argmax compare as the
 *    degenerate case, the extra token honouring top-k/top-p/penalties; table "The existing
 *    base": greedy accepts while draft == argmax, the extra token is the argmax at the first
 *    mismatch.
 *  - FreeToken PR #836, section "Design": each verify row samples with its own request's
 *    temperature, top-k, top-p and greedy flag, and presence/frequency penalties count the
 *    drafts before the row as already generated (and, given a prior history, the tokens the
 *    request generated before its drafts).
 *
 * Conventions shared by every entry point:
 *  - Pointers named as device arrays must be CUDA device memory (or managed memory) that the
 *    caller owns and keeps alive until the work on `stream` has finished.  The library
 *    allocates no memory, makes no host<->device copy and does not synchronise; all work is
 *    enqueued on `stream` (a cudaStream_t; NULL means the legacy default stream).
 *  - Errors the host can see (null pointers, bad sizes, an unsupported shape, a workspace that
 *    is too small or misaligned) return at once with nothing enqueued.
 *  - Errors in device data (a draft token outside [0, V), num_drafts outside its range,
 *    T <= 0 or non-finite on a sampled request, top_p outside (0, 1], a uniform outside [0, 1),
 *    a non-finite penalty, inconsistent row_offsets, a malformed prior history) are found by
 *    the kernels.  The affected request's outputs become -1 and a sticky error word in the
 *    workspace records the first code; the call itself still returns SV_OK.
 *    sv_read_device_error() fetches the word.
 *    No kernel traps or asserts.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SV_OK = 0,
    SV_ERR_INVALID_ARG = 1,   /* null pointer, negative or inconsistent size, bad dtype  */
    SV_ERR_WORKSPACE = 2,     /* workspace too small or not 256-byte aligned             */
    SV_ERR_CUDA = 3,          /* a CUDA runtime call failed (a kernel launch)            */
    SV_ERR_UNSUPPORTED = 4,   /* shape outside what the kernels handle (V, k_max, B)     */
    SV_ERR_DEVICE_DATA = 5    /* returned only by sv_read_device_error: bad device data  */
} sv_status;

typedef enum { SV_F32 = 0, SV_BF16 = 1 } sv_dtype;

/* Device-data error codes stored in the workspace's sticky error word. */
enum {
    SV_DEV_OK = 0,
    SV_DEV_BAD_LAYOUT = 1,    /* num_drafts[b] < 0, > k_max, or rows of b inconsistent   */
    SV_DEV_BAD_TOKEN = 2,     /* a draft token outside [0, V)                            */
    SV_DEV_BAD_TEMPERATURE = 3,
    SV_DEV_BAD_TOP_P = 4,
    SV_DEV_BAD_UNIFORM = 5,
    SV_DEV_BAD_PENALTY = 6,
    SV_DEV_TIMEOUT = 7,       /* a wait of the streaming kernel ran out (2 s): every request
                                 has -1 outputs (spec_verify_lazy: every one not yet decided),
                                 except in one-pass calls over more rows than the select kernel
                                 holds at once (9 per SM), where only the requests with a row
                                 that was not streamed do; the others' outputs are exact    */
    SV_DEV_BAD_HISTORY = 8    /* prior history: offsets decrease or pass prior_len, an id outside
                                 [0, V), ids not strictly ascending, or a count below 1      */
};

/* Per-request sampling parameters: structure of device arrays, each of length B. */
typedef struct sv_params {
    const float *temperature;       /* > 0 and finite for sampled requests; unread when greedy   */
    const int32_t *top_k;           /* <= 0 or >= V: top-k off; else keep tokens >= k-th largest */
    const float *top_p;             /* in (0, 1]; 1 = off; keep v while mass strictly above < p  */
    const float *presence_penalty;  /* may be NULL (all 0): subtracted once from a drafted token */
    const float *frequency_penalty; /* may be NULL (all 0): subtracted per earlier occurrence    */
    const uint8_t *greedy;          /* 1 = greedy request (argmax prefix match), 0 = sampled     */
    /* Optional prior history of each request for the penalties (all three NULL: none).
     * Request b generated, before its drafts, the tokens prior_tokens[o_b .. o_{b+1}) --
     * distinct ids in [0, V), strictly ascending -- prior_counts[...] >= 1 times each, with
     * o = prior_offsets [B+1], o_0 = 0, non-decreasing, o_B <= prior_len.  A token's penalty
     * count on row i is its history count plus its count among the drafts before row i. */
    const int32_t *prior_offsets;
    const int32_t *prior_tokens;
    const int32_t *prior_counts;
    int32_t prior_len;              /* entries in prior_tokens / prior_counts (offsets beyond it are
                                       SV_DEV_BAD_HISTORY); ignored without a history            */
} sv_params;

/* Size in bytes of the device workspace spec_verify and spec_rollback need for a batch of B
 * requests and total_rows target rows of vocabulary V.  The workspace is caller-owned
 * device memory, 256-byte aligned; it needs no initialisation and may be reused by later
 * calls on the same stream (not by calls that run concurrently).  Returns 0 for invalid
 * sizes. */
size_t sv_workspace_bytes(int32_t B, int32_t total_rows, int32_t V);

/*
 * spec_verify -- verify the drafts of a batch of requests in one pass.
 *
 * Layout.  Request b owns target rows [row_offsets[b], row_offsets[b+1]) of target_logits and
 * the draft rows [row_offsets[b] - b, row_offsets[b+1] - b - 1) of draft_probs/draft_tokens; it
 * uses its first num_drafts[b] + 1 rows and num_drafts[b] drafts (ragged batches: pack with
 * row_offsets[b+1] - row_offsets[b] = num_drafts[b] + 1).  A request that owns no rows is a
 * layout error (-1 outputs); the draft rows of the request after it then start one slot early,
 * on the last draft slot of the requests before it, and either may write that slot's out_pq.
 * With row_offsets == NULL the
 * batch is uniform: target_logits [B, k_max+1, V], draft_probs [B, k_max, V], draft_tokens
 * [B, k_max], uniforms [B, k_max+1, 2], total_rows = B * (k_max + 1); requests may still use
 * fewer than k_max drafts.
 *
 *   target_logits  device [total_rows, V], row-major, dtype logits_dtype (bf16 or fp32);
 *                  16-byte aligned for the vectorised path (any alignment is accepted).
 *   draft_probs    device fp32 [total_rows - B, V]: the draft's distribution q_i per draft row.
 *                  Only q_i(x_i) is read for every sampled draft; whole rows only at a rejection.
 *   draft_tokens   device int32 [total_rows - B]: x_i, the drafted token ids.
 *   num_drafts     device int32 [B]: k_b, 0 <= k_b <= k_max.
 *   row_offsets    device int32 [B+1] (row_offsets[0] = 0, row_offsets[B] = total_rows), or NULL.
 *   B, k_max, V, total_rows: host sizes; 1 <= V <= 2^21, 0 <= k_max <= 64, 1 <= B < 2^25.
 *   params         per-request sampling parameters (device arrays of length B).
 *   uniforms       device fp32 [total_rows, 2] in [0, 1): slot 0 of row i is the accept test of
 *                  draft i; slot 1 of the row where the request stops is the residual draw (at a
 *                  rejection) or the extra-token draw (all drafts accepted).  Greedy requests read
 *                  none.
 *   out_tokens     device int32 [B, k_max+1]: accepted drafts, then the correction/extra token,
 *                  then -1 padding.  All -1 for a request with a device-data error.
 *   accept_len     device int32 [B]: number of accepted drafts a_b (-1 on a device-data error).
 *   out_pq         optional device fp32 [total_rows - B, 2]: (p_i(x_i), q_i(x_i)) for every draft
 *                  of a sampled request, whether or not the loop reached it; NaN for greedy
 *                  requests.  NULL skips it.
 *   workspace      device, sv_workspace_bytes() bytes, 256-byte aligned.
 *                  With a prior history, params.prior_tokens and prior_counts must be non-NULL
 *                  whenever prior_offsets is (SV_ERR_INVALID_ARG otherwise); a short prepass
 *                  kernel then checks each request's history and indexes it by 256-token
 *                  segment in the workspace.
 *   stream         cudaStream_t.  The call enqueues its kernels in stream order.  Its first
 *                  kernel is a programmatic dependent of the work before it on the stream and
 *                  waits for that work to complete; its last kernel lets the next launch on
 *                  the stream be scheduled early, so a kernel launched after it with
 *                  programmatic stream serialization must wait for its prerequisite grid
 *                  (cudaGridDependencySynchronize) before reading the outputs, as such a kernel
 *                  always must.  Ordinary launches, copies and events are unaffected.
 *
 * Per row the target distribution is p = softmax(z / T) over the tokens kept by top-k (every
 * token >= the k-th largest, ties kept) and then top-p (tokens whose renormalised mass strictly
 * above them is < top_p), renormalised; z_v = logit_v - presence * [c_v > 0] - frequency * c_v
 * with c_v the count of v among the request's drafts before the row plus its count in the
 * request's prior history (params.prior_*, optional).  A draft is accepted iff
 * p > 0 and (q == 0 or u < min(1, p/q)).  Draws use the inverse CDF in token-id order.
 * Arithmetic is fp32 (exp via ex2); a greedy row's argmax breaks ties toward the lowest id.
 * A logit of -inf masks its token: weight 0 under every filter, so it is never accepted
 * (p = 0) or drawn.  A row whose logits are all -inf has no distribution, and the results of
 * its request are unspecified.
 */
sv_status spec_verify(const void *target_logits, sv_dtype logits_dtype, const float *draft_probs,
                      const int32_t *draft_tokens, const int32_t *num_drafts, const int32_t *row_offsets,
                      int32_t B, int32_t k_max, int32_t V, int32_t total_rows, sv_params params,
                      const float *uniforms, int32_t *out_tokens, int32_t *accept_len, float *out_pq,
                      void *workspace, size_t workspace_bytes, void *stream);

/*
 * spec_verify_lazy -- spec_verify that reads no row after a request's first rejection.
 *
 * "Speculative Decoding in Custom LLM Servicing: Implementing Draft Models in Rust", section
 * "The Verification Algorithm": the verification loop returns at the first rejected draft, so
 * the target rows after it are never needed.  spec_verify reads every row in one pass, because
 * it cannot know the rejection point in advance; this entry point reads each request's row 0
 * first, decides that row, and then reads rows 1..k only of the requests whose draft 0 was
 * kept.  A rejection that needs the residual max(0, p - q) over a whole row (a row whose kept
 * set is too large for a list) is drawn by a last launch that splits the row over several
 * CTAs.  Fewer bytes are read when drafts are often rejected early; the second phase costs a
 * second round of row selection, so with high acceptance spec_verify is the faster call.
 *
 *   Arguments, layout, results, errors and workspace are those of spec_verify, and the results
 *   are the same, except out_pq: a request whose draft 0 is rejected has (p, q) for draft 0
 *   and NaN for the drafts after it (their rows are never read); the others have every draft's.
 *   The phase-event measurement aid does not apply.  Rows that are not 16-byte aligned, or a
 *   vocabulary the two-kernel path cannot hold, take spec_verify's one-pass path.
 */
sv_status spec_verify_lazy(const void *target_logits, sv_dtype logits_dtype, const float *draft_probs,
                           const int32_t *draft_tokens, const int32_t *num_drafts, const int32_t *row_offsets,
                           int32_t B, int32_t k_max, int32_t V, int32_t total_rows, sv_params params,
                           const float *uniforms, int32_t *out_tokens, int32_t *accept_len, float *out_pq,
                           void *workspace, size_t workspace_bytes, void *stream);

/*
 * spec_verify_onehot -- verify drafts proposed as one-hot (argmax) tokens.
 *
 * FreeToken PR #836, section "Design": when the draft model proposes its argmax, q_i is one-hot
 * at x_i, and sampling every verify row exactly as a decode step would (with the request's
 * temperature, top-k, top-p, greedy flag and the penalties of the drafts before the row), then
 * keeping the drafts while they equal those samples, is exact rejection sampling.  It reaches
 * the same distribution as spec_verify given one-hot q rows (accept with probability p_i(x_i);
 * at a rejection draw from p_i without x_i), but it uses the uniforms differently and reads no
 * q at all.
 *
 *   Arguments, layout and results are those of spec_verify, without draft_probs:
 *   uniforms       device fp32 [total_rows, 2]; only slot 1 is read: slot 1 of row i is row i's
 *                  sample (t_i = inverse CDF of p_i at u_{i,1}).  Slot 0 is not read or checked.
 *                  Greedy requests read none (their sample is the row's argmax).
 *   accept_len     a_b = the first i < k_b with t_i != x_i, else k_b.
 *   out_tokens     x_0 .. x_{a-1}, then t_a (the sample of the row where the request stops),
 *                  then -1 padding.
 *   out_pq         optional: (p_i(x_i), 1) for every draft of a sampled request (the one-hot q
 *                  puts mass 1 on its own token); NaN for greedy requests.
 *   workspace      sv_workspace_bytes(B, total_rows, V) bytes, as for spec_verify; spec_rollback
 *                  applies unchanged.
 * Errors are those of spec_verify, except that only slot 1 of the uniforms is checked.
 */
sv_status spec_verify_onehot(const void *target_logits, sv_dtype logits_dtype, const int32_t *draft_tokens,
                             const int32_t *num_drafts, const int32_t *row_offsets, int32_t B, int32_t k_max,
                             int32_t V, int32_t total_rows, sv_params params, const float *uniforms,
                             int32_t *out_tokens, int32_t *accept_len, float *out_pq, void *workspace,
                             size_t workspace_bytes, void *stream);

/*
 * spec_rollback -- commit the verify step to the target KV lengths.
 *
 * From "Speculative Decoding in Custom LLM Servicing: Implementing Draft Models in Rust",
 * "Orchestrating the Inference Loop": the verify step appended k_b + 1 rows to request b's
 * target KV cache and keeps 1 + accept_len[b] of them, so
 *     kv_seq_len[b] <- kv_seq_len[b] - (k_b + 1) + 1 + accept_len[b].
 * ("KV Cache Rollback Mechanics": rolling back forward is an error.)
 *
 *   kv_seq_len   device int32 [B], updated in place; it is also the committed length returned.
 *   accept_len   device int32 [B], as written by spec_verify.
 *   num_drafts   device int32 [B]: k_b (the argument spec_verify got).
 *   workspace    the spec_verify workspace (its sticky error word records failures).
 * A request with accept_len < 0 or > k_b, k_b < 0, or a result outside [0, kv_seq_len] keeps
 * its length and records SV_DEV_BAD_LAYOUT.
 *
 * The same call rolls back the draft model's cache: it appended the k_b drafts and keeps the
 * accepted ones, L - k_b + accept_len[b] (same section), which is the same update.
 */
sv_status spec_rollback(int32_t *kv_seq_len, const int32_t *accept_len, const int32_t *num_drafts,
                        int32_t B, void *workspace, void *stream);

/*
 * spec_verify_static -- spec_verify with a workspace that the library owns.
 *
 * The paper has no counterpart for this entry point (in place of a citation): its sources
 * verify drafts with whatever memory the serving process provides.  It exists for callers that
 * cannot provide device memory for a
 * workspace -- a host program with no device allocator of its own, or code that must not
 * allocate on the verification path.  It allocates nothing: the workspace is a device array of
 * SV_STATIC_WORKSPACE_BYTES (32 MiB) compiled into the library, present once per device.
 *
 *   Arguments, layout and results are those of spec_verify, without workspace and
 *   workspace_bytes.
 *   The first call on a device looks up the array's address (cudaGetSymbolAddress) with that
 *   device current; make that first call before any stream capture begins.
 *   A batch whose sv_workspace_bytes(B, total_rows, V) exceeds SV_STATIC_WORKSPACE_BYTES is
 *   rejected with SV_ERR_WORKSPACE before anything is enqueued.
 *   Every call on a device shares the one array: calls must be ordered (one stream, or events
 *   between streams).  Two calls that overlap in time race on it and their results are
 *   undefined.
 *   Device-data errors still turn the affected request's outputs into -1; the sticky error word
 *   itself stays inside the library's array.
 */
#define SV_STATIC_WORKSPACE_BYTES (32u << 20)

sv_status spec_verify_static(const void *target_logits, sv_dtype logits_dtype, const float *draft_probs,
                             const int32_t *draft_tokens, const int32_t *num_drafts, const int32_t *row_offsets,
                             int32_t B, int32_t k_max, int32_t V, int32_t total_rows, sv_params params,
                             const float *uniforms, int32_t *out_tokens, int32_t *accept_len, float *out_pq,
                             void *stream);

/* Reads the sticky device-data error word of a workspace (synchronises the device; meant for
 * tests and debugging).  *code receives an SV_DEV_* value, *first_bad_request the lowest
 * request index that set it (-1 if none).  Returns SV_OK when no error was recorded,
 * SV_ERR_DEVICE_DATA when one was, or SV_ERR_CUDA. */
sv_status sv_read_device_error(const void *workspace, int32_t *code, int32_t *first_bad_request);

/* Measurement aid: while set, every spec_verify call that takes the two-kernel path records
 * the two cudaEvent_t handles on its stream immediately before and after the stream kernel
 * (the kernel that reads every target row), so that the caller can time that kernel alone with
 * cudaEventElapsedTime.  Recording them separates the two kernels: the select kernel then no
 * longer overlaps the end of the stream kernel, so calls made while events are set run a
 * little slower.  Pass NULL, NULL to stop.  Process-wide, not thread-safe; the events stay
 * owned by the caller.  Returns SV_ERR_INVALID_ARG if only one handle is NULL. */
sv_status sv_set_phase_events(void *stream_kernel_start, void *stream_kernel_end);

/* Testing aid for the failure path: while `on` is nonzero, the streaming kernel of every
 * spec_verify / spec_verify_onehot / spec_verify_lazy call that takes the streaming path
 * (16-byte aligned rows) withholds one work unit from its copy and reduction warps, as a
 * stalled scheduler would.  Their bounded waits run out after 2 s; the call then completes
 * with -1 outputs for the requests SV_DEV_TIMEOUT describes, that code in the workspace's
 * error word, and the device stays usable.  No page has a counterpart: it exists so that the
 * timeout path can be tested without a GPU fault.  Process-wide, for every device; returns
 * SV_OK.  Never set it in production. */
sv_status sv_set_test_withhold(int32_t on);

/*
 * sv_prefer_lazy -- host-side choice between spec_verify and spec_verify_lazy for a batch.
 *
 * "Speculative Decoding in Custom LLM Servicing: Implementing Draft Models in Rust", section
 * "The Verification Algorithm": the loop returns at the first rejection, so spec_verify_lazy
 * skips the rows after row 0 of every request whose draft 0 is rejected, and pays a second
 * round of streaming and row selection for the requests that kept it.  Which call is faster
 * depends on how many requests reject draft 0, which only the caller can estimate (for example
 * the share of the previous step's requests that returned accept_len 0).  The function weighs
 * the two with a cost model fitted to both calls timed on a GB300: the skipped rows save their
 * bytes at 6.8 TB/s; the second round costs 10.3 us + 0.146 ns per vocabulary entry; with every
 * request rejecting draft 0 there is no second round.  Near the crossover the model leans to
 * spec_verify: it does not count the whole-row residual draws of rejected rows, which the
 * one-pass call pays more for.
 *
 *   B, total_rows, V, logits_dtype: the batch's sizes and logits type, as for spec_verify.
 *   row0_reject_share: the expected share, in [0, 1], of the B requests whose draft 0 is
 *                  rejected.
 * Returns 1 when spec_verify_lazy is expected to be the faster call, 0 when spec_verify is, and
 * -1 for invalid arguments (sizes as sv_workspace_bytes rejects them, an unknown dtype, a share
 * outside [0, 1] or NaN).  Host computation only: no device access, thread-safe.
 */
int32_t sv_prefer_lazy(int32_t B, int32_t total_rows, int32_t V, sv_dtype logits_dtype, float row0_reject_share);

/* Human-readable name of a status code. */
const char *sv_status_string(sv_status s);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
