/*
 * spec_verify.h -- C ABI of the GB300 (sm_103a) batched speculative-sampling
 * verify step.
 *
 * The operation (one call, B independent requests):
 *   For request b with gamma_b draft tokens x_0..x_{gamma_b-1}:
 *   1. p_i = softmax(t[b][i] / T_b) for the gamma_b + 1 target rows and
 *      q_i = softmax(d[b][i] / T_b) for the gamma_b draft rows.
 *      ("Fast Inference from Transformers via Speculative Decoding" explainer,
 *      PyTorch sketch Steps 1-2; toolsku "LLM speculative decoding
 *      optimisation", verify sketch.)
 *   2. Draft i is accepted iff u[b][i] < p_i(x_i) / q_i(x_i), the
 *      min(1, p/q) acceptance test; k is the first rejected position, or
 *      gamma_b when none is rejected.
 *      (disassemble-channel "Speculative Decoding theory", Step 3.)
 *   3. If k < gamma_b, one token is drawn at k from the residual
 *      max(0, p_k - q_k) / sum max(0, p_k - q_k) (from p_k if that sum is 0);
 *      otherwise a bonus token is drawn from p_{gamma_b}.  The draw is the
 *      inverse CDF over ascending token id driven by u[b][G]: the smallest j
 *      whose prefix sum exceeds u[b][G] times the total.
 *      (disassemble-channel, "modified distribution" and Step 3 bonus token.)
 *   Greedy mode replaces 1-3 by argmax matching: g_i = argmax t[b][i]
 *   (lowest id on ties), k = first i with x_i != g_i, and g_k is emitted.
 *   In spec_verify_sample a request with temperature exactly 0 takes these
 *   greedy steps (temperature -> 0 makes the acceptance an argmax match).
 *   (explainer, "Implementation points", greedy paragraph; zvxbase "draft
 *   length by load", K = 3 worked example.)
 *
 * Layouts (all row-major, rows contiguous with pitch V elements):
 *   target_logits  [B][G+1][V]  float32 or bf16
 *   draft_logits   [B][G][V]    same dtype as target_logits
 *   draft_tokens   [B][G]       int32, entries past gamma_b are ignored
 *   gamma          [B]          int32, 0 <= gamma_b <= G
 *   uniforms       [B][G+1]     float32 in [0,1): column i < gamma_b is the
 *                               acceptance draw of position i, column G the
 *                               resample/bonus draw
 *   temperature    [B]          float32, >= 0; 0 verifies that request by the
 *                               greedy steps below (no draft logits read)
 *   out_tokens     [B][G+1]     int32: x_0..x_{k-1}, the drawn token, then -1
 *   num_accepted   [B]          int32: accepted drafts k (emitted = k + 1)
 *
 * Ownership and concurrency: every pointer is caller-owned DEVICE memory, except
 * where a comment says host.  The library allocates and frees nothing and never
 * synchronises the stream (spec_verify_status excepted).  The workspace must be
 * zero-filled once when allocated; every call leaves it zeroed again, so one
 * workspace serves any number of calls issued in order on one stream.  Two
 * calls that may run concurrently need two workspaces.
 *
 * Errors: each entry point returns SV_OK (0) or a negative SV_ERR_* code, and
 * on error launches nothing.  Values inside device arrays cannot be checked on
 * the host: a gamma_b outside [0, G], a draft token outside [0, V), a uniform
 * outside [0, 1), a negative or non-finite temperature, or a row with no
 * finite logit (among the rows a call reads: spec_verify_set_lazy) sets a
 * bit in the workspace's status word (read it with
 * spec_verify_status) and is clamped to a legal value, so no call reads or
 * writes outside the arrays described above.  NaN logits are not supported.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t); NULL means the legacy default stream. */
typedef struct CUstream_st *sv_stream_t;

typedef enum { SV_F32 = 0, SV_BF16 = 1 } sv_dtype;

enum {
  SV_OK = 0,
  SV_ERR_SCALAR = -1,    /* B < 0, G outside [0, SV_MAX_GAMMA], V outside [1, SV_MAX_VOCAB], bad dtype */
  SV_ERR_NULL = -2,      /* a required pointer is NULL */
  SV_ERR_ALIGN = -3,     /* a pointer is not aligned to its element (workspace: 256 bytes) */
  SV_ERR_WORKSPACE = -4, /* ws_bytes < spec_verify_workspace_size(B, G, V) */
  SV_ERR_CUDA = -5,      /* the kernel launch failed (cudaGetLastError) */
  SV_ERR_STATIC_LIMIT = -6 /* spec_verify_sample_noalloc: the sizes need more scratch than
                              SV_NOALLOC_SCRATCH_BYTES */
};

/* Status-word bits set on the device for invalid values inside arrays. */
enum {
  SV_STATUS_BAD_GAMMA = 1u,       /* gamma_b outside [0, G]: clamped */
  SV_STATUS_BAD_TOKEN = 2u,       /* draft token outside [0, V): clamped */
  SV_STATUS_BAD_UNIFORM = 4u,     /* uniform outside [0, 1) or NaN: replaced by 0 */
  SV_STATUS_BAD_TEMPERATURE = 8u, /* temperature < 0, inf or NaN: replaced by 1 */
  SV_STATUS_NONFINITE_ROW = 16u,  /* a row whose maximum is not finite (among the rows the
                                     call reads: see spec_verify_set_lazy) */
  SV_STATUS_INTERNAL = 32u,       /* an inverse-CDF draw found no token (never expected) */
  SV_STATUS_TIMEOUT = 64u         /* a bounded wait for a request's decision ran out; the
                                     request's outputs are incomplete and the workspace must
                                     be zero-filled again before reuse */
};

#define SV_MAX_GAMMA 31
#define SV_MAX_VOCAB (1 << 24)
/* Size of the scratch array built into the library for spec_verify_sample_noalloc. */
#define SV_NOALLOC_SCRATCH_BYTES (4u << 20)

/*
 * Bytes of device workspace that spec_verify_sample / spec_verify_greedy need
 * for these sizes (a multiple of 256); 0 if the sizes are invalid.
 */
size_t spec_verify_workspace_size(int B, int G, int V);

/*
 * Sampling verify step (steps 1-3 above) for B requests on `stream`.
 *   target_logits, draft_logits: device, dtype `dtype`, layouts above;
 *     draft_logits may be NULL when G == 0.
 *   draft_tokens: device int32 [B][G] (may be NULL when G == 0).
 *   gamma, uniforms, temperature: device, layouts above.
 *   out_tokens, num_accepted: device outputs, layouts above.
 *   p_tok, q_tok: optional device float64 [B][G] outputs (NULL to skip):
 *     p_i(x_i) and q_i(x_i) for evaluated positions i <= k (i < gamma_b), NaN
 *     elsewhere.
 *   workspace: device, 256-byte aligned, ws_bytes >= spec_verify_workspace_size,
 *     zero-filled before its first use.
 * B == 0 is a no-op.  Returns SV_OK or an SV_ERR_* code.
 */
int spec_verify_sample(const void *target_logits, const void *draft_logits, sv_dtype dtype,
                       int B, int G, int V, const int32_t *draft_tokens,
                       const int32_t *gamma, const float *uniforms,
                       const float *temperature, int32_t *out_tokens,
                       int32_t *num_accepted, double *p_tok, double *q_tok,
                       void *workspace, size_t ws_bytes, sv_stream_t stream);

/*
 * Greedy (argmax-match) verify step on the target rows only; no draft logits,
 * uniforms or temperature.  Arguments as for spec_verify_sample.
 */
int spec_verify_greedy(const void *target_logits, sv_dtype dtype, int B, int G, int V,
                       const int32_t *draft_tokens, const int32_t *gamma,
                       int32_t *out_tokens, int32_t *num_accepted, void *workspace,
                       size_t ws_bytes, sv_stream_t stream);

/*
 * Packed (varlen) layout: the same steps for requests whose rows are stored
 * back to back without padding, as serving engines lay out ragged verify
 * batches ("speculative decoding: draft length by load", per-request draft
 * lengths K; the padded layout above wastes (G - gamma_b) rows per request).
 *   cu_draft      device int32 [B+1]: cu_draft[0] = 0, cu_draft[b+1] - cu_draft[b]
 *                 = gamma_b in [0, G]; total_drafts (host) = cu_draft[B].
 *   target_logits [total_drafts + B][V]: request b's gamma_b + 1 target rows start
 *                 at row cu_draft[b] + b.
 *   draft_logits  [total_drafts][V]: request b's rows start at cu_draft[b]
 *                 (may be NULL when total_drafts == 0).
 *   draft_tokens  [total_drafts] int32, aligned with the draft rows.
 *   uniforms      [total_drafts + B] float32, one per target row: request b's
 *                 entry cu_draft[b] + b + i is the acceptance draw of draft i
 *                 (i < gamma_b), entry cu_draft[b] + b + gamma_b its final draw.
 *   p_tok, q_tok  optional float64 [total_drafts], aligned with the draft tokens.
 *   temperature [B], out_tokens [B][G+1], num_accepted [B]: as in the padded calls
 *   (G is the largest draft length; it sizes out_tokens and the workspace,
 *   spec_verify_workspace_size(B, G, V)).
 * A request whose cu_draft entries are inconsistent (negative, decreasing, past
 * total_drafts, or a length above G) sets SV_STATUS_BAD_GAMMA and is verified with
 * no drafts at an offset clamped into the arrays: no access leaves them.
 * Returns SV_OK, or SV_ERR_* as the padded calls (SV_ERR_SCALAR also for
 * total_drafts < 0).
 */
int spec_verify_sample_packed(const void *target_logits, const void *draft_logits,
                              sv_dtype dtype, int B, int G, int V, const int32_t *cu_draft,
                              int total_drafts, const int32_t *draft_tokens,
                              const float *uniforms, const float *temperature,
                              int32_t *out_tokens, int32_t *num_accepted, double *p_tok,
                              double *q_tok, void *workspace, size_t ws_bytes,
                              sv_stream_t stream);

/* Greedy verify step on the packed layout (target rows and draft tokens as in
 * spec_verify_sample_packed; no draft logits, uniforms or temperature). */
int spec_verify_greedy_packed(const void *target_logits, sv_dtype dtype, int B, int G, int V,
                              const int32_t *cu_draft, int total_drafts,
                              const int32_t *draft_tokens, int32_t *out_tokens,
                              int32_t *num_accepted, void *workspace, size_t ws_bytes,
                              sv_stream_t stream);

/*
 * Draft-token sampler: for each of B rows, one token from softmax(logits[b] /
 * temperature[b]) by the inverse CDF over ascending token id driven by
 * uniforms[b] (the smallest j whose prefix sum exceeds uniforms[b] times the
 * total); temperature[b] == 0 returns the row's argmax (lowest id on ties).
 * This is the draw a draft model makes at each of its steps ("Speculative
 * Decoding theory", step 1, draft generation x ~ q), and the same computation
 * as spec_verify_sample's bonus draw with G == 0.
 *   logits: device [B][V] float32 or bf16; uniforms, temperature: device [B]
 *   float32; tokens: device int32 [B] output.
 *   workspace: as for spec_verify_sample, sized spec_verify_workspace_size(B, 0, V).
 * Returns SV_OK or an SV_ERR_* code; invalid device values set status bits as
 * described above.
 */
int spec_verify_draw(const void *logits, sv_dtype dtype, int B, int V, const float *uniforms,
                     const float *temperature, int32_t *tokens, void *workspace,
                     size_t ws_bytes, sv_stream_t stream);

/*
 * spec_verify_sample_noalloc: spec_verify_sample with no caller workspace.
 * The pages on speculative decoding describe no such call: this is a
 * convenience of this library's interface, not a step of the method.
 *
 * Who needs it: callers that may not obtain device memory when they verify.
 * A serving loop that handed all free device memory to weights and the KV
 * cache when it started, and must not grow its footprint later, is one; C
 * code that drives this library without any device allocator of its own is
 * another.  This call allocates and frees nothing.
 *
 * Scratch: an array of SV_NOALLOC_SCRATCH_BYTES (4 MiB) that lives in the
 * library's device image.  If spec_verify_workspace_size(B, G, V) is larger,
 * the call returns SV_ERR_STATIC_LIMIT and runs nothing (4 MiB holds, for
 * example, B = 512 requests with G = 3 and V = 128256).
 *
 * First call on a device: it looks up the array's device address with
 * cudaGetSymbolAddress while that device is current and keeps it for later
 * calls on the same device (SV_ERR_CUDA if the look-up fails).  Make that
 * first call before any stream capture begins.  The kept address belongs to
 * the device's primary context: after cudaDeviceReset on that device it is
 * stale, and a later call would launch on a freed address.  A process that
 * resets a device must not call spec_verify_sample_noalloc on it again.
 *
 * Sharing: every call in the process uses the same array.  Each call first
 * zeroes the array's counters and flags (an asynchronous memset on `stream`),
 * then launches the same kernel as spec_verify_sample; the per-chunk partial
 * results stay in the array as the last call left them.  Calls that can
 * overlap on the GPU (other streams without ordering between them, other host
 * threads) race on the array and produce wrong results: issue them in order
 * on one stream.  Because of the memset, the status bits of spec_verify_status
 * are not available from this call; invalid device values are still clamped
 * as described at the top of this file.
 *
 * Arguments, layouts and the other return codes: as spec_verify_sample,
 * without workspace and ws_bytes.
 */
int spec_verify_sample_noalloc(const void *target_logits, const void *draft_logits,
                               sv_dtype dtype, int B, int G, int V,
                               const int32_t *draft_tokens, const int32_t *gamma,
                               const float *uniforms, const float *temperature,
                               int32_t *out_tokens, int32_t *num_accepted, double *p_tok,
                               double *q_tok, sv_stream_t stream);

/*
 * Copies the workspace's status word (SV_STATUS_* bits accumulated since the
 * last read) to *status_host (a HOST pointer), then clears it.  Synchronises
 * `stream`.  Returns SV_OK, SV_ERR_NULL or SV_ERR_CUDA.
 */
int spec_verify_status(void *workspace, sv_stream_t stream, uint32_t *status_host);

/* Static English text for an SV_OK / SV_ERR_* code. */
const char *spec_verify_strerror(int code);

/*
 * Schedules.  Three kernels compute every value with the same arithmetic, so
 * outputs do not depend on the schedule:
 *   - the resident cluster path: a batch small enough that one thread-block
 *     cluster per request fits on the GPU at once, with each warp holding one
 *     chunk of a draft position's target and draft rows in shared memory.  The
 *     partials, the decision and the residual block sums move through the
 *     cluster's shared memory, and the final draw walks resident data;
 *   - the streaming cluster path: one cluster per request as well, for batches
 *     of up to one cluster per SM (clusters of up to 16 CTAs, at least one),
 *     the warps streaming the request's chunks two at a time and re-reading
 *     the rejected row's chunks for the residual.  For larger batches the same
 *     kernel runs as one CTA per SM (sampling) or two (greedy), each taking
 *     whole requests in turn from a claim counter, longest request first
 *     (SV_ROUTE_CLAIMS).  The claim order takes 5 bytes of shared memory per
 *     request.  A sampling call of at least two requests per SM whose
 *     positions are read lazily (spec_verify_set_lazy) runs instead on a
 *     pipeline kernel (SV_ROUTE_PIPELINE): one CTA per SM keeps two requests
 *     in flight, its warps moving from one request's items to the other's
 *     without a barrier, and the warp that completes a stage, a residual pass
 *     or a draw runs what follows it;
 *   - the persistent grid, for batches whose claim order does not fit (tens
 *     of thousands of requests): chunks claimed from global counters,
 *     decisions published through global records.
 * The cluster paths replace the persistent grid's chain of global-memory
 * synchronisations (arrival counters, decision records, queue) with cluster
 * barriers.  These calls are not steps of the method: they exist for testing
 * and measurement.
 *
 * spec_verify_set_schedule: the policy for the calls that follow in this
 * process: SV_SCHEDULE_AUTO (the default: the first of the resident cluster
 * path, the streaming cluster path and the persistent grid that applies, as
 * above), SV_SCHEDULE_PERSISTENT (every call on the persistent grid) or
 * SV_SCHEDULE_STREAM (as AUTO without the resident path).  Returns the
 * previous policy, or SV_ERR_SCALAR for an unknown value.  SV_SCHEDULE_STREAM
 * also leaves out the pipeline kernel (its claims run on the streaming
 * kernel).
 *
 * spec_verify_route: the kernel (SV_ROUTE_*) that the next sampling
 * (greedy == 0) or greedy call of this shape, in the padded layout, on the
 * current device would use under the current policy, or SV_ERR_SCALAR for
 * invalid sizes.  If cluster_size is not NULL (a HOST pointer), it receives
 * the cluster size (CTAs per request) of a cluster path (1 for claims and the
 * pipeline), or 0.
 *
 * spec_verify_cluster_size: that cluster size alone (0 for the persistent
 * grid), or SV_ERR_SCALAR.
 */
#define SV_SCHEDULE_AUTO 0
#define SV_SCHEDULE_PERSISTENT 1
#define SV_SCHEDULE_STREAM 2
#define SV_ROUTE_PERSISTENT 0
#define SV_ROUTE_CLUSTER 1
#define SV_ROUTE_STREAM 2
#define SV_ROUTE_CLAIMS 3
#define SV_ROUTE_PIPELINE 4
int spec_verify_set_schedule(int schedule);
int spec_verify_route(sv_dtype dtype, int B, int G, int V, int greedy, int *cluster_size);

/*
 * spec_verify_set_wait_limit: the limit, in nanoseconds of the GPU's global
 * timer, of every bounded wait in the calls that follow in this process (a
 * bulk copy's completion, a decision record, a queue slot); 0 restores the
 * default of 2 s.  A wait that runs out sets SV_STATUS_TIMEOUT and its warp
 * stops taking work, so the call returns with incomplete outputs and the
 * workspace must be zero-filled again (as documented for that bit).  Not a
 * step of the method: it exists so that tests can make a wait run out
 * quickly.  Returns the previous limit.
 */
unsigned long long spec_verify_set_wait_limit(unsigned long long ns);

/*
 * spec_verify_set_lazy: how the request-claims schedules (SV_ROUTE_CLAIMS,
 * SV_ROUTE_PIPELINE) read a request's rows in the calls that follow in this
 * process.
 * 1 (the default): position by position.  In a greedy call (or a request
 * with temperature 0) target row i is reduced to its argmax and compared
 * with draft i before row i + 1 is read; the call stops at the first draft
 * that differs.  For a sampled request the target and draft rows of
 * position i are reduced and draft i is tested before the rows of position
 * i + 1 matter, and the bonus row gamma_b only after every draft was
 * accepted, as in the verification loop of disassemble-channel
 * "Speculative Decoding theory", Step 3, which stops at the first rejected
 * draft.  On the streaming kernel's claims, for a request with at least four
 * drafts, the CTA streams the next position while one is tested (what it read
 * of a position after the first rejection is not used); the pipeline kernel
 * instead streams its other request's position meanwhile.  Lazy stages lengthen a request while they shorten
 * the batch, so sampled requests are read this way only where the batch
 * holds at least two requests per CTA, and not when a request's rows alone
 * reach 80 % of a CTA's share of the batch's rows.  0: every row of every
 * request is reduced before any
 * test.  The outputs are identical either way: a position's arithmetic does
 * not depend on the order.  The other schedules always read every row.
 * Returns the previous setting, or SV_ERR_SCALAR for a value other than 0
 * or 1.
 */
int spec_verify_set_lazy(int on);
int spec_verify_cluster_size(sv_dtype dtype, int B, int G, int V, int greedy);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
