/*
 * cpe.h — C ABI of libcpe, chunked-prefill extend attention on GB300 (sm_103a).
 *
 * The library computes one round of chunked prefill for a batch of sequences:
 * sequence s has P_s tokens already in a paged KV cache (prefix_len) and E_s new
 * query tokens at positions [P_s, P_s + E_s) (qo_indptr).  Each new query row i
 * attends to keys [0, P_s + i]: the cached prefix as an unmasked rectangle and
 * its own chunk as a causal triangle, merged by their log-sum-exp statistics.
 *   SGLang chunked-prefill article (zdszero.github.io/chunked_prefill.html),
 *   section "turning one prefill into resumable extends": P_t, E_t, S_t, the
 *   output o_i, Stage 1 / Stage 2 and the online-softmax merge.
 * Decode rows are sequences with E_s = 1 (context length L = P_s + 1).
 *
 * Conventions shared by every entry point
 *  - The caller owns all memory.  The library allocates nothing and frees
 *    nothing, and it never synchronises a stream except in
 *    cpe_get_device_status().
 *  - Host arrays are marked (host); every other pointer is device memory.
 *  - Launches are asynchronous on the given stream (NULL = legacy default).
 *  - Errors are returned as cpe_status, never thrown.  Argument errors are
 *    found on the host before any launch and nothing is launched; a message is
 *    available from cpe_last_error() on the calling thread.  Errors found on
 *    the device (a page id out of range, a length above max_kv_len, a pipeline
 *    wait that gave up) are recorded in a device status word that
 *    cpe_get_device_status() reads and clears.  The library looks up the
 *    word's device address once per device and keeps it, so a
 *    cudaDeviceReset in the process voids it: use the library on a device
 *    only while the context of its first call there is alive.
 *  - Layouts are row-major with the last dimension contiguous:
 *      q, out       [total_q, H_q, d]
 *      k_new, v_new [total_q, H_kv, d]
 *      k/v cache    [num_pages, page_size, H_kv, d]
 *      page_table   [n_seqs, max_pages] int32 (page ids; entries past a
 *                   sequence's last page are never read)
 *    Cache slots past a sequence's last token in its last page must hold
 *    finite values (zero-initialised pages do): the tensor-core path loads
 *    whole 16-token steps and meets them with zero weights, and 0 x (inf or
 *    NaN) is NaN.
 *      qo_indptr    [n_seqs + 1] int32, qo_indptr[0] = 0, non-decreasing,
 *                   qo_indptr[n_seqs] = total_q
 *      prefix_len   [n_seqs] int32
 *      lse          [total_q, H_q] float32, natural log, m + ln(l) over the
 *                   scaled scores
 *  - Query head h reads KV head floor(h / G), G = H_q / H_kv.
 *  - Supported: d in {64, 128}; H_q % H_kv == 0 and G in {1, 2, 4, 8, 16};
 *    page_size = 16; dtype CPE_BF16 (bf16 in and out, fp32 accumulation) or
 *    CPE_F32 (fp32 in and out).  Every device pointer 16-byte aligned.
 */
#ifndef CPE_H
#define CPE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* cpe_stream_t; /* the same type as cudaStream_t */

typedef enum cpe_status {
    CPE_OK = 0,
    CPE_ERR_INVALID_ARG = 1, /* null pointer, length <= 0, inconsistent sizes     */
    CPE_ERR_UNSUPPORTED = 2, /* shape or dtype outside the supported set         */
    CPE_ERR_CAPACITY = 3,    /* output or workspace buffer too small             */
    CPE_ERR_CUDA = 4,        /* a CUDA runtime or driver call failed             */
    CPE_ERR_TIMEOUT = 5,     /* device: a pipeline wait gave up (kernel returned) */
    CPE_ERR_DEVICE_ARG = 6   /* device: bad page id / length found in device data */
} cpe_status;

typedef enum cpe_dtype { CPE_F32 = 0, CPE_BF16 = 1 } cpe_dtype;

/*
 * One chunk of a chunked prefill.
 *   msmodeling RFC "Chunked Prefill modelling support", section 3.1.3
 *   (PrefillChunk: index, query_len, seq_len), extended with the cursor of the
 *   SGLang article: the round computes positions [prefix_len, seq_len).
 *   prefix_len    P_t: tokens before this chunk, cached prefix included
 *   query_len     E_t: tokens computed in this chunk
 *   seq_len       S_t = P_t + E_t
 *   model_seq_len the RFC's seq_len: tokens of the effective (uncached) part
 *                 consumed once this chunk is done (cached prefix left out)
 */
typedef struct cpe_chunk {
    int32_t index;
    int32_t prefix_len;
    int32_t query_len;
    int32_t seq_len;
    int32_t model_seq_len;
} cpe_chunk;

/*
 * cpe_plan_chunks — the chunk plan of one request (host only).
 *   msmodeling RFC, section 2.2: cached = floor(input_len * prefix_hit_rate)
 *   in IEEE double, effective = input_len - cached; section 3.1.3: chunks of
 *   min(chunk_size, remaining) tokens.  SGLang article, implementation
 *   section: with align_to > 0 only a truncated first chunk has its absolute
 *   end rounded down to a multiple of align_to (0 = no alignment).
 * out (host) receives up to cap records; *n_out (host) the number of chunks.
 * cached_out / effective_out (host, nullable) receive the two lengths; the
 * decode context stays input_len.
 * Errors: CPE_ERR_INVALID_ARG if chunk_size <= 0, input_len <= 0, the hit
 * rate is outside [0, 1], effective < 1, align_to < 0, or a position exceeds
 * INT32_MAX; CPE_ERR_CAPACITY if cap is below the chunk count (*n_out still
 * holds the count).
 */
cpe_status cpe_plan_chunks(int64_t input_len, double prefix_hit_rate, int32_t chunk_size,
                           int32_t align_to, cpe_chunk* out, int32_t cap, int32_t* n_out,
                           int64_t* cached_out, int64_t* effective_out);

/*
 * cpe_plan_budget — token-budget truncation (host only).
 *   vLLM token-budget tutorial, section 5: requests in order each take
 *   min(need, remaining budget); a decode request needs 1 token.
 * need[n_req] (host) in, granted[n_req] (host) out, *used (host, nullable) =
 * sum of granted.  Errors: CPE_ERR_INVALID_ARG for token_budget <= 0,
 * n_req < 0, a negative need, or null arrays with n_req > 0.
 */
cpe_status cpe_plan_budget(int32_t token_budget, int32_t n_req, const int32_t* need,
                           int32_t* granted, int32_t* used);

/*
 * cpe_plan_mixed_step — one mixed step: decode rows first, then one prefill
 * chunk from the budget that is left (host only).
 *   vLLM tutorial, section 5 (running requests first, one token per decode);
 *   SGLang article, mixed-chunk section (the chunk shrinks by the number of
 *   running decode requests).
 * decode_ctx_len[n_decode] (host): each decode row's context length L >= 1,
 * the token appended this step included (its cached prefix is L-1).
 * The prefill request has prefill_prefix_len tokens cached and
 * prefill_remaining still to compute.
 * Outputs (host), for the scheduled sequences in batch order (decode rows
 * first; rows that did not fit are left out, in order; the prefill sequence
 * last if it got any tokens):
 *   qo_indptr[n_decode + 2], prefix_len[n_decode + 1], kv_len[n_decode + 1],
 *   *n_seqs, *n_decode_out (decode rows scheduled), *extend_len_out.
 * Errors: CPE_ERR_INVALID_ARG for token_budget <= 0, n_decode < 0, L < 1,
 * negative prefill lengths, or null outputs.
 */
cpe_status cpe_plan_mixed_step(int32_t token_budget, int32_t n_decode,
                               const int32_t* decode_ctx_len, int32_t prefill_prefix_len,
                               int32_t prefill_remaining, int32_t* qo_indptr, int32_t* prefix_len,
                               int32_t* kv_len, int32_t* n_seqs, int32_t* n_decode_out,
                               int32_t* extend_len_out);

/*
 * cpe_plan_schedule — one scheduling step over running and waiting requests
 * under one token budget, laid out as the varlen batch cpe_mixed_step takes
 * (host only).
 *   vLLM tutorial, section 5 (the schedule() sketch and its worked example):
 *   running requests, in order, each take min(need, budget left); then waiting
 *   requests, in order, are admitted the same way while budget is left.  A
 *   prompt that does not fit is cut there: the granted count is its chunk.
 *   Memory allocation and preemption are the caller's and are not modelled.
 * running_computed[n_running], running_need[n_running] (host): tokens whose
 *   K/V are already cached, and tokens still to process (>= 1; 1 for a decode,
 *   the unfinished part of the prompt for a prefill continuation).
 * waiting_cached[n_waiting], waiting_prompt[n_waiting] (host): prefix-cache hit
 *   and prompt length; a waiting request needs prompt - cached >= 1 tokens.
 * Outputs (host, caller-owned; let n = n_running + n_waiting):
 *   granted[n]: tokens granted per request (running first, then waiting);
 *   *n_admitted: waiting requests granted any tokens (a prefix of the queue);
 *   the batch, one sequence per request granted tokens: those granted exactly
 *   one token first (decode rows; sequences 0 .. *n_decode-1, in scheduling
 *   order), then the others in scheduling order:
 *   qo_indptr[n + 1], prefix_len[n] (= the request's cached tokens),
 *   kv_len[n] (= prefix_len + granted), seq_request[n] (the request's index:
 *   r for running r, n_running + w for waiting w), *n_seqs, *n_decode.
 * Errors: CPE_ERR_INVALID_ARG for token_budget <= 0, negative counts, null
 * arrays, computed < 0, need < 1, cached < 0, prompt - cached < 1, or a
 * length that overflows int32.  Nothing is written on error.
 */
cpe_status cpe_plan_schedule(int32_t token_budget, int32_t n_running, const int32_t* running_computed,
                             const int32_t* running_need, int32_t n_waiting, const int32_t* waiting_cached,
                             const int32_t* waiting_prompt, int32_t* granted, int32_t* n_admitted,
                             int32_t* qo_indptr, int32_t* prefix_len, int32_t* kv_len, int32_t* seq_request,
                             int32_t* n_seqs, int32_t* n_decode);

/*
 * cpe_decide_decode_first — one step decision of the decode-first scheduler
 * with slack (host only).
 *   msmodeling chunked-prefill RFC, section 3.1.4 (DecodeFirstWithSlack):
 *   limit = floor(B * slack_percent / 100) (integer arithmetic; 115 for the
 *   RFC's 15 % slack), d_step = min(ready_decode, B),
 *   p_step = max(0, min(pending_prefill, floor((limit - d_step) / chunk_query_len))).
 * Errors: CPE_ERR_INVALID_ARG for B <= 0, chunk_query_len <= 0,
 * slack_percent < 100, negative counts or null outputs.
 */
cpe_status cpe_decide_decode_first(int32_t max_batched_tokens, int32_t ready_decode, int32_t pending_prefill,
                                   int32_t chunk_query_len, int32_t slack_percent, int32_t* p_step,
                                   int32_t* d_step);

/* Latency model of the time simulation: milliseconds of one prefill step of
 * `batch` requests running a chunk of query_len tokens at context seq_len
 * (is_decode 0), or of one decode step of `batch` requests whose mean context
 * is seq_len (is_decode 1, query_len 1). */
typedef double (*cpe_latency_fn)(void* ctx, int32_t is_decode, int32_t batch, int32_t query_len,
                                 int32_t seq_len);
/* Scheduler of the time simulation: writes the step's prefill and decode
 * request counts for the state; returns 0 on success. */
typedef int32_t (*cpe_decide_fn)(void* ctx, int32_t ready_decode, int32_t pending_prefill,
                                 int32_t chunk_query_len, int32_t max_batched_tokens, int32_t* p_step,
                                 int32_t* d_step);
/* How the scheduler combines a step's prefill and decode latencies. */
typedef double (*cpe_merge_fn)(void* ctx, double prefill_ms, double decode_ms);

typedef struct cpe_sim_result {
  double ttft_ms;             /* mean first-token time */
  double tpot_ms;             /* mean time per output token after the first (0 if output_len == 1) */
  double makespan_ms;         /* last request's finish time */
  double request_throughput;  /* requests per second over the makespan */
  double output_throughput;   /* output tokens per second over the makespan */
  int64_t steps;
} cpe_sim_result;

/*
 * cpe_simulate_requests — lightweight time simulation of n_requests identical
 * requests entering together (host only).
 *   msmodeling chunked-prefill RFC, section 3.1.5.  Each step asks the
 *   scheduler for (p_step, d_step) given the ready decode requests and the
 *   pending group: the requests at the chunk of the earliest request still in
 *   prefill (earlier requests run their chunks first).  The earliest requests
 *   of the group prefill and the earliest ready requests (by first-token
 *   time) decode one token; the step lasts merge(prefill latency, decode
 *   latency).  A request's last chunk produces its first token; it then needs
 *   max(output_len - 1, 0) decode steps, the first at context seq_len of the
 *   last chunk + 1.  The decode latency gets the decode batch's mean context,
 *   rounded up.  No barrier separates prefill from decode.
 * chunk_query_len[n_chunks], chunk_seq_len[n_chunks] (host): one request's
 *   chunk plan.  latency (required) with latency_ctx.  decide and merge
 *   (nullable, with sched_ctx): NULL decide means the decode-first scheduler
 *   with 15 % slack, NULL merge the larger of the two latencies.
 * first_token_ms[n_requests], finish_ms[n_requests] (host, nullable) receive
 * each request's times; *out the metrics.
 * Counts the scheduler returns beyond the pending group or the ready requests
 * are clamped to them.
 * Errors: CPE_ERR_INVALID_ARG for empty or non-positive lengths, a null
 * latency or out, a scheduler that fails or schedules nothing, or a negative
 * latency; CPE_ERR_CAPACITY if the simulation exceeds 2^31 steps.
 */
cpe_status cpe_simulate_requests(int32_t n_chunks, const int32_t* chunk_query_len, const int32_t* chunk_seq_len,
                                 int32_t n_requests, int32_t output_len, int32_t max_batched_tokens,
                                 cpe_latency_fn latency, void* latency_ctx, cpe_decide_fn decide,
                                 cpe_merge_fn merge, void* sched_ctx, double* first_token_ms, double* finish_ms,
                                 cpe_sim_result* out);

/*
 * cpe_kv_append — write the round's new K/V rows into the paged caches.
 *   SGLang article, implementation section (the request's req_to_token row
 *   keeps its page slots across chunks); mini-infer article, write_prefill_kv.
 * Row r of sequence s (qo_indptr[s] <= r < qo_indptr[s+1]) goes to position
 * pos = prefix_len[s] + r - qo_indptr[s], i.e. page page_table[s][pos /
 * page_size], slot pos % page_size.  A bitwise copy.
 * Device errors: a page id outside [0, num_pages) or pos / page_size >=
 * max_pages skips the row and records CPE_ERR_DEVICE_ARG.
 */
cpe_status cpe_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                         int64_t num_pages, const int32_t* page_table, int32_t max_pages,
                         const int32_t* qo_indptr, const int32_t* prefix_len, int32_t n_seqs,
                         int32_t total_q, int32_t h_kv, int32_t d, int32_t page_size,
                         cpe_dtype dtype, cpe_stream_t stream);

/*
 * cpe_workspace_size — bytes of device workspace the attention entry points
 * need for these sizes (the tile list and split-KV partial results).
 * max_kv_len bounds prefix_len[s] + E_s over all sequences.
 */
size_t cpe_workspace_size(int32_t n_seqs, int32_t total_q, int32_t h_q, int32_t h_kv, int32_t d,
                          int32_t max_kv_len);

/*
 * cpe_extend_attention — the extend output for every query row (all rows of
 * all sequences): out[r, h] = sum_{j <= P_s + i} softmax_j(q . k_j * sm_scale) v_j.
 *   SGLang article, equation for o_i; Stage 1 (prefix rectangle, no mask) and
 *   Stage 2 (causal triangle in the chunk) run as separate tile classes whose
 *   partials are merged by their (m, l) statistics.
 * The keys of the chunk itself (positions [P_s, P_s + E_s)) must already be
 * in the cache (cpe_kv_append first).
 * sm_scale: softmax scale (pass 1/sqrt(d) for the pages' definition).
 * max_kv_len: an upper bound on prefix_len[s] + E_s; sequences above it are
 * not computed and CPE_ERR_DEVICE_ARG is recorded.
 * lse: nullable.  workspace: at least cpe_workspace_size(...) bytes, 256-byte
 * aligned; its contents need not be initialised and are clobbered.  A
 * workspace serves one stream at a time.  Consecutive calls on one stream
 * that alternate between two workspaces overlap more: a call's tile list is
 * built while the previous call finishes.  With one workspace, the tile list
 * is written only after the previous call is done.  Results are the same
 * either way.
 * Errors: CPE_ERR_INVALID_ARG / CPE_ERR_UNSUPPORTED / CPE_ERR_CAPACITY before
 * any launch; CPE_ERR_CUDA if a launch fails.
 */
cpe_status cpe_extend_attention(const void* q, const void* k_cache, const void* v_cache,
                                int64_t num_pages, const int32_t* page_table, int32_t max_pages,
                                const int32_t* qo_indptr, const int32_t* prefix_len,
                                int32_t n_seqs, int32_t total_q, int32_t max_kv_len, int32_t h_q,
                                int32_t h_kv, int32_t d, int32_t page_size, float sm_scale,
                                cpe_dtype dtype, void* out, float* lse, void* workspace,
                                size_t workspace_bytes, cpe_stream_t stream);

/*
 * cpe_mixed_step — one mixed forward step of attention: n_decode decode rows
 * (sequences 0 .. n_decode-1, one query each) and the remaining sequences'
 * prefill chunks, under one token budget, as cpe_plan_mixed_step lays them out.
 *   SGLang article, mixed-chunk section (ForwardMode.MIXED); vLLM tutorial,
 *   section 4 ({request_id: num_tokens} in one forward).
 * Appends k_new / v_new for every row (as cpe_kv_append), then computes the
 * decode rows with the split-KV path (HBM-bound, one CTA per (row, KV head,
 * split), merged by LSE) and the prefill chunks with the extend path.
 * Same arguments as cpe_extend_attention plus k_new, v_new, the writable
 * caches and n_decode (0 <= n_decode <= n_seqs).  A decode sequence whose
 * query length is not 1 records CPE_ERR_DEVICE_ARG and is not computed.
 */
cpe_status cpe_mixed_step(const void* q, const void* k_new, const void* v_new, void* k_cache,
                          void* v_cache, int64_t num_pages, const int32_t* page_table,
                          int32_t max_pages, const int32_t* qo_indptr, const int32_t* prefix_len,
                          int32_t n_seqs, int32_t n_decode, int32_t total_q, int32_t max_kv_len,
                          int32_t h_q, int32_t h_kv, int32_t d, int32_t page_size, float sm_scale,
                          cpe_dtype dtype, void* out, float* lse, void* workspace,
                          size_t workspace_bytes, cpe_stream_t stream);

/*
 * cpe_decode_attention — the decode-row path on its own: every sequence has
 * one query row (qo_indptr[s] = s).  Split-KV over each row's context, merged
 * by LSE.  Arguments as cpe_extend_attention.
 */
cpe_status cpe_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                                int64_t num_pages, const int32_t* page_table, int32_t max_pages,
                                const int32_t* prefix_len, int32_t n_seqs, int32_t max_kv_len,
                                int32_t h_q, int32_t h_kv, int32_t d, int32_t page_size,
                                float sm_scale, cpe_dtype dtype, void* out, float* lse,
                                void* workspace, size_t workspace_bytes, cpe_stream_t stream);

/*
 * cpe_decode_attention_noalloc — the decode-row path of cpe_decode_attention
 * for callers that cannot allocate device memory.  The pages describe no such
 * entry point; it has no counterpart there.
 *
 * Who needs it: a caller that may not call cudaMalloc or any allocator of its
 * own — for instance a plugin inside a host program that owns every byte of
 * device memory through its own pool, or a serving loop that must not enter
 * an allocator on its hot path (cudaMalloc can synchronise the device and can
 * fail when memory is fragmented).  cpe_decode_attention needs a caller-made
 * workspace for its split partials; this entry point keeps them instead in a
 * fixed array of CPE_DECODE_NOALLOC_SCRATCH_BYTES (8 MiB) of device memory
 * that the library declares statically, so the call itself allocates nothing
 * (no cudaMalloc, no cudaFree, no allocating library routine).
 *
 * Arguments, layouts and results are those of cpe_decode_attention, without
 * the workspace.  Limits and behaviour:
 *  - The scratch needed is n_seqs * h_q * ceil(max_kv_len / 2048) * (d + 2)
 *    * 4 bytes (each part rounded up to 256 bytes).  Above 8 MiB the call
 *    returns CPE_ERR_CAPACITY before any launch; split the batch or use
 *    cpe_decode_attention.  Only bf16 is taken (CPE_ERR_UNSUPPORTED).
 *  - The array exists on every GPU that loads the library and stays there
 *    until the process exits.  CUDA loads a library's device code lazily by
 *    default, so the array is placed on a device when the library's first
 *    kernel there is loaded, which may be this entry point's first call;
 *    later calls take no device memory.
 *  - The first call on a device, with that device current, looks up the
 *    array's device address (cudaGetSymbolAddress) and keeps it; make that
 *    first call before any stream capture.  A cudaDeviceReset of that device
 *    later in the process voids the kept address: call this entry point on a
 *    device only while the context it first ran in is alive.
 *  - Every call uses the same array, which keeps the last call's contents.
 *    Nothing in it has to start at zero: each call writes every partial it
 *    reads.  Calls whose kernels overlap on the GPU (different streams, or
 *    different host threads, on one device) race on the array: order them on
 *    one stream or synchronise between them.
 */
cpe_status cpe_decode_attention_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                        int64_t num_pages, const int32_t* page_table,
                                        int32_t max_pages, const int32_t* prefix_len, int32_t n_seqs,
                                        int32_t max_kv_len, int32_t h_q, int32_t h_kv, int32_t d,
                                        int32_t page_size, float sm_scale, cpe_dtype dtype, void* out,
                                        float* lse, cpe_stream_t stream);

#define CPE_DECODE_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)

/*
 * cpe_get_device_status — synchronise `stream`, then read and clear the
 * device status word of the current device.  Returns CPE_OK, the first device
 * error recorded since the last call (CPE_ERR_TIMEOUT, CPE_ERR_DEVICE_ARG), or
 * CPE_ERR_CUDA if the synchronisation itself failed.  *detail (host,
 * nullable) receives a code naming the wait or check that failed.
 */
cpe_status cpe_get_device_status(cpe_stream_t stream, int32_t* detail);

/*
 * cpe_set_wait_limit_ns — time after which a device pipeline wait gives up,
 * records CPE_ERR_TIMEOUT and lets its kernel return (default 4e9 ns).  A
 * test hook: 0 makes every wait that is not already satisfied give up at
 * once, so the timeout path can be checked without a stalled kernel.
 * Applies to launches made after the call; returns the previous value.
 */
int64_t cpe_set_wait_limit_ns(int64_t ns);

/* Static description of a status code. */
const char* cpe_status_string(cpe_status status);

/* Message of the last host-side error on the calling thread ("" if none). */
const char* cpe_last_error(void);

/* Number of CUDA kernels this library has launched in this process. */
int64_t cpe_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* CPE_H */
