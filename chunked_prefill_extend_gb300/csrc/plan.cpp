// Host planners of libcpe: the chunk plan of one request, token-budget
// truncation, and the mixed-step batch layout.
//
// msmodeling RFC "Chunked Prefill modelling support": section 2.2 (cached
// prefix = floor(input_length * hit_rate), effective length = the rest; decode
// keeps the full input length) and section 3.1.3 (one chunk per
// min(chunk_size, remaining) tokens).  SGLang chunked-prefill article: the
// round cursor [prefix_len, extend_end) and, in its implementation section,
// page alignment of a new request's first cut only.  vLLM token-budget
// tutorial, section 5: min(need, remaining budget) per request, decode rows
// first at one token each; SGLang article, mixed-chunk section: the chunk
// shrinks by the number of running decode requests.
#include <climits>
#include <cmath>
#include <cstdint>
#include <string>

#include "cpe.h"

namespace cpe {
void set_last_error(const std::string& msg);
}

extern "C" cpe_status cpe_plan_chunks(int64_t input_len, double prefix_hit_rate, int32_t chunk_size,
                                      int32_t align_to, cpe_chunk* out, int32_t cap, int32_t* n_out,
                                      int64_t* cached_out, int64_t* effective_out) {
  if (n_out == nullptr || (cap > 0 && out == nullptr) || cap < 0) {
    cpe::set_last_error("cpe_plan_chunks: null output or negative capacity");
    return CPE_ERR_INVALID_ARG;
  }
  if (chunk_size <= 0) {
    cpe::set_last_error("cpe_plan_chunks: chunk_size (max_batched_tokens) must be > 0");
    return CPE_ERR_INVALID_ARG;
  }
  if (input_len <= 0 || input_len > INT32_MAX || !(prefix_hit_rate >= 0.0 && prefix_hit_rate <= 1.0) ||
      align_to < 0) {
    cpe::set_last_error("cpe_plan_chunks: input_len must be in [1, INT32_MAX], hit rate in [0, 1], align_to >= 0");
    return CPE_ERR_INVALID_ARG;
  }
  const int64_t cached = static_cast<int64_t>(std::floor(static_cast<double>(input_len) * prefix_hit_rate));
  const int64_t effective = input_len - cached;
  if (cached_out) *cached_out = cached;
  if (effective_out) *effective_out = effective;
  if (effective < 1) {
    cpe::set_last_error("cpe_plan_chunks: effective_input_length must be >= 1");
    return CPE_ERR_INVALID_ARG;
  }
  int32_t n = 0;
  int64_t consumed = 0;
  while (consumed < effective) {
    const int64_t remaining = effective - consumed;
    int64_t take = remaining < chunk_size ? remaining : chunk_size;
    if (align_to > 0 && n == 0 && take < remaining) {
      const int64_t end = ((cached + take) / align_to) * align_to;
      if (end > cached) take = end - cached;
    }
    if (n < cap) {
      cpe_chunk& c = out[n];
      c.index = n;
      c.prefix_len = static_cast<int32_t>(cached + consumed);
      c.query_len = static_cast<int32_t>(take);
      c.seq_len = static_cast<int32_t>(cached + consumed + take);
      c.model_seq_len = static_cast<int32_t>(consumed + take);
    }
    consumed += take;
    ++n;
  }
  *n_out = n;
  if (n > cap) {
    cpe::set_last_error("cpe_plan_chunks: output capacity below the chunk count");
    return CPE_ERR_CAPACITY;
  }
  return CPE_OK;
}

extern "C" cpe_status cpe_plan_budget(int32_t token_budget, int32_t n_req, const int32_t* need,
                                      int32_t* granted, int32_t* used) {
  if (token_budget <= 0 || n_req < 0 || (n_req > 0 && (need == nullptr || granted == nullptr))) {
    cpe::set_last_error("cpe_plan_budget: token_budget must be > 0 and arrays non-null");
    return CPE_ERR_INVALID_ARG;
  }
  for (int32_t k = 0; k < n_req; ++k)
    if (need[k] < 0) {
      cpe::set_last_error("cpe_plan_budget: negative need");
      return CPE_ERR_INVALID_ARG;
    }
  int32_t left = token_budget;
  for (int32_t k = 0; k < n_req; ++k) {
    const int32_t take = left > 0 ? (need[k] < left ? need[k] : left) : 0;
    granted[k] = take;
    left -= take;
  }
  if (used) *used = token_budget - left;
  return CPE_OK;
}

extern "C" cpe_status cpe_plan_mixed_step(int32_t token_budget, int32_t n_decode,
                                          const int32_t* decode_ctx_len, int32_t prefill_prefix_len,
                                          int32_t prefill_remaining, int32_t* qo_indptr,
                                          int32_t* prefix_len, int32_t* kv_len, int32_t* n_seqs,
                                          int32_t* n_decode_out, int32_t* extend_len_out) {
  if (token_budget <= 0 || n_decode < 0 || (n_decode > 0 && decode_ctx_len == nullptr) ||
      prefill_prefix_len < 0 || prefill_remaining < 0 || !qo_indptr || !prefix_len || !kv_len ||
      !n_seqs || !n_decode_out || !extend_len_out) {
    cpe::set_last_error("cpe_plan_mixed_step: bad arguments");
    return CPE_ERR_INVALID_ARG;
  }
  for (int32_t k = 0; k < n_decode; ++k)
    if (decode_ctx_len[k] < 1) {
      cpe::set_last_error("cpe_plan_mixed_step: a decode context length is < 1");
      return CPE_ERR_INVALID_ARG;
    }
  if (static_cast<int64_t>(prefill_prefix_len) + prefill_remaining > INT32_MAX) {
    cpe::set_last_error("cpe_plan_mixed_step: prefill length overflows int32");
    return CPE_ERR_INVALID_ARG;
  }
  int32_t left = token_budget;
  int32_t ns = 0;
  qo_indptr[0] = 0;
  for (int32_t k = 0; k < n_decode; ++k) {
    if (left <= 0) break;  // decode rows that do not fit sit this step out
    prefix_len[ns] = decode_ctx_len[k] - 1;
    kv_len[ns] = decode_ctx_len[k];
    qo_indptr[ns + 1] = qo_indptr[ns] + 1;
    ++ns;
    --left;
  }
  *n_decode_out = ns;
  const int32_t extend = left > 0 ? (prefill_remaining < left ? prefill_remaining : left) : 0;
  if (extend > 0) {
    prefix_len[ns] = prefill_prefix_len;
    kv_len[ns] = prefill_prefix_len + extend;
    qo_indptr[ns + 1] = qo_indptr[ns] + extend;
    ++ns;
  }
  *extend_len_out = extend;
  *n_seqs = ns;
  return CPE_OK;
}

extern "C" cpe_status cpe_plan_schedule(int32_t token_budget, int32_t n_running, const int32_t* running_computed,
                                        const int32_t* running_need, int32_t n_waiting,
                                        const int32_t* waiting_cached, const int32_t* waiting_prompt,
                                        int32_t* granted, int32_t* n_admitted, int32_t* qo_indptr,
                                        int32_t* prefix_len, int32_t* kv_len, int32_t* seq_request,
                                        int32_t* n_seqs, int32_t* n_decode) {
  const char* fn = "cpe_plan_schedule";
  auto bad = [&](const char* why) {
    cpe::set_last_error(std::string(fn) + ": " + why);
    return CPE_ERR_INVALID_ARG;
  };
  if (token_budget <= 0) return bad("token_budget must be > 0");
  if (n_running < 0 || n_waiting < 0 || static_cast<int64_t>(n_running) + n_waiting > INT32_MAX - 1)
    return bad("request counts must be >= 0");
  if ((n_running > 0 && (!running_computed || !running_need)) ||
      (n_waiting > 0 && (!waiting_cached || !waiting_prompt)))
    return bad("null request arrays");
  const int32_t n = n_running + n_waiting;
  if (!n_admitted || !qo_indptr || !n_seqs || !n_decode ||
      (n > 0 && (!granted || !prefix_len || !kv_len || !seq_request)))
    return bad("null output arrays");
  for (int32_t r = 0; r < n_running; ++r) {
    if (running_computed[r] < 0 || running_need[r] < 1) return bad("a running request needs computed >= 0, need >= 1");
    if (static_cast<int64_t>(running_computed[r]) + running_need[r] > INT32_MAX) return bad("length overflows int32");
  }
  for (int32_t w = 0; w < n_waiting; ++w)
    if (waiting_cached[w] < 0 || static_cast<int64_t>(waiting_prompt[w]) - waiting_cached[w] < 1)
      return bad("a waiting request needs cached >= 0 and prompt - cached >= 1");
  // grants: running requests in order, then waiting ones while budget is left
  int32_t left = token_budget;
  int32_t admitted = 0;
  for (int32_t k = 0; k < n; ++k) {
    const int32_t need = k < n_running ? running_need[k] : waiting_prompt[k - n_running] - waiting_cached[k - n_running];
    const int32_t take = need < left ? need : left;
    granted[k] = take;
    left -= take;
    if (k >= n_running && take > 0) ++admitted;
  }
  // the batch: one-token sequences first, then the chunks, each in scheduling order
  int32_t ns = 0, nd = 0;
  qo_indptr[0] = 0;
  for (int pass = 0; pass < 2; ++pass)
    for (int32_t k = 0; k < n; ++k) {
      if (granted[k] == 0 || (pass == 0) != (granted[k] == 1)) continue;
      const int32_t base = k < n_running ? running_computed[k] : waiting_cached[k - n_running];
      prefix_len[ns] = base;
      kv_len[ns] = base + granted[k];
      seq_request[ns] = k;
      qo_indptr[ns + 1] = qo_indptr[ns] + granted[k];
      ++ns;
      if (pass == 0) ++nd;
    }
  *n_admitted = admitted;
  *n_seqs = ns;
  *n_decode = nd;
  return CPE_OK;
}
