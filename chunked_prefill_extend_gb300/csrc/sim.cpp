// Host-side scheduling policy and time simulation of concurrent requests.
//
// msmodeling chunked-prefill RFC (gitcode.com/Ascend/msmodeling,
// docs/RFC/rfc_chunked_prefill_support_zh.md), sections 3.1.4 and 3.1.5:
// the decode-first scheduler with 15 % slack on the mixed-step token budget,
// and the lightweight simulation that advances request groups through their
// prefill chunks and decode steps to TTFT, TPOT, makespan and throughput.  The
// latency of a step comes from a caller-supplied model (the kernels' measured
// per-shape latencies, for instance).
#include <climits>
#include <string>
#include <vector>

#include "cpe.h"

namespace cpe {
void set_last_error(const std::string& msg);
}

namespace {

int32_t decide_default(int32_t B, int32_t ready, int32_t pending, int32_t qlen, int32_t slack_percent, int32_t* p,
                       int32_t* d) {
  const int64_t limit = static_cast<int64_t>(B) * slack_percent / 100;
  const int32_t dd = ready < B ? ready : B;
  const int64_t fit = (limit - dd) / qlen;
  const int64_t pp = fit < pending ? fit : pending;
  *d = dd;
  *p = static_cast<int32_t>(pp > 0 ? pp : 0);
  return 0;
}

cpe_status bad(const char* fn, const char* why) {
  cpe::set_last_error(std::string(fn) + ": " + why);
  return CPE_ERR_INVALID_ARG;
}

}  // namespace

extern "C" cpe_status cpe_decide_decode_first(int32_t max_batched_tokens, int32_t ready_decode,
                                              int32_t pending_prefill, int32_t chunk_query_len,
                                              int32_t slack_percent, int32_t* p_step, int32_t* d_step) {
  const char* fn = "cpe_decide_decode_first";
  if (max_batched_tokens <= 0 || chunk_query_len <= 0 || slack_percent < 100 || ready_decode < 0 ||
      pending_prefill < 0 || !p_step || !d_step)
    return bad(fn, "need B > 0, chunk_query_len > 0, slack_percent >= 100, counts >= 0 and outputs");
  decide_default(max_batched_tokens, ready_decode, pending_prefill, chunk_query_len, slack_percent, p_step, d_step);
  return CPE_OK;
}

extern "C" cpe_status cpe_simulate_requests(int32_t n_chunks, const int32_t* chunk_query_len,
                                            const int32_t* chunk_seq_len, int32_t n_requests, int32_t output_len,
                                            int32_t max_batched_tokens, cpe_latency_fn latency, void* latency_ctx,
                                            cpe_decide_fn decide, cpe_merge_fn merge, void* sched_ctx,
                                            double* first_token_ms, double* finish_ms, cpe_sim_result* out) {
  const char* fn = "cpe_simulate_requests";
  if (n_chunks < 1 || !chunk_query_len || !chunk_seq_len || n_requests < 1 || output_len < 1 ||
      max_batched_tokens < 1 || !latency || !out)
    return bad(fn, "need chunks, n_requests >= 1, output_len >= 1, max_batched_tokens >= 1, latency and out");
  for (int32_t c = 0; c < n_chunks; ++c)
    if (chunk_query_len[c] < 1 || chunk_seq_len[c] < chunk_query_len[c]) return bad(fn, "bad chunk lengths");
  const int32_t K = n_chunks;
  const int32_t R = output_len > 1 ? output_len - 1 : 0;
  const int64_t ctx0 = chunk_seq_len[K - 1];
  std::vector<int32_t> nxt(n_requests, 0), left(n_requests, 0);
  std::vector<int64_t> ctx(n_requests, 0);
  std::vector<double> first(n_requests, 0.0), finish(n_requests, 0.0);
  std::vector<int32_t> ready;    // requests with decode tokens left, earliest first token first
  std::vector<int32_t> group;
  double t = 0.0;
  int64_t steps = 0;
  int32_t done = 0;
  int32_t lead = 0;              // earliest request still in prefill (requests finish prefill in order)
  while (done < n_requests) {
    while (lead < n_requests && nxt[lead] >= K) ++lead;
    group.clear();
    int32_t c = -1;
    if (lead < n_requests) {
      c = nxt[lead];
      for (int32_t r = lead; r < n_requests; ++r)
        if (nxt[r] == c) group.push_back(r);
    }
    const int32_t n_ready = static_cast<int32_t>(ready.size());
    const int32_t qlen = c >= 0 ? chunk_query_len[c] : max_batched_tokens;
    int32_t P = 0, D = 0;
    const int32_t rc = decide ? decide(sched_ctx, n_ready, static_cast<int32_t>(group.size()), qlen,
                                       max_batched_tokens, &P, &D)
                              : decide_default(max_batched_tokens, n_ready, static_cast<int32_t>(group.size()), qlen,
                                               115, &P, &D);
    if (rc != 0) return bad(fn, "the scheduler failed");
    if (P > static_cast<int32_t>(group.size())) P = static_cast<int32_t>(group.size());
    if (D > n_ready) D = n_ready;
    if (P < 0) P = 0;
    if (D < 0) D = 0;
    if (P == 0 && D == 0) return bad(fn, "the scheduler chose an empty step");
    const double pl = P > 0 ? latency(latency_ctx, 0, P, chunk_query_len[c], chunk_seq_len[c]) : 0.0;
    double dl = 0.0;
    if (D > 0) {
      int64_t sum = 0;
      for (int32_t k = 0; k < D; ++k) sum += ctx[ready[k]];
      const int64_t mean = (sum + D - 1) / D;
      dl = latency(latency_ctx, 1, D, 1, static_cast<int32_t>(mean < INT32_MAX ? mean : INT32_MAX));
    }
    if (!(pl >= 0.0) || !(dl >= 0.0)) return bad(fn, "the latency model returned a negative or NaN latency");
    t += merge ? merge(sched_ctx, pl, dl) : (pl > dl ? pl : dl);
    if (++steps > INT32_MAX) {
      cpe::set_last_error(std::string(fn) + ": more than 2^31 steps");
      return CPE_ERR_CAPACITY;
    }
    // decode first (over the requests ready before this step), then prefill
    std::vector<int32_t> still;
    still.reserve(ready.size());
    for (int32_t k = 0; k < n_ready; ++k) {
      const int32_t r = ready[k];
      if (k < D) {
        --left[r];
        ++ctx[r];
        if (left[r] == 0) {
          finish[r] = t;
          ++done;
          continue;
        }
      }
      still.push_back(r);
    }
    ready.swap(still);
    for (int32_t k = 0; k < P; ++k) {
      const int32_t r = group[k];
      if (++nxt[r] == K) {
        first[r] = t;
        if (R > 0) {
          left[r] = R;
          ctx[r] = ctx0 + 1;
          ready.push_back(r);
        } else {
          finish[r] = t;
          ++done;
        }
      }
    }
  }
  double sf = 0.0, st = 0.0, mk = 0.0;
  for (int32_t r = 0; r < n_requests; ++r) {
    sf += first[r];
    if (R > 0) st += (finish[r] - first[r]) / R;
    if (finish[r] > mk) mk = finish[r];
  }
  out->ttft_ms = sf / n_requests;
  out->tpot_ms = R > 0 ? st / n_requests : 0.0;
  out->makespan_ms = mk;
  out->request_throughput = 1000.0 * n_requests / mk;
  out->output_throughput = 1000.0 * n_requests * output_len / mk;
  out->steps = steps;
  if (first_token_ms)
    for (int32_t r = 0; r < n_requests; ++r) first_token_ms[r] = first[r];
  if (finish_ms)
    for (int32_t r = 0; r < n_requests; ++r) finish_ms[r] = finish[r];
  return CPE_OK;
}
