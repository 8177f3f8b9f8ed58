"""Decode-first scheduling with slack and the lightweight time simulation of a
group of concurrent requests, written out plainly from the pages.

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
benchmark's CPU-baseline leg may use this module; the product path may not.

Source: msmodeling chunked-prefill RFC (gitcode.com/Ascend/msmodeling,
docs/RFC/rfc_chunked_prefill_support_zh.md), section 3.1.4 (mixed-step token
budget with 15 % slack; the Scheduler interface of StepDecision /
SchedulerState and its default DecodeFirstWithSlack) and section 3.1.5 (the
lightweight time simulation: pending prefill, ready decode and finished
requests; TTFT, TPOT, makespan and throughputs), with the unit-test vectors of
section 4.

Readings where the RFC is silent or loose:
- The slack limit floor(B * 1.15) is taken in integers as B * 115 // 100 (the
  "15 % slack" it describes); the double expression differs from it for some B
  (B = 100 gives 114 instead of 115), not for the RFC's B = 4000.
- "The next pending prefill chunk" is the chunk of the earliest request still
  in prefill, and the pending group is every pending request at that chunk
  index.  Requests are picked earliest first, so earlier requests run their
  chunks first and start decoding while later ones are still in prefill.
- When more requests are ready to decode than the step takes, the earliest
  ones (by first-token time, then request order) decode.
- The latency model is called as latency(is_decode, batch, query_len, seq_len)
  in milliseconds; a prefill call gets the chunk's query and sequence length,
  a decode call query length 1 and the decode batch's mean context length
  (input plus tokens produced so far), rounded up.
- A request's first token is produced by its last prefill chunk; it then needs
  R = max(O - 1, 0) decode steps.
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class StepDecision:
    p_step: int
    d_step: int


@dataclass(frozen=True)
class SchedulerState:
    ready_decode: int
    pending_prefill: int
    chunk_query_len: int
    max_batched_tokens: int


def slack_limit(max_batched_tokens: int, slack_percent: int = 115) -> int:
    return max_batched_tokens * slack_percent // 100


class DecodeFirstWithSlack:
    """Decode requests first, one token each, up to the budget; then as many
    requests of the pending chunk as fit under the slack limit."""
    slack_percent = 115

    def decide(self, st: SchedulerState) -> StepDecision:
        limit = slack_limit(st.max_batched_tokens, self.slack_percent)
        d = min(st.ready_decode, st.max_batched_tokens)
        p = max(0, min(st.pending_prefill, (limit - d) // st.chunk_query_len))
        return StepDecision(p, d)

    def step_latency(self, prefill_ms: float, decode_ms: float) -> float:
        return max(prefill_ms, decode_ms)  # prefill and decode run side by side in one step


def simulate(chunks: list[tuple[int, int]], n_requests: int, output_len: int, max_batched_tokens: int,
             latency, scheduler=None) -> dict:
    """Time simulation of n_requests identical requests entering together.

    chunks: (query_len, seq_len) of each prefill chunk of one request, in order
    (its chunk plan); the last seq_len is the prompt's full context.
    latency(is_decode, batch, query_len, seq_len) -> ms.
    """
    if scheduler is None:
        scheduler = DecodeFirstWithSlack()
    if not chunks or n_requests < 1 or output_len < 1 or max_batched_tokens < 1:
        raise ValueError("need chunks, n_requests >= 1, output_len >= 1, max_batched_tokens >= 1")
    K = len(chunks)
    R = max(output_len - 1, 0)
    ctx0 = chunks[-1][1]
    nxt = [0] * n_requests           # next prefill chunk (K: prefill done)
    left = [0] * n_requests          # decode tokens still to produce
    ctx = [0] * n_requests           # context of the next decode step
    first = [None] * n_requests
    finish = [None] * n_requests
    t = 0.0
    steps = 0
    done = 0
    while done < n_requests:
        pending = [r for r in range(n_requests) if nxt[r] < K]
        ready = sorted((r for r in range(n_requests) if nxt[r] == K and left[r] > 0),
                       key=lambda r: (first[r], r))
        if pending:
            c = nxt[pending[0]]
            group = [r for r in pending if nxt[r] == c]
            st = SchedulerState(len(ready), len(group), chunks[c][0], max_batched_tokens)
        else:
            c, group = None, []
            st = SchedulerState(len(ready), 0, max_batched_tokens, max_batched_tokens)
        dec = scheduler.decide(st)
        P = min(dec.p_step, len(group))
        D = min(dec.d_step, len(ready))
        if P == 0 and D == 0:
            raise RuntimeError("the scheduler chose an empty step")
        pl = latency(False, P, chunks[c][0], chunks[c][1]) if P > 0 else 0.0
        dsel = ready[:D]
        dl = latency(True, D, 1, -(-sum(ctx[r] for r in dsel) // D)) if D > 0 else 0.0
        t += scheduler.step_latency(pl, dl)
        steps += 1
        for r in group[:P]:
            nxt[r] += 1
            if nxt[r] == K:
                first[r] = t
                if R > 0:
                    left[r] = R
                    ctx[r] = ctx0 + 1
                else:
                    finish[r] = t
                    done += 1
        for r in dsel:
            left[r] -= 1
            ctx[r] += 1
            if left[r] == 0:
                finish[r] = t
                done += 1
    makespan = max(finish)
    return {"ttft": sum(first) / n_requests,
            "tpot": 0.0 if R == 0 else sum((finish[r] - first[r]) / R for r in range(n_requests)) / n_requests,
            "makespan": makespan,
            "request_throughput": 1000.0 * n_requests / makespan,
            "output_throughput": 1000.0 * n_requests * output_len / makespan,
            "steps": steps, "first_token_time": first, "finish_time": finish}
