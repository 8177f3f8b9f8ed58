"""Pins for the oracle's decode-first scheduler and time simulation: the
RFC's printed decision vector, closed forms of small schedules worked by hand,
an injected scheduler, and invariants."""
import json
import os
import random

import pytest

from oracle import sched_sim as S

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "sched_vectors.json")))


@pytest.mark.parametrize("case", GOLDEN["decide"], ids=lambda c: str(c["max_batched_tokens"]))
def test_decide_matches_pages(case):
    d = S.DecodeFirstWithSlack().decide(S.SchedulerState(case["ready_decode"], case["pending_prefill"],
                                                         case["chunk_query_len"], case["max_batched_tokens"]))
    assert (d.p_step, d.d_step) == (case["p_step"], case["d_step"])


def test_slack_limit_matches_pages():
    for case in GOLDEN["slack_limit"]:
        assert S.slack_limit(case["max_batched_tokens"]) == case["limit"]


def test_decide_beyond_slack_shrinks_prefill():
    """Over floor(B * 1.15) the prefill concurrency drops, to zero if need be
    (the RFC's second DecodeFirstWithSlack test)."""
    sch = S.DecodeFirstWithSlack()
    assert sch.decide(S.SchedulerState(601, 1, 4000, 4000)) == S.StepDecision(0, 601)  # 4601 > 4600
    assert sch.decide(S.SchedulerState(600, 1, 4000, 4000)) == S.StepDecision(1, 600)  # 4600 fits
    assert sch.decide(S.SchedulerState(512, 8, 1000, 4000)) == S.StepDecision(4, 512)  # (4600-512)//1000
    assert sch.decide(S.SchedulerState(5000, 3, 100, 4000)) == S.StepDecision(3, 4000)  # (4600-4000)//100 = 6 > 3 pending
    assert sch.decide(S.SchedulerState(0, 9, 4000, 4000)) == S.StepDecision(1, 0)     # 4600 // 4000


def test_step_latency_is_the_larger():
    assert S.DecodeFirstWithSlack().step_latency(3.0, 7.5) == 7.5
    assert S.DecodeFirstWithSlack().step_latency(9.0, 2.0) == 9.0


def _const(lp, ld):
    return lambda is_decode, b, q, s: ld if is_decode else lp


def test_single_request_prefill_only():
    """One request, O = 1: TTFT is the sum of its chunks' latencies, no TPOT."""
    chunks = [(4096, 4096), (4096, 8192), (1808, 10000)]
    lat = lambda is_decode, b, q, s: 0.5 + q * 1e-3 + s * 1e-4
    out = S.simulate(chunks, 1, 1, 4096, lat)
    want = sum(0.5 + q * 1e-3 + s * 1e-4 for q, s in chunks)
    assert out["ttft"] == pytest.approx(want, rel=1e-15) and out["makespan"] == out["ttft"]
    assert out["tpot"] == 0.0 and out["steps"] == 3


def test_single_request_decode_steps():
    """One request, one chunk, O = 5: prefill, then four decode steps."""
    out = S.simulate([(512, 512)], 1, 5, 4096, _const(7.0, 2.0))
    assert out["ttft"] == 7.0 and out["makespan"] == 15.0 and out["tpot"] == 2.0
    assert out["output_throughput"] == pytest.approx(1000.0 * 5 / 15.0)


def test_two_requests_overlap_without_a_barrier():
    """B = chunk = 4000: one prefill per step.  Request 0 decodes in the step
    where request 1 prefills (max of the two latencies), so there is no global
    barrier between prefill and decode."""
    lp, ld = 10.0, 3.0
    out = S.simulate([(4000, 4000)], 2, 2, 4000, _const(lp, ld))
    assert out["first_token_time"] == [lp, lp + max(lp, ld)]
    assert out["finish_time"] == [lp + max(lp, ld), lp + max(lp, ld) + ld]
    assert out["ttft"] == pytest.approx((2 * lp + max(lp, ld)) / 2)
    assert out["tpot"] == pytest.approx((max(lp, ld) + ld) / 2)
    assert out["makespan"] == lp + max(lp, ld) + ld


def test_slack_admits_prefill_beside_decodes():
    """With 512 decoding requests a full 4000-token chunk still runs in the same
    step (the RFC's 4000 + 512 <= 4600 example)."""
    calls = []

    def lat(is_decode, b, q, s):
        calls.append((is_decode, b, q))
        return 1.0
    S.simulate([(4000, 4000)], 513, 3, 4000, lat)
    # step 1 prefills request 0 alone; step 2 decodes it beside request 1's prefill
    assert calls[0] == (False, 1, 4000) and (True, 1, 1) in calls[1:3] and (False, 1, 4000) in calls[1:3]


def test_injected_scheduler_drives_the_loop():
    """A prefill-first scheduler with summed latencies changes the timeline
    without touching the simulation loop (the RFC's pluggability test)."""
    class PrefillFirst:
        def decide(self, st):
            if st.pending_prefill:
                return S.StepDecision(st.pending_prefill, 0)
            return S.StepDecision(0, min(st.ready_decode, st.max_batched_tokens))

        def step_latency(self, p, d):
            return p + d
    out = S.simulate([(100, 100), (100, 200)], 3, 3, 4096, _const(5.0, 1.0), PrefillFirst())
    # both chunks for all three requests first (10 ms), then two decode steps
    assert out["first_token_time"] == [10.0] * 3 and out["finish_time"] == [12.0] * 3 and out["steps"] == 4


def test_decode_latency_sees_the_growing_context():
    seen = []

    def lat(is_decode, b, q, s):
        if is_decode:
            seen.append(s)
        return 1.0
    S.simulate([(1000, 1000)], 1, 4, 4096, lat)
    assert seen == [1001, 1002, 1003]  # the first token joins the context at the first decode step


def test_invariants_random():
    rng = random.Random(5)
    for _ in range(60):
        B = rng.choice([256, 512, 2048, 4000])
        n_in = rng.randint(1, 9000)
        chunks, done = [], 0
        while done < n_in:
            q = min(B, n_in - done)
            done += q
            chunks.append((q, done))
        N, O = rng.randint(1, 40), rng.randint(1, 30)
        lat = lambda d, b, q, s: (0.2 + 1e-4 * b * s) if d else (0.5 + 1e-6 * b * q * s)
        out = S.simulate(chunks, N, O, B, lat)
        f, e = out["first_token_time"], out["finish_time"]
        assert all(x is not None for x in f + e) and all(b >= a for a, b in zip(f, e))
        assert out["makespan"] == max(e) and out["ttft"] <= out["makespan"]
        # no step is empty and at least K prefill steps ran for the earliest request
        assert out["steps"] >= len(chunks) + max(O - 1, 0)


def test_argument_errors():
    with pytest.raises(ValueError):
        S.simulate([], 1, 1, 10, _const(1, 1))
    with pytest.raises(ValueError):
        S.simulate([(5, 5)], 0, 1, 10, _const(1, 1))
