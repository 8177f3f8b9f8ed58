"""The C-ABI library loads, exports what include/cpe.h declares, validates
arguments on the host, and its planners match the oracle's bit for bit.
No CUDA call is made here (host-only entry points and pre-launch checks)."""
import json
import os
import random
import re

import pytest

import oracle
from chunked_prefill_extend_gb300 import cpe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "cpe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cpe_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = _declared()
    assert "cpe_extend_attention" in names and "cpe_mixed_step" in names and "cpe_kv_append" in names
    for n in names:
        assert hasattr(cpe._lib, n), f"libcpe.so does not export {n}"
    assert sorted(cpe.EXPORTS) == names


@pytest.mark.parametrize("n,hit,c,align", [(4000, 0.0, 512, 0), (32768, 0.5, 8192, 0), (131072, 0.0, 1024, 0),
                                           (10000, 0.0, 4096, 0), (4096, 0.0, 8192, 0), (1000, 0.01, 100, 16),
                                           (1, 0.0, 1, 0), (99991, 0.37, 333, 16), (7, 0.5, 2, 4)])
def test_plan_chunks_matches_oracle(n, hit, c, align):
    chunks, cached, eff = cpe.cpe_plan_chunks(n, hit, c, align)
    ref = oracle.plan_chunks(n, hit, c, align)
    assert [tuple(vars(x).values()) for x in chunks] == [tuple(vars(x).values()) for x in ref]
    assert (cached, eff) == oracle.effective_input_length(n, hit)


def test_plan_chunks_random_against_oracle():
    rng = random.Random(7)
    for _ in range(300):
        n = rng.randint(1, 200000)
        hit = rng.choice([0.0, 0.5, rng.random()])
        c = rng.randint(1, 9000)
        align = rng.choice([0, 0, 16, 64])
        try:
            ref = oracle.plan_chunks(n, hit, c, align)
        except ValueError:
            with pytest.raises(cpe.CpeError):
                cpe.cpe_plan_chunks(n, hit, c, align)
            continue
        got, _, _ = cpe.cpe_plan_chunks(n, hit, c, align)
        assert [tuple(vars(x).values()) for x in got] == [tuple(vars(x).values()) for x in ref]


@pytest.mark.parametrize("bad", [0, -1])
def test_plan_chunks_rejects_nonpositive_chunk(bad):
    with pytest.raises(cpe.CpeError) as e:
        cpe.cpe_plan_chunks(1000, 0.0, bad)
    assert e.value.status == cpe.CPE_ERR_INVALID_ARG


def test_plan_budget_and_mixed_step_match_oracle():
    rng = random.Random(11)
    for _ in range(200):
        budget = rng.randint(1, 5000)
        needs = [rng.randint(0, 3000) for _ in range(rng.randint(0, 12))]
        got, used = cpe.cpe_plan_budget(budget, needs)
        assert got == oracle.budget_truncate(budget, needs) and used == sum(got)
        ctx = [rng.randint(1, 40000) for _ in range(rng.randint(0, 300))]
        P, rem = rng.randint(0, 50000), rng.randint(0, 9000)
        a = cpe.cpe_plan_mixed_step(budget, ctx, P, rem)
        b = oracle.plan_mixed_step(budget, ctx, P, rem)
        assert a == b


def test_plan_schedule_matches_oracle():
    rng = random.Random(12)
    for _ in range(300):
        budget = rng.randint(1, 6000)
        running = [(rng.randint(0, 40000), rng.choice([1, 1, rng.randint(1, 4000)])) for _ in range(rng.randint(0, 40))]
        waiting = []
        for _ in range(rng.randint(0, 8)):
            cached = rng.randint(0, 5000)
            waiting.append((cached, cached + rng.randint(1, 6000)))
        assert cpe.cpe_plan_schedule(budget, running, waiting) == oracle.plan_schedule(budget, running, waiting)
    golden = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "plan_vectors.json")))
    for case in golden["schedule_examples"]:
        out = cpe.cpe_plan_schedule(case["budget"], [tuple(x) for x in case["running"]],
                                    [tuple(x) for x in case["waiting"]])
        assert out["granted"] == case["granted"] and out["n_admitted"] == case["n_admitted"]


def test_plan_schedule_errors():
    for budget, running, waiting in [(0, [], [(0, 5)]), (8, [(-1, 2)], []), (8, [(3, 0)], []), (8, [], [(5, 5)]),
                                     (8, [], [(-2, 5)]), (8, [(2**31 - 10, 20)], [])]:
        with pytest.raises(cpe.CpeError):
            cpe.cpe_plan_schedule(budget, running, waiting)


def test_mixed_step_budget_2304_shape():
    out = cpe.cpe_plan_mixed_step(2304, [1000] * 256, 30720, 4096)
    assert out["extend_len"] == 2048 and out["n_decode"] == 256 and out["qo_indptr"][-1] == 2304


def test_host_validation_happens_before_any_launch():
    """Bad arguments come back as status codes; nothing touches a device."""
    f = cpe._lib.cpe_extend_attention
    fake = 1 << 20  # never dereferenced: validation fails first
    args = dict(q=fake, k=fake, v=fake, num_pages=10, pt=fake, max_pages=4, qo=fake, pl=fake, n_seqs=1,
                total_q=16, max_kv=64, h_q=32, h_kv=8, d=128, page=16, scale=0.088, dt=cpe.CPE_BF16,
                out=fake, lse=None, ws=fake, ws_bytes=1 << 30, stream=None)

    def call(**kw):
        a = dict(args, **kw)
        return f(a["q"], a["k"], a["v"], a["num_pages"], a["pt"], a["max_pages"], a["qo"], a["pl"], a["n_seqs"],
                 a["total_q"], a["max_kv"], a["h_q"], a["h_kv"], a["d"], a["page"], a["scale"], a["dt"], a["out"],
                 a["lse"], a["ws"], a["ws_bytes"], a["stream"])

    assert call(q=None) == cpe.CPE_ERR_INVALID_ARG
    assert call(d=96) == cpe.CPE_ERR_UNSUPPORTED
    assert call(page=32) == cpe.CPE_ERR_UNSUPPORTED
    assert call(h_q=24, h_kv=8) == cpe.CPE_ERR_UNSUPPORTED       # G = 3
    assert call(h_q=30, h_kv=8) == cpe.CPE_ERR_INVALID_ARG       # not a multiple
    assert call(n_seqs=0) == cpe.CPE_ERR_INVALID_ARG
    assert call(ws_bytes=16) == cpe.CPE_ERR_CAPACITY
    assert call(q=fake + 8) == cpe.CPE_ERR_INVALID_ARG           # misaligned
    assert call(scale=float("nan")) == cpe.CPE_ERR_INVALID_ARG
    assert "workspace" in cpe.cpe_last_error() or "scale" in cpe.cpe_last_error()
    assert cpe.cpe_status_string(cpe.CPE_ERR_TIMEOUT) == "device wait timed out"


def test_workspace_size_is_monotone_and_zero_for_bad_sizes():
    a = cpe.cpe_workspace_size(1, 512, 32, 8, 128, 4000)
    b = cpe.cpe_workspace_size(257, 2304, 32, 8, 128, 32768)
    assert 0 < a < b and b % 256 == 0
    assert cpe.cpe_workspace_size(0, 1, 32, 8, 128, 10) == 0


def test_decide_decode_first_matches_oracle_and_pages():
    from oracle import sched_sim
    golden = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "sched_vectors.json")))
    for c in golden["decide"]:
        assert cpe.cpe_decide_decode_first(c["max_batched_tokens"], c["ready_decode"], c["pending_prefill"],
                                           c["chunk_query_len"]) == (c["p_step"], c["d_step"])
    rng = random.Random(13)
    sch = sched_sim.DecodeFirstWithSlack()
    for _ in range(500):
        B = rng.randint(1, 9000)
        st = sched_sim.SchedulerState(rng.randint(0, 12000), rng.randint(0, 50), rng.randint(1, B), B)
        want = sch.decide(st)
        assert tuple(cpe.cpe_decide_decode_first(B, st.ready_decode, st.pending_prefill, st.chunk_query_len)) == \
            (want.p_step, want.d_step)
    with pytest.raises(cpe.CpeError):
        cpe.cpe_decide_decode_first(0, 1, 1, 1)


def test_simulate_requests_matches_oracle():
    """The native simulation gives bit-identical times to the oracle's for the
    same latency model, with the default and with an injected scheduler."""
    from oracle import sched_sim

    class PrefillFirst:
        def decide(self, st):
            if st.pending_prefill:
                return sched_sim.StepDecision(st.pending_prefill, 0)
            return sched_sim.StepDecision(0, min(st.ready_decode, st.max_batched_tokens))

        def step_latency(self, p, d):
            return p + d

    rng = random.Random(14)
    for trial in range(40):
        B = rng.choice([128, 512, 2048, 4000])
        n_in = rng.randint(1, 12000)
        chunks, done = [], 0
        while done < n_in:
            q = min(B, n_in - done)
            done += q
            chunks.append((q, done))
        N, O = rng.randint(1, 60), rng.randint(1, 40)
        lat = lambda d, b, q, s: (0.25 + 3e-5 * b * s) if d else (0.5 + 2e-8 * b * q * s)
        sch = PrefillFirst() if trial % 4 == 3 else None
        a = cpe.cpe_simulate_requests(chunks, N, O, B, lat, sch)
        b = sched_sim.simulate(chunks, N, O, B, lat, sch)
        for k in ("makespan", "steps", "first_token_time", "finish_time"):
            assert a[k] == b[k], (trial, k)
        # means: Python's float sum() compensates rounding, the native loop adds plainly
        for k in ("ttft", "tpot", "request_throughput", "output_throughput"):
            assert a[k] == pytest.approx(b[k], rel=1e-12, abs=1e-12), (trial, k)


def test_simulate_requests_errors():
    lat = lambda d, b, q, s: 1.0
    with pytest.raises(cpe.CpeError):
        cpe.cpe_simulate_requests([], 1, 1, 10, lat)
    with pytest.raises(cpe.CpeError):
        cpe.cpe_simulate_requests([(5, 5)], 1, 1, 10, lambda d, b, q, s: -1.0)

    class Idle:
        def decide(self, st):
            return (0, 0)

        def step_latency(self, p, d):
            return 0.0
    with pytest.raises(cpe.CpeError):
        cpe.cpe_simulate_requests([(5, 5)], 2, 2, 10, lat, Idle())
