"""Pins for the oracle's planners: the pages' printed chunk plans and budgets."""
import json
import math
import os

import pytest

from oracle import plan

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "plan_vectors.json")))


@pytest.mark.parametrize("case", GOLDEN["chunk_plans"], ids=lambda c: f"{c['input_len']}@{c['chunk']}")
def test_chunk_plan_matches_pages(case):
    chunks = plan.plan_chunks(case["input_len"], case["hit_rate"], case["chunk"])
    if "query_lens" in case:
        assert [c.query_len for c in chunks] == case["query_lens"]
    if "count" in case:
        assert len(chunks) == case["count"]
    if "effective" in case:
        cached, eff = plan.effective_input_length(case["input_len"], case["hit_rate"])
        assert (cached, eff) == (case["cached"], case["effective"])
    if "seq_len_step" in case:
        assert [c.model_seq_len for c in chunks] == [case["seq_len_step"] * (k + 1)
                                                     for k in range(len(chunks))]


@pytest.mark.parametrize("bad", GOLDEN["invalid_chunk_sizes"]["values"])
def test_chunk_size_must_be_positive(bad):
    with pytest.raises(ValueError):
        plan.plan_chunks(1000, 0.0, bad)


def test_effective_length_below_one_is_an_error():
    with pytest.raises(ValueError):
        plan.plan_chunks(100, 1.0, 64)


@pytest.mark.parametrize("n,hit,c", [(1, 0.0, 1), (17, 0.0, 16), (4000, 0.0, 512), (32768, 0.5, 8192),
                                      (10001, 0.3, 777), (131072, 0.0, 1024), (99, 0.99, 7)])
def test_plan_closed_form(n, hit, c):
    """Count = ceil(E/C); query lengths sum to E; the cursor advances by E_t;
    every chunk but the last is full; P_t = cached + t*C (the SGLang round formulas)."""
    chunks = plan.plan_chunks(n, hit, c)
    cached = math.floor(n * hit)
    eff = n - cached
    assert len(chunks) == -(-eff // c)
    assert sum(ch.query_len for ch in chunks) == eff
    for t, ch in enumerate(chunks):
        assert ch.index == t
        assert ch.prefix_len == cached + min(t * c, eff)
        assert ch.query_len == min(c, eff - t * c)
        assert ch.seq_len == ch.prefix_len + ch.query_len
        assert ch.model_seq_len == ch.seq_len - cached
    assert chunks[-1].seq_len == n


def test_first_cut_page_alignment():
    """Only a truncated first chunk has its absolute end aligned to the page."""
    chunks = plan.plan_chunks(1000, 0.01, 100, align_to=16)   # cached 10
    assert chunks[0].prefix_len == 10
    assert chunks[0].seq_len % 16 == 0 and chunks[0].seq_len == 96
    assert all(c.query_len == 100 for c in chunks[1:-1])      # continuations not re-aligned
    assert sum(c.query_len for c in chunks) == 990
    # aligned already: identical to the unaligned plan
    assert plan.plan_chunks(32768, 0.5, 8192, align_to=16) == plan.plan_chunks(32768, 0.5, 8192)
    # a single chunk is never truncated, so never aligned
    assert plan.plan_chunks(50, 0.1, 100, align_to=16)[0].query_len == 45


@pytest.mark.parametrize("case", GOLDEN["budget_examples"], ids=lambda c: str(c["budget"]))
def test_budget_truncation_matches_pages(case):
    assert plan.budget_truncate(case["budget"], case["needs"]) == case["granted"]


def test_mixed_chunk_size():
    g = GOLDEN["mixed_chunk"]
    ctx = list(range(600, 600 + g["n_decode"]))
    out = plan.plan_mixed_step(g["token_budget"], ctx, 30720, 10000)
    assert out["extend_len"] == g["extend_len"]
    assert out["n_decode"] == g["n_decode"]
    assert out["qo_indptr"][-1] == g["token_budget"]
    # decode rows: one token each, context L includes it
    assert out["prefix_len"][:3] == [599, 600, 601]
    assert out["kv_len"][:3] == [600, 601, 602]
    assert out["prefix_len"][-1] == 30720 and out["kv_len"][-1] == 30720 + 2048


def test_mixed_step_edges():
    # decode-only: no prefill left
    out = plan.plan_mixed_step(64, [5, 6], 100, 0)
    assert out["extend_len"] == 0 and out["qo_indptr"] == [0, 1, 2]
    # budget smaller than the decode count: later decode rows sit out, no prefill
    out = plan.plan_mixed_step(3, [5, 6, 7, 8], 100, 50)
    assert out["n_decode"] == 3 and out["extend_len"] == 0
    # prefill only
    out = plan.plan_mixed_step(64, [], 0, 1000)
    assert out["qo_indptr"] == [0, 64] and out["prefix_len"] == [0]
    with pytest.raises(ValueError):
        plan.plan_mixed_step(0, [5], 0, 10)


@pytest.mark.parametrize("case", GOLDEN["schedule_examples"], ids=lambda c: str(c["budget"]))
def test_schedule_matches_pages(case):
    out = plan.plan_schedule(case["budget"], [tuple(x) for x in case["running"]],
                             [tuple(x) for x in case["waiting"]])
    assert out["granted"] == case["granted"]
    assert out["n_admitted"] == case["n_admitted"]
    reqs = [tuple(x) for x in case["running"]] + [(c, p - c) for c, p in case["waiting"]]
    # one-token sequences first, then the chunks, each in scheduling order
    ones = [r for r, g in enumerate(case["granted"]) if g == 1]
    many = [r for r, g in enumerate(case["granted"]) if g > 1]
    assert out["seq_request"] == ones + many
    assert out["prefix_len"] == [reqs[r][0] for r in ones + many]
    assert out["kv_len"] == [reqs[r][0] + case["granted"][r] for r in ones + many]
    assert out["qo_indptr"][-1] == sum(case["granted"])
    if "next_step_running" in case:  # the cut prompt continues from where it stopped
        (cached, prompt), = case["waiting"]
        nxt = [(cached + case["granted"][0], prompt - cached - case["granted"][0])]
        assert nxt == [tuple(x) for x in case["next_step_running"]]


def test_schedule_waiting_need_excludes_prefix_cache_hit():
    """A waiting request needs its prompt minus the cached prefix, and its
    chunk starts after that prefix (the sketch's num_tokens - num_cached)."""
    out = plan.plan_schedule(2048, [], [(1000, 1500), (256, 4096)])
    assert out["granted"] == [500, 1548]
    assert out["prefix_len"] == [1000, 256] and out["kv_len"] == [1500, 1804]


def test_schedule_reproduces_chunk_plan():
    """One request scheduled step after step under a fixed budget is cut exactly
    as the chunk planner cuts it (same query and prefix lengths)."""
    for n, hit, c in [(4000, 0.0, 512), (10000, 0.0, 4096), (32768, 0.5, 8192), (999, 0.3, 128)]:
        cached, eff = plan.effective_input_length(n, hit)
        steps = []
        out = plan.plan_schedule(c, [], [(cached, n)])
        while True:
            steps.append((out["prefix_len"][0], out["qo_indptr"][-1]))
            done = out["kv_len"][0]
            if done == n:
                break
            out = plan.plan_schedule(c, [(done, n - done)], [])
        assert steps == [(ch.prefix_len, ch.query_len) for ch in plan.plan_chunks(n, hit, c)]


def test_schedule_reduces_to_mixed_step():
    """Decode rows plus one running prefill: the same batch as the mixed-step planner."""
    for budget, ctx, P, rem in [(2304, list(range(600, 856)), 30720, 10000), (64, [5, 6], 100, 0),
                                (3, [5, 6, 7, 8], 100, 50), (64, [], 0, 1000), (300, [9] * 10, 4096, 100)]:
        running = [(L - 1, 1) for L in ctx] + ([(P, rem)] if rem > 0 else [])
        a = plan.plan_schedule(budget, running, [])
        b = plan.plan_mixed_step(budget, ctx, P, rem)
        assert a["qo_indptr"] == b["qo_indptr"] and a["prefix_len"] == b["prefix_len"]
        assert a["kv_len"] == b["kv_len"]
        if b["extend_len"] != 1:
            assert a["n_decode"] == b["n_decode"]


def test_schedule_invariants():
    import random
    rng = random.Random(7)
    for _ in range(300):
        budget = rng.randint(1, 5000)
        running = [(rng.randint(0, 9000), rng.choice([1, 1, 1, rng.randint(1, 3000)])) for _ in range(rng.randint(0, 12))]
        waiting = []
        for _ in range(rng.randint(0, 6)):
            cached = rng.randint(0, 2000)
            waiting.append((cached, cached + rng.randint(1, 3000)))
        out = plan.plan_schedule(budget, running, waiting)
        g = out["granted"]
        needs = [nd for _, nd in running] + [p - c for c, p in waiting]
        assert sum(g) <= budget and all(0 <= x <= nd for x, nd in zip(g, needs))
        # a request cut short (or skipped) means the budget ran out at it
        for r, (x, nd) in enumerate(zip(g, needs)):
            if x < nd:
                assert sum(g[:r + 1]) == budget and all(y == 0 for y in g[r + 1:])
        # admitted waiting requests are a prefix of the queue
        gw = g[len(running):]
        assert out["n_admitted"] == sum(1 for x in gw if x > 0) and all(x > 0 for x in gw[:out["n_admitted"]])
        assert out["qo_indptr"][-1] == sum(g) and out["n_decode"] == sum(1 for x in g if x == 1)


def test_schedule_argument_errors():
    for args in [(0, [], [(0, 10)]), (10, [(-1, 1)], []), (10, [(5, 0)], []), (10, [], [(10, 10)]),
                 (10, [], [(-1, 5)])]:
        with pytest.raises(ValueError):
            plan.plan_schedule(*args)
