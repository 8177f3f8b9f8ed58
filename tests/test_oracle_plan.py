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
