"""Chunk and mixed-step planning, written out plainly from the pages.

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
benchmark's CPU-baseline leg may use this module; the product path may not.

Sources:
- msmodeling chunked-prefill RFC (gitcode.com/Ascend/msmodeling, docs/RFC/
  rfc_chunked_prefill_support_zh.md), section 2.2 (prefix cache: cached prefix
  = floor(input_length * hit_rate), effective length = the rest; decode keeps the
  full input length) and section 3.1.3 (chunk plan: a loop taking
  min(chunk_size, remaining) tokens per chunk, with seq_len = tokens consumed
  so far in the effective part).
- SGLang chunked-prefill article (zdszero.github.io/chunked_prefill.html),
  section on turning one prefill into resumable extends: P_t, E_t, S_t and the
  cursor [prefix_len, extend_end); section on the implementation details: only
  the first cut of a new request aligns its absolute end to the page size.
- vLLM token-budget tutorial (hyflu.top/posts/chunked-prefill-token-budget),
  section 5: each scheduled request takes min(need, remaining budget), running
  requests first, then waiting ones; a decode request needs one token.
- SGLang article, mixed-chunk section: with mixed chunks the chunk shrinks by
  the number of running decode requests.

Readings where the pages are silent or disagree:
- prefix_len / seq_len carry the attention-exact context (cached prefix
  included, as the SGLang cursor needs), model_seq_len carries the RFC's
  modeller value (cached prefix left out).  Chunk counts and query lengths are
  the same under both.
- Alignment is off unless ``align_to`` > 0; then only a truncated first chunk
  has its absolute end rounded down to a multiple of ``align_to`` (kept
  unaligned if rounding would leave it empty).
- A decode row of context length L has L-1 cached tokens and appends one.
"""
from __future__ import annotations

import math
from dataclasses import dataclass


@dataclass(frozen=True)
class Chunk:
    index: int
    prefix_len: int
    query_len: int
    seq_len: int
    model_seq_len: int


def effective_input_length(input_len: int, hit_rate: float) -> tuple[int, int]:
    """(cached_prefix_tokens, effective_input_length) from the RFC's section 2.2."""
    cached = math.floor(input_len * hit_rate)
    return cached, input_len - cached


def plan_chunks(input_len: int, hit_rate: float, chunk_size: int, align_to: int = 0) -> list[Chunk]:
    if chunk_size <= 0:
        raise ValueError("chunk_size (max_batched_tokens) must be > 0")
    if input_len <= 0 or not (0.0 <= hit_rate <= 1.0):
        raise ValueError("input_len must be > 0 and hit_rate in [0, 1]")
    cached, effective = effective_input_length(input_len, hit_rate)
    if effective < 1:
        raise ValueError("effective_input_length must be >= 1")
    chunks = []
    consumed = 0
    index = 0
    while consumed < effective:
        remaining = effective - consumed
        take = min(chunk_size, remaining)
        if align_to > 0 and index == 0 and take < remaining:
            end = ((cached + take) // align_to) * align_to
            if end > cached:
                take = end - cached
        prefix = cached + consumed
        chunks.append(Chunk(index, prefix, take, prefix + take, consumed + take))
        consumed += take
        index += 1
    return chunks


def budget_truncate(token_budget: int, needs: list[int]) -> list[int]:
    """Tokens granted to each request, in order: min(need, what is left)."""
    granted = []
    left = token_budget
    for need in needs:
        take = min(need, left) if left > 0 else 0
        granted.append(take)
        left -= take
    return granted


def plan_mixed_step(token_budget: int, decode_ctx_len: list[int], prefill_prefix_len: int,
                    prefill_remaining: int) -> dict:
    """Decode rows first (one token each), then one prefill chunk from what is left.

    Returns the varlen batch: qo_indptr, prefix_len, kv_len (all per scheduled
    sequence, decode rows first), the number of decode rows scheduled and the
    prefill extend length (0 for a decode-only step).
    """
    if token_budget <= 0:
        raise ValueError("token_budget must be > 0")
    if any(L < 1 for L in decode_ctx_len) or prefill_prefix_len < 0 or prefill_remaining < 0:
        raise ValueError("bad lengths")
    granted = budget_truncate(token_budget, [1] * len(decode_ctx_len) + [prefill_remaining])
    qo = [0]
    prefix = []
    kv = []
    n_dec = 0
    for L, g in zip(decode_ctx_len, granted[:-1]):
        if g == 1:
            prefix.append(L - 1)
            kv.append(L)
            qo.append(qo[-1] + 1)
            n_dec += 1
    extend = granted[-1]
    if extend > 0:
        prefix.append(prefill_prefix_len)
        kv.append(prefill_prefix_len + extend)
        qo.append(qo[-1] + extend)
    return {"qo_indptr": qo, "prefix_len": prefix, "kv_len": kv, "n_decode": n_dec,
            "extend_len": extend}


def plan_schedule(token_budget: int, running: list[tuple[int, int]],
                  waiting: list[tuple[int, int]]) -> dict:
    """One scheduling step over running and waiting requests, as the vLLM
    tutorial's section 5 sketches ``schedule()`` (memory allocation and
    preemption left out: the caller owns the cache).

    running: (computed, need) per running request, in queue order: tokens whose
        K/V are already cached and tokens still to process (1 for a decode, the
        unfinished part of a prompt for a prefill continuation).
    waiting: (cached, prompt) per waiting request, in queue order: prefix-cache
        hit and prompt length; such a request needs prompt - cached tokens.

    Running requests take min(need, budget left) in order until the budget is
    spent; then waiting requests are admitted in order the same way while any
    budget is left.  The granted token count is the chunk: a prompt that does
    not fit is cut, and the rest waits for the next step.

    The batch lists every scheduled request as one sequence: those granted a
    single token first (decode rows, in scheduling order), then the others in
    scheduling order.  prefix_len is the request's cached tokens, kv_len adds
    the granted ones; seq_request names the request (running index r, or
    len(running) + waiting index).
    """
    if token_budget <= 0:
        raise ValueError("token_budget must be > 0")
    for computed, need in running:
        if computed < 0 or need < 1:
            raise ValueError("a running request needs computed >= 0 and need >= 1")
    for cached, prompt in waiting:
        if cached < 0 or prompt - cached < 1:
            raise ValueError("a waiting request needs cached >= 0 and prompt - cached >= 1")
    left = token_budget
    granted = []
    for computed, need in running:
        take = min(need, left)
        granted.append(take)
        left -= take
    admitted = 0
    for cached, prompt in waiting:
        if left == 0:
            granted.append(0)
            continue
        take = min(prompt - cached, left)
        granted.append(take)
        left -= take
        admitted += 1
    base = [c for c, _ in running] + [c for c, _ in waiting]
    order = ([r for r, g in enumerate(granted) if g == 1] +
             [r for r, g in enumerate(granted) if g > 1])
    qo = [0]
    for r in order:
        qo.append(qo[-1] + granted[r])
    return {"granted": granted, "n_admitted": admitted, "qo_indptr": qo,
            "prefix_len": [base[r] for r in order],
            "kv_len": [base[r] + granted[r] for r in order],
            "seq_request": order, "n_decode": sum(1 for g in granted if g == 1)}
