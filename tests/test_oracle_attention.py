"""Pins for the float64 attention oracle.

Each test checks the oracle against something other than itself: closed forms
(one key, zero queries), a library routine (torch's float64 scaled-dot-product
attention and logsumexp with an explicit extend mask), and the invariants the
SGLang chunked-prefill article states (chunked extend equals one-shot causal
prefill; the two-stage merge equals the direct softmax).  The last test plants
mistakes in the oracle and checks that a pin catches each one.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from chunked_prefill_extend_gb300 import workloads as W

PG = 16


def _varlen_case(seed, lens, h_q, h_kv, d, dtype=torch.bfloat16, perm=True, std=1.0):
    """Random varlen batch: lens = [(P, E), ...] per sequence, pages shuffled."""
    g = torch.Generator().manual_seed(seed)
    npages = [-(-(P + E) // PG) for P, E in lens]
    total_pages = sum(npages) + 3
    order = torch.randperm(total_pages, generator=g) if perm else torch.arange(total_pages)
    max_pages = max(npages)
    pt = torch.full((len(lens), max_pages), -1, dtype=torch.int32)
    off = 0
    for s, n in enumerate(npages):
        pt[s, :n] = order[off:off + n].to(torch.int32)
        off += n
    kc = (torch.randn(total_pages, PG, h_kv, d, generator=g) * std).to(dtype)
    vc = (torch.randn(total_pages, PG, h_kv, d, generator=g) * std).to(dtype)
    total_q = sum(E for _, E in lens)
    q = (torch.randn(total_q, h_q, d, generator=g) * std).to(dtype)
    qo = [0]
    for _, E in lens:
        qo.append(qo[-1] + E)
    return q, kc, vc, pt, qo, [P for P, _ in lens]


def _gather_seq(kc, pt, s, n):
    """K (or V) of positions [0, n) of sequence s, contiguous [n, H_kv, d], by indexing."""
    pos = torch.arange(n)
    return kc[pt[s, pos // PG].long(), pos % PG]


def _sdpa_reference(q, kc, vc, pt, qo, prefix, h_q, h_kv):
    """Library routine: torch SDPA in float64 with the extend mask j <= P+i."""
    G = h_q // h_kv
    outs, lses = [], []
    for s in range(len(prefix)):
        P, E = prefix[s], qo[s + 1] - qo[s]
        qs = q[qo[s]:qo[s + 1]].double().transpose(0, 1)                 # [H, E, d]
        ks = _gather_seq(kc, pt, s, P + E).double().repeat_interleave(G, dim=1).transpose(0, 1)
        vs = _gather_seq(vc, pt, s, P + E).double().repeat_interleave(G, dim=1).transpose(0, 1)
        mask = torch.arange(P + E)[None, :] <= (P + torch.arange(E))[:, None]
        o = torch.nn.functional.scaled_dot_product_attention(qs, ks, vs, attn_mask=mask)
        scores = (qs @ ks.transpose(1, 2)) / math.sqrt(q.shape[-1])
        lse = torch.logsumexp(scores.masked_fill(~mask, float("-inf")), dim=-1)
        outs.append(o.transpose(0, 1))
        lses.append(lse.transpose(0, 1))
    return torch.cat(outs).numpy(), torch.cat(lses).numpy()


CASES = [
    # (seed, [(P, E), ...], h_q, h_kv, d)
    (11, [(0, 1)], 2, 1, 4),
    (12, [(0, 37)], 4, 4, 8),
    (13, [(16, 16), (5, 1), (0, 20), (33, 7)], 8, 2, 16),
    (14, [(40, 24), (63, 1), (1, 1)], 4, 1, 64),
    (15, [(100, 30)], 16, 2, 32),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"seed{c[0]}")
def test_direct_matches_library_sdpa(case):
    seed, lens, h_q, h_kv, d = case
    q, kc, vc, pt, qo, prefix = _varlen_case(seed, lens, h_q, h_kv, d)
    out, lse = oracle.extend_attention(q, kc, vc, pt, qo, prefix, h_q, h_kv)
    ref_o, ref_l = _sdpa_reference(q, kc, vc, pt, qo, prefix, h_q, h_kv)
    np.testing.assert_allclose(out, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, rtol=0, atol=1e-12)


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"seed{c[0]}")
def test_two_stage_merge_equals_direct(case):
    seed, lens, h_q, h_kv, d = case
    q, kc, vc, pt, qo, prefix = _varlen_case(seed, lens, h_q, h_kv, d)
    o1, l1 = oracle.extend_attention(q, kc, vc, pt, qo, prefix, h_q, h_kv)
    o2, l2 = oracle.extend_attention_two_stage(q, kc, vc, pt, qo, prefix, h_q, h_kv)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l2, l1, rtol=1e-12, atol=1e-13)


def test_single_key_returns_its_value():
    q, kc, vc, pt, qo, prefix = _varlen_case(21, [(0, 1)], 4, 2, 8)
    out, lse = oracle.extend_attention(q, kc, vc, pt, qo, prefix, 4, 2)
    page = int(pt[0, 0])
    for h in range(4):
        np.testing.assert_array_equal(out[0, h], vc[page, 0, h // 2].double().numpy())
        dot = float((q[0, h].double() * kc[page, 0, h // 2].double()).sum())
        assert lse[0, h] == pytest.approx(dot / math.sqrt(8), abs=1e-14)


def test_zero_query_gives_running_mean():
    """q = 0 makes every score 0: o_i is the plain mean of v_0..v_{P+i} and
    lse = ln(P+i+1)."""
    q, kc, vc, pt, qo, prefix = _varlen_case(22, [(9, 12), (0, 5)], 4, 2, 16)
    q.zero_()
    out, lse = oracle.extend_attention(q, kc, vc, pt, qo, prefix, 4, 2)
    for s in range(2):
        P, E = prefix[s], qo[s + 1] - qo[s]
        v = _gather_seq(vc, pt, s, P + E).double()
        for i in range(E):
            mean = v[:P + i + 1].mean(0)                        # [H_kv, d]
            for h in range(4):
                np.testing.assert_allclose(out[qo[s] + i, h], mean[h // 2].numpy(), atol=1e-14)
                assert lse[qo[s] + i, h] == pytest.approx(math.log(P + i + 1), abs=1e-14)


def test_dominant_key_selects_its_value():
    q, kc, vc, pt, qo, prefix = _varlen_case(23, [(20, 4)], 2, 1, 8, dtype=torch.float32)
    # make key at position 7 align with every query very strongly
    page, slot = int(pt[0, 7 // PG]), 7 % PG
    kc[page, slot, 0] = 4.0
    q.fill_(4.0)
    out, _ = oracle.extend_attention(q, kc, vc, pt, qo, prefix, 2, 1)
    for i in range(4):
        np.testing.assert_allclose(out[i, 0], vc[page, slot, 0].double().numpy(), atol=1e-9)


def test_chunked_equals_one_shot_fp32_512():
    """The article's exactness claim on the fp32 workload: four 128-token
    extend rounds through the paged cache equal one-shot causal prefill."""
    spec = W.CONFIGS["fp32-512"]
    req = W.make_chunked(spec, oracle.plan_chunks(spec.input_len, spec.hit_rate, spec.chunk)[0].prefix_len)
    one, one_lse = oracle.causal_attention(req.q, req.k, req.v, spec.h_q, spec.h_kv)
    outs, lses = [], []
    for ch in oracle.plan_chunks(spec.input_len, spec.hit_rate, spec.chunk):
        q, k, v = req.round_inputs(ch.prefix_len, ch.query_len)
        qo = [0, ch.query_len]
        oracle.kv_append(k, v, req.k_cache, req.v_cache, req.page_table, qo, [ch.prefix_len])
        o, l = oracle.extend_attention(q, req.k_cache, req.v_cache, req.page_table, qo,
                                       [ch.prefix_len], spec.h_q, spec.h_kv)
        outs.append(o)
        lses.append(l)
    np.testing.assert_allclose(np.concatenate(outs), one, rtol=0, atol=1e-12)
    np.testing.assert_allclose(np.concatenate(lses), one_lse, rtol=0, atol=1e-12)


def test_chunked_equals_one_shot_gqa_bf16():
    spec = W.shrink(W.CONFIGS["prefill-4000-c512"], input_len=300, chunk=64, h_q=8, h_kv=2, d=32, page_perm=True)
    req = W.make_chunked(spec, oracle.plan_chunks(spec.input_len, spec.hit_rate, spec.chunk)[0].prefix_len)
    one, _ = oracle.causal_attention(req.q, req.k, req.v, spec.h_q, spec.h_kv)
    outs = []
    for ch in oracle.plan_chunks(spec.input_len, 0.0, spec.chunk):
        q, k, v = req.round_inputs(ch.prefix_len, ch.query_len)
        oracle.kv_append(k, v, req.k_cache, req.v_cache, req.page_table, [0, ch.query_len],
                         [ch.prefix_len])
        outs.append(oracle.extend_attention(q, req.k_cache, req.v_cache, req.page_table,
                                            [0, ch.query_len], [ch.prefix_len], spec.h_q,
                                            spec.h_kv)[0])
    np.testing.assert_allclose(np.concatenate(outs), one, rtol=0, atol=1e-12)


def test_decode_row_equals_last_prefill_row():
    """A decode row (E=1 at P=L-1) is the last row of a one-shot prefill of L tokens."""
    g = torch.Generator().manual_seed(31)
    L, h_q, h_kv, d = 45, 8, 2, 16
    q = torch.randn(L, h_q, d, generator=g).to(torch.bfloat16)
    k = torch.randn(L, h_kv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(L, h_kv, d, generator=g).to(torch.bfloat16)
    one, _ = oracle.causal_attention(q, k, v, h_q, h_kv)
    npg = -(-L // PG)
    pt = torch.arange(npg, dtype=torch.int32).flip(0).view(1, -1).contiguous()
    kc = torch.zeros(npg, PG, h_kv, d, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    oracle.kv_append(k, v, kc, vc, pt, [0, L], [0])
    out, _ = oracle.extend_attention(q[L - 1:], kc, vc, pt, [0, 1], [L - 1], h_q, h_kv)
    np.testing.assert_allclose(out[0], one[L - 1], rtol=0, atol=1e-12)


def test_page_permutation_leaves_output_bitwise_unchanged():
    q, kc, vc, pt, qo, prefix = _varlen_case(41, [(30, 10), (7, 3)], 4, 2, 16, perm=False)
    out_a, lse_a = oracle.extend_attention(q, kc, vc, pt, qo, prefix, 4, 2)
    perm = torch.randperm(kc.shape[0], generator=torch.Generator().manual_seed(5))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(len(perm))
    kc2, vc2 = kc[perm].contiguous(), vc[perm].contiguous()      # physical page p moves to inv[p]
    pt2 = torch.where(pt >= 0, inv[pt.clamp(min=0).long()].to(torch.int32), pt)
    out_b, lse_b = oracle.extend_attention(q, kc2, vc2, pt2, qo, prefix, 4, 2)
    assert np.array_equal(out_a, out_b) and np.array_equal(lse_a, lse_b)


def test_kv_append_scatter_pins():
    g = torch.Generator().manual_seed(51)
    h_kv, d = 2, 8
    k_new = torch.randn(40, h_kv, d, generator=g).to(torch.bfloat16)
    v_new = torch.randn(40, h_kv, d, generator=g).to(torch.bfloat16)
    # identity pages, one sequence starting at 0: cache rows are the new rows in order
    kc = torch.zeros(3, PG, h_kv, d, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    pt = torch.arange(3, dtype=torch.int32).view(1, 3)
    oracle.kv_append(k_new, v_new, kc, vc, pt, [0, 40], [0])
    assert torch.equal(kc.view(-1, h_kv, d)[:40], k_new)
    assert torch.equal(vc.view(-1, h_kv, d)[:40], v_new)
    # two sequences at prefixes 5 and 17 on shuffled pages
    kc = torch.zeros(6, PG, h_kv, d, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    pt = torch.tensor([[4, 0, -1], [2, 5, 1]], dtype=torch.int32)
    oracle.kv_append(k_new, v_new, kc, vc, pt, [0, 10, 40], [5, 17])
    for r in range(10):
        pos = 5 + r
        assert torch.equal(kc[pt[0, pos // PG], pos % PG], k_new[r])
    for r in range(30):
        pos = 17 + r
        assert torch.equal(vc[pt[1, pos // PG], pos % PG], v_new[10 + r])
    with pytest.raises(RuntimeError):      # position 10+... past the page table
        oracle.kv_append(k_new, v_new, kc, vc, pt, [0, 40, 40], [40, 0])


@pytest.mark.parametrize("fault", [1, 2, 3], ids=["diagonal-dropped", "wrong-scale", "wrong-gqa-map"])
def test_planted_mistakes_are_caught(fault):
    seed, lens, h_q, h_kv, d = CASES[2]
    q, kc, vc, pt, qo, prefix = _varlen_case(seed, lens, h_q, h_kv, d)
    ref_o, _ = _sdpa_reference(q, kc, vc, pt, qo, prefix, h_q, h_kv)
    oracle.set_fault(fault)
    try:
        out, _ = oracle.extend_attention(q, kc, vc, pt, qo, prefix, h_q, h_kv)
    finally:
        oracle.set_fault(0)
    assert not np.allclose(out, ref_o, rtol=0, atol=1e-3)
