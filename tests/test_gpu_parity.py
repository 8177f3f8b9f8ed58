"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Small cases are compared element by element; the full-size workloads on
sampled rows (first, last, both sides of tile boundaries, seeded picks).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from chunked_prefill_extend_gb300 import workloads as W
from tests._util import check_close, extract_pages, i32, varlen_batch, LSE_ABS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cpe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunked_prefill_extend_gb300 import cpe as lib
    st, _ = lib.cpe_get_device_status()
    assert st == lib.CPE_OK
    return lib


def _cached(cpe, spec):
    """The prefix-cache hit of a chunked workload, from the chunk planner."""
    return cpe.cpe_plan_chunks(spec.input_len, spec.hit_rate, spec.chunk)[1]


def _status_ok(cpe):
    st, detail = cpe.cpe_get_device_status()
    assert st == cpe.CPE_OK, f"device status {cpe.cpe_status_string(st)} detail {detail}"


def _append_and_attend(cpe, b, lse=True):
    qo, pl = i32(b["qo"]), i32(b["pl"])
    cpe.cpe_kv_append(b["k_new"], b["v_new"], b["k_cache"], b["v_cache"], b["page_table"], qo, pl)
    lse_t = torch.empty(b["q"].shape[0], b["h_q"], dtype=torch.float32, device="cuda") if lse else None
    out, _ = cpe.cpe_extend_attention(b["q"], b["k_cache"], b["v_cache"], b["page_table"], qo, pl, b["max_kv"],
                                      lse=lse_t)
    _status_ok(cpe)
    return out, lse_t


def _oracle_batch(b):
    return oracle.extend_attention(b["q"].cpu(), b["k_cache"].cpu(), b["v_cache"].cpu(), b["page_table_host"],
                                   b["qo"], b["pl"], b["h_q"], b["h_kv"])


# ---------------------------------------------------------------- kv append

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_kv_append_bitwise(cpe, dtype):
    b = varlen_batch(1, [(0, 40), (17, 1), (100, 77), (5, 0), (33, 16)], 8, 2, 128, dtype=dtype)
    kc_ref, vc_ref = b["k_cache"].cpu().clone(), b["v_cache"].cpu().clone()
    oracle.kv_append(b["k_new"].cpu(), b["v_new"].cpu(), kc_ref, vc_ref, b["page_table_host"], b["qo"], b["pl"])
    cpe.cpe_kv_append(b["k_new"], b["v_new"], b["k_cache"], b["v_cache"], b["page_table"], i32(b["qo"]),
                      i32(b["pl"]))
    _status_ok(cpe)
    assert torch.equal(b["k_cache"].cpu(), kc_ref) and torch.equal(b["v_cache"].cpu(), vc_ref)


@pytest.mark.parametrize("h_q,h_kv,d,n_decode,long_seq", [(32, 8, 128, 0, None), (32, 8, 128, 0, (8192, 1024)),
                                                        (32, 2, 128, 0, (8192, 1024)), (8, 1, 64, 0, (32768, 2048)),
                                                        (32, 8, 128, 3, (8192, 1024))])
def test_mixed_step_cache_written_bitwise(cpe, h_q, h_kv, d, n_decode, long_seq):
    """cpe_mixed_step writes the round's K/V rows into the cache exactly as the
    append does.  On a long launch (a long sequence in the batch) the extend
    launch reads the chunk's keys from the new rows and writes the full new
    pages of sequences whose prefix ends on a page boundary from its staged
    tiles, the prep launch appending the rest; on a short one the prep launch
    appends every row.  Cache bitwise against the oracle's append, output
    against the oracle; page-aligned and unaligned prefixes, chunk lengths
    with and without a partial last page, G = 4, 16, 8, decode rows beside."""
    lens = [(L - 1, 1) for L in (40, 1, 2049)][:n_decode] + \
        [(0, 45), (32, 300), (17, 100), (512, 128), (100, 7), (2048, 700), (160, 16)] + ([long_seq] if long_seq else [])
    b = varlen_batch(80 + h_kv + n_decode + (1 if long_seq else 0), lens, h_q, h_kv, d)
    kc_ref, vc_ref = b["k_cache"].cpu().clone(), b["v_cache"].cpu().clone()
    oracle.kv_append(b["k_new"].cpu(), b["v_new"].cpu(), kc_ref, vc_ref, b["page_table_host"], b["qo"], b["pl"])
    lse = torch.empty(b["q"].shape[0], h_q, dtype=torch.float32, device="cuda")
    out, _ = cpe.cpe_mixed_step(b["q"], b["k_new"], b["v_new"], b["k_cache"], b["v_cache"], b["page_table"],
                                i32(b["qo"]), i32(b["pl"]), n_decode, b["max_kv"], lse=lse)
    _status_ok(cpe)
    assert torch.equal(b["k_cache"].cpu(), kc_ref) and torch.equal(b["v_cache"].cpu(), vc_ref)
    ref_o, ref_l = oracle.extend_attention(b["q"].cpu(), kc_ref, vc_ref, b["page_table_host"], b["qo"], b["pl"],
                                           h_q, h_kv)
    check_close(out, ref_o, f"mixed step {h_q}/{h_kv} d={d} decode={n_decode} long={long_seq}")
    np.testing.assert_allclose(lse.cpu().numpy(), ref_l, atol=LSE_ABS, rtol=0)


# ---------------------------------------------------------------- extend, small, full compare

SMALL = [
    # (seed, [(P, E), ...], h_q, h_kv, d)
    (10, [(0, 1)], 32, 8, 128),                       # one key
    (11, [(0, 300)], 32, 8, 128),                     # P = 0, several tiles, ragged tail
    (12, [(517, 45)], 32, 8, 128),                    # prefix + short chunk
    (13, [(129, 1)], 32, 8, 128),                     # E = 1 at a tile boundary
    (14, [(100, 64), (0, 33), (2000, 130), (7, 0), (256, 128)], 32, 8, 128),  # varlen incl. empty
    (15, [(300, 200)], 8, 8, 128),                    # G = 1
    (16, [(250, 170)], 16, 8, 128),                   # G = 2
    (17, [(333, 99)], 64, 8, 128),                    # G = 8
    (18, [(140, 77)], 32, 2, 128),                    # G = 16
    (19, [(411, 150), (0, 20)], 32, 8, 64),           # d = 64
    (20, [(1000, 257)], 8, 1, 64),                    # G = 8, d = 64
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"seed{c[0]}")
def test_extend_small_full(cpe, case):
    seed, lens, h_q, h_kv, d = case
    b = varlen_batch(seed, lens, h_q, h_kv, d)
    out, lse = _append_and_attend(cpe, b)
    ref_o, ref_l = _oracle_batch(b)
    check_close(out, ref_o, f"out {case}")
    np.testing.assert_allclose(lse.cpu().numpy(), ref_l, atol=LSE_ABS, rtol=0)


def test_extend_fp32_path(cpe):
    b = varlen_batch(21, [(50, 70), (0, 9)], 4, 4, 64, dtype=torch.float32, std=1.0)
    out, lse = _append_and_attend(cpe, b)
    ref_o, ref_l = _oracle_batch(b)
    check_close(out, ref_o, "fp32", max_abs=1e-4, rel_rms=1e-5)
    np.testing.assert_allclose(lse.cpu().numpy(), ref_l, atol=1e-4, rtol=0)


def test_page_permutation_gives_bitwise_equal_output(cpe):
    b = varlen_batch(22, [(700, 300)], 32, 8, 128)
    out_a, _ = _append_and_attend(cpe, b, lse=False)
    perm = torch.randperm(b["k_cache"].shape[0], generator=torch.Generator().manual_seed(3))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(len(perm))
    b2 = dict(b)
    b2["k_cache"] = b["k_cache"][perm.cuda()].contiguous()
    b2["v_cache"] = b["v_cache"][perm.cuda()].contiguous()
    pth = b["page_table_host"]
    b2["page_table_host"] = torch.where(pth >= 0, inv[pth.clamp(min=0).long()].to(torch.int32), pth)
    b2["page_table"] = b2["page_table_host"].cuda()
    out_b, _ = _append_and_attend(cpe, b2, lse=False)
    assert torch.equal(out_a, out_b)


# ---------------------------------------------------------------- chunked == one-shot

def _chunked_run(cpe, spec, device="cuda", one_call=False, n_workspaces=0):
    """Every round through cpe_kv_append + cpe_extend_attention, or (one_call)
    through cpe_mixed_step with no decode rows (append and schedule share a launch).
    n_workspaces: 0 lets each call allocate its own; 1 reuses one workspace for
    every round; 2 alternates two (the rounds' launches then overlap more)."""
    req = W.make_chunked(spec, _cached(cpe, spec), device=device)
    chunks, _, _ = cpe.cpe_plan_chunks(spec.input_len, spec.hit_rate, spec.chunk)
    wss = [cpe.alloc_workspace(1, spec.chunk, spec.h_q, spec.h_kv, spec.d, spec.input_len, device)
           for _ in range(n_workspaces)]
    outs = []
    for ch in chunks:
        q, k, v = req.round_inputs(ch.prefix_len, ch.query_len)
        qo, pl = i32([0, ch.query_len]), i32([ch.prefix_len])
        ws = wss[ch.index % len(wss)] if wss else None
        if one_call:
            out, _ = cpe.cpe_mixed_step(q, k, v, req.k_cache, req.v_cache, req.page_table, qo, pl, 0, ch.seq_len,
                                        workspace=ws)
        else:
            cpe.cpe_kv_append(k, v, req.k_cache, req.v_cache, req.page_table, qo, pl)
            out, _ = cpe.cpe_extend_attention(q, req.k_cache, req.v_cache, req.page_table, qo, pl, ch.seq_len,
                                              workspace=ws)
        outs.append(out)
    _status_ok(cpe)
    return req, chunks, torch.cat(outs)


def test_fp32_512_chunked_equals_one_shot(cpe):
    spec = W.CONFIGS["fp32-512"]
    req, chunks, out = _chunked_run(cpe, spec)
    assert [c.query_len for c in chunks] == [128] * 4
    one, _ = oracle.causal_attention(req.q.cpu(), req.k.cpu(), req.v.cpu(), spec.h_q, spec.h_kv)
    check_close(out, one, "fp32-512 chunked vs one-shot", max_abs=1e-4, rel_rms=1e-5)
    # the GPU's own one-shot run (one chunk of 512) agrees with its chunked run
    spec1 = W.shrink(spec, chunk=512)
    _, _, out1 = _chunked_run(cpe, spec1)
    check_close(out, out1.double().cpu().numpy(), "fp32-512 gpu chunked vs gpu one-shot", max_abs=1e-4, rel_rms=1e-5)


def test_bf16_chunked_equals_one_shot(cpe):
    spec = W.shrink(W.CONFIGS["prefill-4000-c512"], input_len=1500, chunk=256)
    req, _, out = _chunked_run(cpe, spec)
    one, _ = oracle.causal_attention(req.q.cpu(), req.k.cpu(), req.v.cpu(), spec.h_q, spec.h_kv)
    check_close(out, one, "bf16 chunked vs one-shot")
    _, _, out1 = _chunked_run(cpe, W.shrink(spec, chunk=1500))
    check_close(out, out1.double().cpu().numpy(), "bf16 gpu chunked vs gpu one-shot")
    # one call per round (append inside the extend schedule's launch): same rounds, same answer
    _, _, out2 = _chunked_run(cpe, spec, one_call=True)
    check_close(out2, one, "bf16 chunked one call per round vs one-shot")
    assert torch.equal(out2, out)


def test_shared_prefix_pages_with_aligned_first_cut(cpe):
    """Radix-style sharing: two requests whose cached prefixes are the same 62
    full pages (992 tokens) in the page pool; each is chunked with the first cut
    aligned to the page size, and their rounds run together as one varlen
    batch.  Every round matches the oracle and the shared pages are never
    written."""
    h_q, h_kv, d, pg = 32, 8, 128, 16
    plans = [cpe.cpe_plan_chunks(3968, 0.25, 500, align_to=pg)[0], cpe.cpe_plan_chunks(1984, 0.5, 500, align_to=pg)[0]]
    assert [c.prefix_len for c in plans[0]][:2] == [992, 1488] and plans[0][0].query_len == 496
    g = torch.Generator().manual_seed(81)
    shared = 992 // pg
    own = [-(-3968 // pg) - shared, -(-1984 // pg) - shared]
    n_pages = shared + sum(own) + 2
    perm = torch.randperm(n_pages, generator=g).to(torch.int32)
    pt = torch.full((2, shared + max(own)), -1, dtype=torch.int32)
    pt[:, :shared] = perm[:shared]  # the same physical pages for both prefixes
    pt[0, shared:shared + own[0]] = perm[shared:shared + own[0]]
    pt[1, shared:shared + own[1]] = perm[shared + own[0]:shared + own[0] + own[1]]
    kc = (torch.randn(n_pages, pg, h_kv, d, generator=g) * 0.5).to(torch.bfloat16).cuda()
    vc = (torch.randn(n_pages, pg, h_kv, d, generator=g) * 0.5).to(torch.bfloat16).cuda()
    ptd = pt.cuda()
    shared_ids = pt[0, :shared].long().cuda()
    k_shared, v_shared = kc[shared_ids].clone(), vc[shared_ids].clone()
    for t in range(max(len(p) for p in plans)):
        seqs = [r for r in range(2) if t < len(plans[r])]
        lens = [(plans[r][t].prefix_len, plans[r][t].query_len) for r in seqs]
        rows = sum(E for _, E in lens)
        q = (torch.randn(rows, h_q, d, generator=g) * 0.5).to(torch.bfloat16).cuda()
        kn = (torch.randn(rows, h_kv, d, generator=g) * 0.5).to(torch.bfloat16).cuda()
        vn = (torch.randn(rows, h_kv, d, generator=g) * 0.5).to(torch.bfloat16).cuda()
        qo = [0]
        for _, E in lens:
            qo.append(qo[-1] + E)
        sub = ptd[seqs].contiguous()
        out, _ = cpe.cpe_mixed_step(q, kn, vn, kc, vc, sub, i32(qo), i32([P for P, _ in lens]), 0,
                                    max(P + E for P, E in lens))
        _status_ok(cpe)
        ref_o, _ = oracle.extend_attention(q.cpu(), kc.cpu(), vc.cpu(), pt[seqs].contiguous(), qo,
                                           [P for P, _ in lens], h_q, h_kv)
        check_close(out, ref_o, f"shared-prefix round {t}")
    assert torch.equal(kc[shared_ids], k_shared) and torch.equal(vc[shared_ids], v_shared)


def test_many_short_sequences(cpe):
    """2100 short sequences (over the schedule's 2048-sequence and 8192-unit
    shared-memory caches, so both fall back to global memory) in one extend
    call; the first and last row of every sequence and 600 more rows checked."""
    g = torch.Generator().manual_seed(91)
    n = 2100
    E = torch.randint(1, 41, (n,), generator=g).tolist()
    P = torch.randint(0, 201, (n,), generator=g).tolist()
    b = varlen_batch(92, list(zip(P, E)), 32, 8, 128, spare_pages=0)
    out, lse = _append_and_attend(cpe, b)
    qo = b["qo"]
    rows = sorted(set([qo[s] for s in range(n)] + [qo[s + 1] - 1 for s in range(n)] +
                      torch.randint(0, qo[-1], (600,), generator=g).tolist()))
    kc, vc = b["k_cache"].cpu().clone(), b["v_cache"].cpu().clone()
    ref_o, ref_l = oracle.extend_attention(b["q"].cpu(), kc, vc, b["page_table_host"], qo, b["pl"], 32, 8, rows=rows)
    check_close(out[rows], ref_o, "many short sequences")
    np.testing.assert_allclose(lse[rows].cpu().numpy(), ref_l, atol=LSE_ABS, rtol=0)


def test_workspace_rotations_and_two_streams(cpe):
    """A round's schedule is written before the previous launch finishes only
    when the previous call on the stream used another workspace.  Rotations
    A,B,A,B..., A,B,C,A,... and A,A,B,B,... and two requests on two streams
    (each stream alternating its own pair) all give the bits of the serial
    run with one workspace."""
    spec = W.shrink(W.CONFIGS["prefill-4000-c512"], input_len=2600, chunk=384)
    _, chunks, ref = _chunked_run(cpe, spec, one_call=True, n_workspaces=1)
    for n in (2, 3):
        _, _, out = _chunked_run(cpe, spec, one_call=True, n_workspaces=n)
        assert torch.equal(out, ref), n
    # A,A,B,B,...: every other call reuses the previous call's workspace
    req = W.make_chunked(spec, _cached(cpe, spec), device="cuda")
    wss = [cpe.alloc_workspace(1, spec.chunk, spec.h_q, spec.h_kv, spec.d, spec.input_len, "cuda") for _ in range(2)]
    outs = []
    for ch in chunks:
        q, k, v = req.round_inputs(ch.prefix_len, ch.query_len)
        out, _ = cpe.cpe_mixed_step(q, k, v, req.k_cache, req.v_cache, req.page_table, i32([0, ch.query_len]),
                                    i32([ch.prefix_len]), 0, ch.seq_len, workspace=wss[(ch.index // 2) % 2])
        outs.append(out)
    _status_ok(cpe)
    assert torch.equal(torch.cat(outs), ref)
    # two requests, one per stream, rounds issued alternately from the host
    reqs = [W.make_chunked(spec, _cached(cpe, spec), device="cuda") for _ in range(2)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    wsp = [[cpe.alloc_workspace(1, spec.chunk, spec.h_q, spec.h_kv, spec.d, spec.input_len, "cuda")
            for _ in range(2)] for _ in range(2)]
    outs = [[], []]
    torch.cuda.synchronize()
    for ch in chunks:
        for r in range(2):
            with torch.cuda.stream(streams[r]):
                q, k, v = reqs[r].round_inputs(ch.prefix_len, ch.query_len)
                out, _ = cpe.cpe_mixed_step(q, k, v, reqs[r].k_cache, reqs[r].v_cache, reqs[r].page_table,
                                            i32([0, ch.query_len]), i32([ch.prefix_len]), 0, ch.seq_len,
                                            workspace=wsp[r][ch.index % 2], stream=streams[r])
                outs[r].append(out)
    torch.cuda.synchronize()
    _status_ok(cpe)
    for r in range(2):
        assert torch.equal(torch.cat(outs[r]), ref), r


# ---------------------------------------------------------------- full-size workloads

def test_prefill_4000_c512_full(cpe):
    """Every row of prefill-4000-c512, each round in one call as the benchmark runs it (two
    workspaces alternated, so a round's tile list is written while the previous
    round runs); one shared workspace gives the same bits."""
    spec = W.CONFIGS["prefill-4000-c512"]
    req, chunks, out = _chunked_run(cpe, spec, one_call=True, n_workspaces=2)
    assert [c.query_len for c in chunks] == [512] * 7 + [416]
    one, _ = oracle.causal_attention(req.q.cpu(), req.k.cpu(), req.v.cpu(), spec.h_q, spec.h_kv)
    check_close(out, one, "prefill-4000-c512 all rows")
    _, _, out1 = _chunked_run(cpe, spec, one_call=True, n_workspaces=1)
    assert torch.equal(out, out1)
    # the separate append + extend calls, alternating too
    _, _, out2 = _chunked_run(cpe, spec, n_workspaces=2)
    assert torch.equal(out, out2)


def _sampled_rounds(cpe, spec, round_ids, n_rows, seed):
    req = W.make_chunked(spec, _cached(cpe, spec), device="cuda")
    chunks, cached, _ = cpe.cpe_plan_chunks(spec.input_len, spec.hit_rate, spec.chunk)
    for ch in chunks:  # every round's keys go into the cache first
        q, k, v = req.round_inputs(ch.prefix_len, ch.query_len)
        cpe.cpe_kv_append(k, v, req.k_cache, req.v_cache, req.page_table, i32([0, ch.query_len]),
                          i32([ch.prefix_len]))
    kc, vc = req.k_cache.cpu(), req.v_cache.cpu()
    G = spec.h_q // spec.h_kv
    for t in round_ids:
        ch = chunks[t]
        q, _, _ = req.round_inputs(ch.prefix_len, ch.query_len)
        lse = torch.empty(ch.query_len, spec.h_q, dtype=torch.float32, device="cuda")
        out, _ = cpe.cpe_extend_attention(q, req.k_cache, req.v_cache, req.page_table, i32([0, ch.query_len]),
                                          i32([ch.prefix_len]), ch.seq_len, lse=lse)
        _status_ok(cpe)
        rows = W.sample_rows(ch.query_len, 128 // G, n_rows, seed + t)
        ref_o, ref_l = oracle.extend_attention(q.cpu(), kc, vc,
                                               torch.tensor([req.page_table_host], dtype=torch.int32),
                                               [0, ch.query_len], [ch.prefix_len], spec.h_q, spec.h_kv, rows=rows)
        check_close(out[rows], ref_o, f"{spec.name} round {t}")
        np.testing.assert_allclose(lse[rows].cpu().numpy(), ref_l, atol=LSE_ABS, rtol=0)
    return chunks


def test_prefill_32k_hit50_sampled(cpe):
    chunks = _sampled_rounds(cpe, W.CONFIGS["prefill-32k-hit50"], [0, 1], 96, 300)
    assert [(c.prefix_len, c.query_len) for c in chunks] == [(16384, 8192), (24576, 8192)]


def test_prefill_128k_c1024_sampled(cpe):
    chunks = _sampled_rounds(cpe, W.CONFIGS["prefill-128k-c1024"], [0, 7, 127], 24, 500)
    assert len(chunks) == 128 and chunks[-1].seq_len == 131072


def test_prefill_128k_c1024_every_round_as_benchmarked(cpe):
    """All 128 rounds of prefill-128k-c1024 exactly as the benchmark runs them:
    one cpe_mixed_step per round (K/V append and extend attention in one
    call), two workspaces alternated, so every per-round schedule the
    benchmark times (1 to 5 key-range parts per unit, last-wave fill) is
    exercised.  In every round the first row, the last row and both rows
    around one query-tile boundary (a different boundary each round) are
    compared, all heads and keys, with the float64 oracle."""
    spec = W.CONFIGS["prefill-128k-c1024"]
    chunks, cached, _ = cpe.cpe_plan_chunks(spec.input_len, spec.hit_rate, spec.chunk)
    assert len(chunks) == 128 and cached == 0
    req = W.make_chunked(spec, cached, device="cuda")
    wss = [cpe.alloc_workspace(1, spec.chunk, spec.h_q, spec.h_kv, spec.d, spec.input_len, "cuda") for _ in range(2)]
    out = torch.empty_like(req.q)
    lse = torch.empty(req.q.shape[0], spec.h_q, dtype=torch.float32, device="cuda")
    tok = 128 // (spec.h_q // spec.h_kv)  # tokens per query tile
    rows = []
    for ch in chunks:
        a = ch.prefix_len - cached
        sl = slice(a, a + ch.query_len)
        cpe.cpe_mixed_step(req.q[sl], req.k[sl], req.v[sl], req.k_cache, req.v_cache, req.page_table,
                           i32([0, ch.query_len]), i32([ch.prefix_len]), 0, ch.seq_len, out=out[sl], lse=lse[sl],
                           workspace=wss[ch.index & 1])
        b = tok * (1 + (ch.index * 37) % (ch.query_len // tok - 1))
        rows += [a + r for r in (0, b - 1, b, ch.query_len - 1)]
    _status_ok(cpe)
    # the whole request as one batch of 128 sequences (one per round) for the oracle
    qo = [c.prefix_len - cached for c in chunks] + [spec.input_len - cached]
    pt = torch.tensor([req.page_table_host] * len(chunks), dtype=torch.int32)
    ref_o, ref_l = oracle.extend_attention(req.q.cpu(), req.k_cache.cpu(), req.v_cache.cpu(), pt, qo,
                                           [c.prefix_len for c in chunks], spec.h_q, spec.h_kv, rows=rows)
    for t in range(len(chunks)):
        r = rows[4 * t:4 * t + 4]
        check_close(out[r], ref_o[4 * t:4 * t + 4], f"prefill-128k-c1024 round {t} rows {r}")
        np.testing.assert_allclose(lse[r].cpu().numpy(), ref_l[4 * t:4 * t + 4], atol=LSE_ABS, rtol=0)


def test_d64_long_rounds_cut_units_sampled(cpe):
    """d = 64 with rounds long enough that the schedule cuts every unit into
    four or five key-range parts and fills the last wave, so the merge
    kernel's d = 64 path (one bf16 pair per lane) combines them; sampled rows
    against the oracle."""
    spec = W.shrink(W.CONFIGS["prefill-128k-c1024"], name="d64", input_len=32768, chunk=2048, h_q=32, h_kv=4, d=64)
    chunks = _sampled_rounds(cpe, spec, [0, 7], 32, 700)
    # the last round again, with a workspace whose schedule header can be read:
    # header[7] counts the units cut into parts
    req = W.make_chunked(spec, _cached(cpe, spec), device="cuda")
    for ch in chunks:
        q, k, v = req.round_inputs(ch.prefix_len, ch.query_len)
        cpe.cpe_kv_append(k, v, req.k_cache, req.v_cache, req.page_table, i32([0, ch.query_len]),
                          i32([ch.prefix_len]))
    ch = chunks[-1]
    q, _, _ = req.round_inputs(ch.prefix_len, ch.query_len)
    ws = cpe.alloc_workspace(1, ch.query_len, spec.h_q, spec.h_kv, spec.d, ch.seq_len, "cuda")
    out, _ = cpe.cpe_extend_attention(q, req.k_cache, req.v_cache, req.page_table, i32([0, ch.query_len]),
                                      i32([ch.prefix_len]), ch.seq_len, workspace=ws)
    _status_ok(cpe)
    assert int(ws[:32].view(torch.int32)[7]) > 0
    rows = W.sample_rows(ch.query_len, 128 // (spec.h_q // spec.h_kv), 32, 715)
    ref_o, _ = oracle.extend_attention(q.cpu(), req.k_cache.cpu(), req.v_cache.cpu(),
                                       torch.tensor([req.page_table_host], dtype=torch.int32),
                                       [0, ch.query_len], [ch.prefix_len], spec.h_q, spec.h_kv, rows=rows)
    check_close(out[rows], ref_o, "d64 last round, cut units")


# ---------------------------------------------------------------- decode rows

@pytest.mark.parametrize("lens", [[1, 2, 15, 16, 17, 100], [2047, 2048, 2049, 4096, 4097, 9000], [32768, 1, 513]])
def test_decode_rows(cpe, lens):
    """Decode rows (E = 1 at P = L-1) through the split-KV path."""
    b = varlen_batch(40 + len(lens), [(L - 1, 1) for L in lens], 32, 8, 128)
    qo, pl = i32(b["qo"]), i32(b["pl"])
    cpe.cpe_kv_append(b["k_new"], b["v_new"], b["k_cache"], b["v_cache"], b["page_table"], qo, pl)
    lse = torch.empty(len(lens), 32, dtype=torch.float32, device="cuda")
    out, _ = cpe.cpe_decode_attention(b["q"], b["k_cache"], b["v_cache"], b["page_table"], pl, b["max_kv"], lse=lse)
    _status_ok(cpe)
    ref_o, ref_l = _oracle_batch(b)
    check_close(out, ref_o, f"decode {lens}")
    np.testing.assert_allclose(lse.cpu().numpy(), ref_l, atol=LSE_ABS, rtol=0)


def test_mixed_step_small_full(cpe):
    ctx = [1, 37, 2048, 2049, 5000, 300, 16, 999]
    plan = cpe.cpe_plan_mixed_step(8 + 200, ctx, 3000, 500)
    assert plan["n_decode"] == 8 and plan["extend_len"] == 200
    lens = [(p, plan["qo_indptr"][i + 1] - plan["qo_indptr"][i]) for i, p in enumerate(plan["prefix_len"])]
    b = varlen_batch(50, lens, 32, 8, 128)
    lse = torch.empty(b["q"].shape[0], 32, dtype=torch.float32, device="cuda")
    out, _ = cpe.cpe_mixed_step(b["q"], b["k_new"], b["v_new"], b["k_cache"], b["v_cache"], b["page_table"],
                                i32(b["qo"]), i32(b["pl"]), plan["n_decode"], b["max_kv"], lse=lse)
    _status_ok(cpe)
    kc, vc = b["k_cache"].cpu().clone(), b["v_cache"].cpu().clone()
    ref_o, ref_l = oracle.extend_attention(b["q"].cpu(), kc, vc, b["page_table_host"], b["qo"], b["pl"], 32, 8)
    check_close(out, ref_o, "mixed small")
    np.testing.assert_allclose(lse.cpu().numpy(), ref_l, atol=LSE_ABS, rtol=0)


@pytest.mark.parametrize("h_q,h_kv,d", [(8, 1, 64), (32, 2, 128)])
def test_mixed_step_fused_shapes_full(cpe, h_q, h_kv, d):
    """Decode rows (one past a split boundary) and two prefill chunks in one
    fused launch, at d = 64 and G = 16; every row checked."""
    ctx = [3, 2049, 4100, 77]
    plan = cpe.cpe_plan_schedule(4 + 300, [(L - 1, 1) for L in ctx] + [(900, 200)], [(64, 300)])
    lens = [(p, plan["qo_indptr"][i + 1] - plan["qo_indptr"][i]) for i, p in enumerate(plan["prefix_len"])]
    b = varlen_batch(51, lens, h_q, h_kv, d)
    lse = torch.empty(b["q"].shape[0], h_q, dtype=torch.float32, device="cuda")
    out, _ = cpe.cpe_mixed_step(b["q"], b["k_new"], b["v_new"], b["k_cache"], b["v_cache"], b["page_table"],
                                i32(b["qo"]), i32(b["pl"]), plan["n_decode"], b["max_kv"], lse=lse)
    _status_ok(cpe)
    kc, vc = b["k_cache"].cpu().clone(), b["v_cache"].cpu().clone()
    ref_o, ref_l = oracle.extend_attention(b["q"].cpu(), kc, vc, b["page_table_host"], b["qo"], b["pl"], h_q, h_kv)
    check_close(out, ref_o, f"fused mixed {h_q}/{h_kv} d={d}")
    np.testing.assert_allclose(lse.cpu().numpy(), ref_l, atol=LSE_ABS, rtol=0)


def test_mixed_256dec_2048_sampled(cpe):
    spec = W.CONFIGS["mixed-256dec-2048"]
    g = torch.Generator().manual_seed(spec.seed)
    ctx = torch.randint(spec.ctx_lo, spec.ctx_hi + 1, (spec.n_decode,), generator=g).tolist()
    plan = cpe.cpe_plan_mixed_step(spec.token_budget, ctx, spec.prefill_prefix, spec.prefill_remaining)
    assert plan["extend_len"] == 2048 and plan["n_decode"] == 256
    mb = W.make_mixed(spec, plan["extend_len"], device="cuda")
    plan = cpe.cpe_plan_mixed_step(spec.token_budget, mb.ctx_len, spec.prefill_prefix, spec.prefill_remaining)
    max_kv = max(plan["kv_len"])
    lse = torch.empty(mb.q.shape[0], spec.h_q, dtype=torch.float32, device="cuda")
    out, _ = cpe.cpe_mixed_step(mb.q, mb.k_new, mb.v_new, mb.k_cache, mb.v_cache, mb.page_table,
                                i32(plan["qo_indptr"]), i32(plan["prefix_len"]), plan["n_decode"], max_kv, lse=lse)
    _status_ok(cpe)
    # decode rows: the longest, the shortest and a seeded sample
    order = sorted(range(256), key=lambda s: mb.ctx_len[s])
    dec = sorted(set([order[0], order[-1]] + torch.randperm(256, generator=g)[:10].tolist()))
    kl = [plan["kv_len"][s] for s in dec]
    kc, vc, pt = extract_pages(mb.k_cache, mb.v_cache, mb.page_table_host, dec, kl)
    q = mb.q[dec].cpu()
    ref_o, ref_l = oracle.extend_attention(q, kc, vc, pt, list(range(len(dec) + 1)),
                                           [plan["prefix_len"][s] for s in dec], spec.h_q, spec.h_kv)
    check_close(out[dec], ref_o, "mixed-256dec-2048 decode rows")
    np.testing.assert_allclose(lse[dec].cpu().numpy(), ref_l, atol=LSE_ABS, rtol=0)
    # prefill rows
    ps = 256
    kc, vc, pt = extract_pages(mb.k_cache, mb.v_cache, mb.page_table_host, [ps], [plan["kv_len"][ps]])
    rows = W.sample_rows(2048, 32, 64, 404)
    q = mb.q[256:]
    ref_o, ref_l = oracle.extend_attention(q.cpu(), kc, vc, pt, [0, 2048], [plan["prefix_len"][ps]], spec.h_q,
                                           spec.h_kv, rows=rows)
    check_close(out[256:][rows], ref_o, "mixed-256dec-2048 prefill rows")
    np.testing.assert_allclose(lse[256:][rows].cpu().numpy(), ref_l, atol=LSE_ABS, rtol=0)


def test_mixed_256dec_2048_every_decode_row(cpe):
    """The mixed step as the benchmark runs it, all 256 decode rows (all heads,
    all keys) against the float64 oracle on the whole page pool."""
    spec = W.CONFIGS["mixed-256dec-2048"]
    g = torch.Generator().manual_seed(spec.seed)
    ctx = torch.randint(spec.ctx_lo, spec.ctx_hi + 1, (spec.n_decode,), generator=g).tolist()
    plan = cpe.cpe_plan_mixed_step(spec.token_budget, ctx, spec.prefill_prefix, spec.prefill_remaining)
    mb = W.make_mixed(spec, plan["extend_len"], device="cuda")
    plan = cpe.cpe_plan_mixed_step(spec.token_budget, mb.ctx_len, spec.prefill_prefix, spec.prefill_remaining)
    nd = plan["n_decode"]
    assert nd == 256
    ws = cpe.alloc_workspace(nd + 1, mb.q.shape[0], spec.h_q, spec.h_kv, spec.d, max(plan["kv_len"]), "cuda")
    lse = torch.empty(mb.q.shape[0], spec.h_q, dtype=torch.float32, device="cuda")
    out, _ = cpe.cpe_mixed_step(mb.q, mb.k_new, mb.v_new, mb.k_cache, mb.v_cache, mb.page_table,
                                i32(plan["qo_indptr"]), i32(plan["prefix_len"]), nd, max(plan["kv_len"]), lse=lse,
                                workspace=ws)
    _status_ok(cpe)
    ref_o, ref_l = oracle.extend_attention(mb.q[:nd].cpu(), mb.k_cache.cpu(), mb.v_cache.cpu(),
                                           mb.page_table_host[:nd], list(range(nd + 1)), plan["prefix_len"][:nd],
                                           spec.h_q, spec.h_kv)
    check_close(out[:nd], ref_o, "mixed-256dec-2048 all decode rows")
    np.testing.assert_allclose(lse[:nd].cpu().numpy(), ref_l, atol=LSE_ABS, rtol=0)


def _scheduled_step(cpe, seed, budget, running, waiting):
    """One step laid out by the scheduling planner and run through cpe_mixed_step."""
    plan = cpe.cpe_plan_schedule(budget, running, waiting)
    lens = [(p, plan["qo_indptr"][i + 1] - plan["qo_indptr"][i]) for i, p in enumerate(plan["prefix_len"])]
    b = varlen_batch(seed, lens, 32, 8, 128)
    lse = torch.empty(b["q"].shape[0], 32, dtype=torch.float32, device="cuda")
    out, _ = cpe.cpe_mixed_step(b["q"], b["k_new"], b["v_new"], b["k_cache"], b["v_cache"], b["page_table"],
                                i32(b["qo"]), i32(b["pl"]), plan["n_decode"], b["max_kv"], lse=lse)
    _status_ok(cpe)
    return plan, b, out, lse


def test_scheduled_step_several_prefills_full(cpe):
    """Decode rows, a running prefill continuation and a waiting request with a
    prefix-cache hit cut to its first chunk, in one step; every row checked."""
    running = [(37, 1), (2048, 1), (5, 1), (999, 1), (900, 300), (0, 1)]
    waiting = [(200, 500), (0, 64)]
    plan, b, out, lse = _scheduled_step(cpe, 70, 512, running, waiting)
    assert plan["granted"] == [1, 1, 1, 1, 300, 1, 207, 0] and plan["n_decode"] == 5
    kc, vc = b["k_cache"].cpu().clone(), b["v_cache"].cpu().clone()
    ref_o, ref_l = oracle.extend_attention(b["q"].cpu(), kc, vc, b["page_table_host"], b["qo"], b["pl"], 32, 8)
    check_close(out, ref_o, "scheduled step")
    np.testing.assert_allclose(lse.cpu().numpy(), ref_l, atol=LSE_ABS, rtol=0)


def test_scheduled_step_pages_example_sampled(cpe):
    """The vLLM tutorial's step at its own sizes: 8 decodes, R's remaining 1440
    tokens, W1 cut to 600 (GQA 32/8, d=128); decode rows in full, chunk rows
    sampled."""
    running = [(600 + 97 * k, 1) for k in range(8)] + [(3000, 1440)]
    waiting = [(0, 900), (0, 700)]
    plan, b, out, lse = _scheduled_step(cpe, 71, 2048, running, waiting)
    assert plan["granted"][8:] == [1440, 600, 0] and plan["qo_indptr"][-1] == 2048
    qo = plan["qo_indptr"]
    for s in range(len(plan["prefix_len"])):
        E = qo[s + 1] - qo[s]
        rows = list(range(E)) if E <= 8 else W.sample_rows(E, 32, 48, 500 + s)
        kc, vc, pt = extract_pages(b["k_cache"], b["v_cache"], b["page_table_host"], [s], [plan["kv_len"][s]])
        q = b["q"][qo[s]:qo[s + 1]].cpu()
        ref_o, ref_l = oracle.extend_attention(q, kc, vc, pt, [0, E], [plan["prefix_len"][s]], 32, 8, rows=rows)
        check_close(out[qo[s]:qo[s + 1]][rows], ref_o, f"sequence {s}")
        np.testing.assert_allclose(lse[qo[s]:qo[s + 1]][rows].cpu().numpy(), ref_l, atol=LSE_ABS, rtol=0)


def test_sched_workload_sampled(cpe):
    """The scheduled-step bench workload at full size, as the bench runs it:
    decode rows (shortest, longest, a seeded sample) and sampled rows of each
    prefill chunk, whose units the scheduler cuts into unequal part counts."""
    spec = W.CONFIGS["sched"]
    running, waiting = W.scheduled_requests(spec)
    plan = cpe.cpe_plan_schedule(spec.token_budget, running, waiting)
    assert plan == oracle.plan_schedule(spec.token_budget, running, waiting)
    qo = plan["qo_indptr"]
    lens = [(p, qo[i + 1] - qo[i]) for i, p in enumerate(plan["prefix_len"])]
    mb = W.make_scheduled(spec, lens, device="cuda")
    nd = plan["n_decode"]
    lse = torch.empty(mb.q.shape[0], spec.h_q, dtype=torch.float32, device="cuda")
    out, _ = cpe.cpe_mixed_step(mb.q, mb.k_new, mb.v_new, mb.k_cache, mb.v_cache, mb.page_table, i32(qo),
                                i32(plan["prefix_len"]), nd, max(plan["kv_len"]), lse=lse)
    _status_ok(cpe)
    g = torch.Generator().manual_seed(606)
    order = sorted(range(nd), key=lambda s: plan["kv_len"][s])
    seqs = sorted(set([order[0], order[-1]] + torch.randperm(nd, generator=g)[:4].tolist())) + list(range(nd, len(lens)))
    for s in seqs:
        E = qo[s + 1] - qo[s]
        rows = [0] if E == 1 else W.sample_rows(E, 32, 40, 700 + s)
        kc, vc, pt = extract_pages(mb.k_cache, mb.v_cache, mb.page_table_host, [s], [plan["kv_len"][s]])
        q = mb.q[qo[s]:qo[s + 1]].cpu()
        ref_o, ref_l = oracle.extend_attention(q, kc, vc, pt, [0, E], [plan["prefix_len"][s]], spec.h_q, spec.h_kv,
                                               rows=rows)
        check_close(out[qo[s]:qo[s + 1]][rows], ref_o, f"sched sequence {s}")
        np.testing.assert_allclose(lse[qo[s]:qo[s + 1]][rows].cpu().numpy(), ref_l, atol=LSE_ABS, rtol=0)


# ---------------------------------------------------------------- device-side errors

def test_bad_page_id_is_reported(cpe):
    b = varlen_batch(60, [(40, 30)], 32, 8, 128)
    b["page_table"][0, 1] = 10 ** 6  # out of range
    qo, pl = i32(b["qo"]), i32(b["pl"])
    cpe.cpe_extend_attention(b["q"], b["k_cache"], b["v_cache"], b["page_table"], qo, pl, b["max_kv"])
    st, _ = cpe.cpe_get_device_status()
    assert st == cpe.CPE_ERR_DEVICE_ARG
    _status_ok(cpe)  # cleared by the read


def test_wait_timeout_path_returns_status(cpe):
    """With a zero wait limit every pipeline wait that is not already
    satisfied gives up: the kernel records a timeout and returns, and the
    context stays usable."""
    b = varlen_batch(61, [(1000, 300)], 32, 8, 128)
    qo, pl = i32(b["qo"]), i32(b["pl"])
    old = cpe.cpe_set_wait_limit_ns(0)
    try:
        cpe.cpe_extend_attention(b["q"], b["k_cache"], b["v_cache"], b["page_table"], qo, pl, b["max_kv"])
        st, _ = cpe.cpe_get_device_status()
    finally:
        cpe.cpe_set_wait_limit_ns(old)
    assert st == cpe.CPE_ERR_TIMEOUT
    out, _ = _append_and_attend(cpe, b)
    ref_o, _ = _oracle_batch(b)
    check_close(out, ref_o, "after timeout")
