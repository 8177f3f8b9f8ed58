"""Seeded synthetic inputs for chunked-prefill extend attention.

This module draws random tensors and lays out pages; it holds none of the
method's arithmetic (no planning, no attention) and is the one piece shared by
the oracle tests and the CUDA tests / benchmark.  Every tensor is drawn from a
``torch.Generator`` seeded per workload, on the device the caller names, in a
fixed order of draws.

Workloads (shapes of the pages' long-context chunked prefill):

``fp32-512``  one request N=512, chunk 128, 4/4 heads, d=64, fp32 N(0,1), contiguous cache
``prefill-4000-c512``  one request N=4000, chunk 512, 32/8 heads, d=128, bf16 N(0,1)*0.5, page 16
``prefill-32k-hit50``  input 32768 with 50% prefix-cache hit: 16384 cached tokens N(0,1), two
          extend rounds of 8192, 32/8, d=128, bf16 N(0,1)*0.5 for the extend part
``mixed-256dec-2048``  mixed step, budget 2304: one prefill chunk at prefix 30720 plus 256
          decode rows with context lengths uniform on {512..32768}, 32/8, d=128,
          bf16 N(0,1)*0.5, all pages drawn from one pool in a random permutation
``prefill-128k-c1024``  one request N=131072, chunk 1024 (128 rounds), 64/8, d=128, bf16 N(0,1)*0.5
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch

PAGE_SIZE = 16


@dataclass(frozen=True)
class ChunkedSpec:
    name: str
    seed: int
    input_len: int
    hit_rate: float
    chunk: int
    h_q: int
    h_kv: int
    d: int
    dtype: torch.dtype
    std: float = 0.5            # extend-part Q/K/V
    prefix_std: float = 0.5     # pre-filled (cached) prefix K/V
    page_perm: bool = False     # random page permutation instead of sequential pages
    page_size: int = PAGE_SIZE


@dataclass(frozen=True)
class MixedSpec:
    name: str
    seed: int
    token_budget: int
    n_decode: int
    ctx_lo: int
    ctx_hi: int
    prefill_prefix: int
    prefill_remaining: int
    h_q: int
    h_kv: int
    d: int
    dtype: torch.dtype
    std: float = 0.5
    page_size: int = PAGE_SIZE


@dataclass(frozen=True)
class ScheduledSpec:
    """One scheduling step over running and waiting requests under one budget:
    ``n_decode`` decode requests (context L ~ U[ctx_lo, ctx_hi], seeded), then
    the running prefill continuations ``running_prefill`` = ((computed, need),
    ...), then the waiting queue ``waiting`` = ((cached, prompt), ...)."""
    name: str
    seed: int
    token_budget: int
    n_decode: int
    ctx_lo: int
    ctx_hi: int
    running_prefill: tuple
    waiting: tuple
    h_q: int
    h_kv: int
    d: int
    dtype: torch.dtype
    std: float = 0.5
    page_size: int = PAGE_SIZE


CONFIGS = {
    "fp32-512": ChunkedSpec("fp32-512", 1, 512, 0.0, 128, 4, 4, 64, torch.float32, std=1.0, prefix_std=1.0),
    "prefill-4000-c512": ChunkedSpec("prefill-4000-c512", 2, 4000, 0.0, 512, 32, 8, 128, torch.bfloat16),
    "prefill-32k-hit50": ChunkedSpec("prefill-32k-hit50", 3, 32768, 0.5, 8192, 32, 8, 128, torch.bfloat16, prefix_std=1.0),
    "mixed-256dec-2048": MixedSpec("mixed-256dec-2048", 4, 2304, 256, 512, 32768, 30720, 4096, 32, 8, 128, torch.bfloat16),
    "prefill-128k-c1024": ChunkedSpec("prefill-128k-c1024", 5, 131072, 0.0, 1024, 64, 8, 128, torch.bfloat16),
    "sched": ScheduledSpec("sched", 6, 8192, 64, 512, 32768, ((8192, 2048), (30720, 2048), (65536, 2048)),
                           ((4096, 16384), (0, 4000)), 32, 8, 128, torch.bfloat16),
}

WORKLOAD_TEXT = {
    "fp32-512": "one request N=512, chunk 128, 4/4 heads, d=64, fp32, contiguous cache",
    "prefill-4000-c512": "one request N=4000, chunk 512 (7x512+416), GQA 32/8, d=128, bf16, page 16",
    "prefill-32k-hit50": "input 32768, 50% prefix hit (16384 cached), 2 chunks of 8192, GQA 32/8, d=128, bf16",
    "mixed-256dec-2048": "mixed step budget 2304: prefill E=2048 at P=30720 + 256 decode rows L~U[512,32768], "
            "GQA 32/8, d=128, bf16, permuted pages",
    "prefill-128k-c1024": "one request N=131072, chunk 1024 (128 chunks), GQA 64/8, d=128, bf16, page 16",
    "sched": "one scheduling step, budget 8192: 64 decode rows L~U[512,32768], running prefills at "
             "P=8192/30720/65536 (2048 tokens each), waiting prompts 16384 (4096 cached, cut to 1984) and 4000 "
             "(left queued); GQA 32/8, d=128, bf16, permuted pages",
}


def _randn(gen: torch.Generator, shape, std: float, dtype: torch.dtype, device) -> torch.Tensor:
    """N(0,1)*std drawn in float32 slices of <=64M elements, then cast."""
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    step = 1 << 26
    for i in range(0, flat.numel(), step):
        n = min(step, flat.numel() - i)
        x = torch.randn(n, generator=gen, dtype=torch.float32, device=device)
        if std != 1.0:
            x.mul_(std)
        flat[i:i + n].copy_(x)
    return out


def _pages(n: int, page_size: int) -> int:
    return (n + page_size - 1) // page_size


@dataclass
class ChunkedRequest:
    """One request's tensors for a chunked prefill.

    Q/K/V rows for positions [cached, input_len) are held in ``q``, ``k``,
    ``v`` (row = position - cached); positions [0, cached) exist only in the
    caches.  ``page_table`` is [1, max_pages] int32 on the device.
    """
    spec: ChunkedSpec
    cached: int
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    page_table: torch.Tensor
    page_table_host: list = field(default_factory=list)

    def round_inputs(self, prefix_len: int, query_len: int):
        """Q and new K/V of the round whose rows are positions [prefix_len, prefix_len+query_len)."""
        a = prefix_len - self.cached
        return self.q[a:a + query_len], self.k[a:a + query_len], self.v[a:a + query_len]


def make_chunked(spec: ChunkedSpec, cached: int, device="cpu", prefill_cache: bool = True) -> ChunkedRequest:
    """Draw the request: pre-filled prefix K/V, extend-part Q/K/V, pages.

    ``cached`` is the prefix-cache hit the caller's chunk plan reports (the
    first chunk's prefix length); those tokens' K/V are written straight into
    their pages here, the way an earlier request would have left them, and are
    not kept elsewhere.
    """
    if not 0 <= cached < spec.input_len:
        raise ValueError("cached must be in [0, input_len)")
    gen = torch.Generator(device=device)
    gen.manual_seed(spec.seed)
    n_new = spec.input_len - cached
    num_pages = _pages(spec.input_len, spec.page_size)
    if spec.page_perm:
        perm = torch.randperm(num_pages, generator=gen, device=device).to(torch.int32)
    else:
        perm = torch.arange(num_pages, dtype=torch.int32, device=device)
    shape_c = (num_pages, spec.page_size, spec.h_kv, spec.d)
    k_cache = torch.zeros(shape_c, dtype=spec.dtype, device=device)
    v_cache = torch.zeros(shape_c, dtype=spec.dtype, device=device)
    if cached > 0 and prefill_cache:
        kp = _randn(gen, (cached, spec.h_kv, spec.d), spec.prefix_std, spec.dtype, device)
        vp = _randn(gen, (cached, spec.h_kv, spec.d), spec.prefix_std, spec.dtype, device)
        pos = torch.arange(cached, device=device)
        slot = perm.long()[pos // spec.page_size] * spec.page_size + pos % spec.page_size
        k_cache.view(-1, spec.h_kv, spec.d)[slot] = kp
        v_cache.view(-1, spec.h_kv, spec.d)[slot] = vp
        del kp, vp
    q = _randn(gen, (n_new, spec.h_q, spec.d), spec.std, spec.dtype, device)
    k = _randn(gen, (n_new, spec.h_kv, spec.d), spec.std, spec.dtype, device)
    v = _randn(gen, (n_new, spec.h_kv, spec.d), spec.std, spec.dtype, device)
    pt = perm.view(1, -1).contiguous()
    return ChunkedRequest(spec, cached, q, k, v, k_cache, v_cache, pt, perm.cpu().tolist())


@dataclass
class MixedBatch:
    """One mixed step: decode rows first, then one prefill sequence.

    ``ctx_len`` are the decode rows' context lengths L (the token appended this
    step included).  ``q``/``k_new``/``v_new`` hold, in batch row order, one
    row per decode sequence followed by the prefill chunk's rows; the batch
    layout itself (qo_indptr etc.) comes from the planner.
    """
    spec: MixedSpec
    ctx_len: list
    q: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    page_table: torch.Tensor        # [n_decode + 1, max_pages] int32 on the device, -1 padded
    page_table_host: torch.Tensor   # same, CPU


def make_mixed(spec: MixedSpec, extend_len: int, device="cpu") -> MixedBatch:
    """Draw the mixed step.  ``extend_len`` is the prefill chunk length the
    planner granted (it sizes Q/K/V for the chunk and the prefill's pages).

    Every page of the shared pool is filled with N(0,1)*std, so each decode
    row's first L-1 positions and the prefill's first P positions read as a
    pre-filled cache; the rows appended this step overwrite their slots.
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(spec.seed)
    ctx = torch.randint(spec.ctx_lo, spec.ctx_hi + 1, (spec.n_decode,), generator=gen,
                        device=device).cpu().tolist()
    lens = ctx + [spec.prefill_prefix + extend_len]
    npages = [_pages(L, spec.page_size) for L in lens]
    total_pages = sum(npages)
    perm = torch.randperm(total_pages, generator=gen, device=device).to(torch.int32).cpu()
    max_pages = max(npages)
    pt = torch.full((len(lens), max_pages), -1, dtype=torch.int32)
    off = 0
    for s, n in enumerate(npages):
        pt[s, :n] = perm[off:off + n]
        off += n
    shape_c = (total_pages, spec.page_size, spec.h_kv, spec.d)
    k_cache = _randn(gen, shape_c, spec.std, spec.dtype, device)
    v_cache = _randn(gen, shape_c, spec.std, spec.dtype, device)
    rows = spec.n_decode + extend_len
    q = _randn(gen, (rows, spec.h_q, spec.d), spec.std, spec.dtype, device)
    k_new = _randn(gen, (rows, spec.h_kv, spec.d), spec.std, spec.dtype, device)
    v_new = _randn(gen, (rows, spec.h_kv, spec.d), spec.std, spec.dtype, device)
    return MixedBatch(spec, ctx, q, k_new, v_new, k_cache, v_cache, pt.to(device), pt)


def shrink(spec, **kw):
    """A copy of a workload spec with some fields replaced (smaller test cases)."""
    return replace(spec, **kw)


def sample_rows(n_rows: int, tile_rows: int, count: int, seed: int) -> list:
    """Seeded sample of query rows: first, last, both sides of every tile
    boundary that fits, then uniform picks, up to ``count`` distinct rows."""
    picks = {0, n_rows - 1}
    b = tile_rows
    while b < n_rows and len(picks) < count // 2:
        picks.update({b - 1, b})
        b += tile_rows
    g = torch.Generator().manual_seed(seed)
    extra = torch.randint(0, n_rows, (count,), generator=g).tolist()
    for r in extra:
        if len(picks) >= count:
            break
        picks.add(r)
    return sorted(x for x in picks if 0 <= x < n_rows)


def scheduled_requests(spec: ScheduledSpec) -> tuple[list, list]:
    """The step's queues: running = decode requests (L-1 cached, 1 needed) then
    the running prefill continuations; waiting = (cached, prompt) per request."""
    g = torch.Generator().manual_seed(spec.seed)
    ctx = torch.randint(spec.ctx_lo, spec.ctx_hi + 1, (spec.n_decode,), generator=g).tolist()
    running = [(L - 1, 1) for L in ctx] + [tuple(x) for x in spec.running_prefill]
    return running, [tuple(x) for x in spec.waiting]


@dataclass
class ScheduledBatch:
    """Inputs of one scheduled step for a given batch layout ``lens`` =
    [(prefix_len, query_len)] per sequence in batch order: a shared page pool
    (seeded permutation, every page filled with N(0,1)*std, so each sequence's
    first prefix_len slots read as its cached K/V), and q/k_new/v_new rows in
    batch row order."""
    lens: list
    q: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    page_table: torch.Tensor
    page_table_host: torch.Tensor


def make_scheduled(spec: ScheduledSpec, lens: list, device="cpu") -> ScheduledBatch:
    gen = torch.Generator(device=device)
    gen.manual_seed(spec.seed + 1000)
    npages = [_pages(P + E, spec.page_size) for P, E in lens]
    total_pages = sum(npages)
    perm = torch.randperm(total_pages, generator=gen, device=device).to(torch.int32).cpu()
    pt = torch.full((len(lens), max(npages)), -1, dtype=torch.int32)
    off = 0
    for s, n in enumerate(npages):
        pt[s, :n] = perm[off:off + n]
        off += n
    shape_c = (total_pages, spec.page_size, spec.h_kv, spec.d)
    k_cache = _randn(gen, shape_c, spec.std, spec.dtype, device)
    v_cache = _randn(gen, shape_c, spec.std, spec.dtype, device)
    rows = sum(E for _, E in lens)
    q = _randn(gen, (rows, spec.h_q, spec.d), spec.std, spec.dtype, device)
    k_new = _randn(gen, (rows, spec.h_kv, spec.d), spec.std, spec.dtype, device)
    v_new = _randn(gen, (rows, spec.h_kv, spec.d), spec.std, spec.dtype, device)
    return ScheduledBatch(list(lens), q, k_new, v_new, k_cache, v_cache, pt.to(device), pt)
