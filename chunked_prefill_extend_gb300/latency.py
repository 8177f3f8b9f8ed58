"""Forward-shape latency table measured with this library's kernels, and the
three-phase replay of the request time simulation.

msmodeling forward-latency-table RFC (the chunked-prefill table section):
ForwardShapeKey (is_decode, model_concurrency, query_len, seq_len) names one
forward shape; ForwardLatencyTable computes each unique key once, in order,
and stops at the first key that does not fit in memory; for mixed
prefill/decode steps the schedule is first run dry (the scheduler's decisions
do not depend on latency) to collect the keys, the unique keys are prefetched,
and the schedule is replayed from the table, with results identical to calling
the latency model at every step.

Here a key's latency is the attention-layer cost of that shape on this GPU:
the step's K/V append plus the extend attention (prefill) or the split-KV
decode attention (decode), timed with CUDA events on synthetic bf16 inputs.
Decode keys carry their mean context rounded up to the decode split length
(2048 keys), the granularity at which the decode kernel's work changes;
prefill keys carry the chunk's exact lengths.
"""
from __future__ import annotations

import statistics
from dataclasses import dataclass

import torch

from . import cpe

DECODE_BUCKET = 2048


@dataclass(frozen=True)
class ForwardShapeKey:
    is_decode: bool
    model_concurrency: int
    query_len: int
    seq_len: int


@dataclass
class ForwardLatencyRecord:
    latency_ms: float
    bytes_needed: int   # device memory the measured inputs took
    launches: int       # library kernels per call of the shape


class KernelLatencyTable:
    """One record per unique shape, measured on first need (or by prefetch)."""

    def __init__(self, h_q: int, h_kv: int, d: int, device="cuda", reps: int = 5, warmup: int = 2,
                 decode_bucket: int = DECODE_BUCKET, decode_pool_bytes: int = 2 << 30, seed: int = 0,
                 memory_reserve_bytes: int = 1 << 30):
        self.h_q, self.h_kv, self.d = h_q, h_kv, d
        self.device = torch.device(device)
        self.reps, self.warmup = reps, warmup
        self.decode_bucket = decode_bucket
        self.decode_pool_bytes = decode_pool_bytes
        self.seed = seed
        self.memory_reserve_bytes = memory_reserve_bytes
        self.records: dict[ForwardShapeKey, ForwardLatencyRecord] = {}
        self.memory_exceeded_key: ForwardShapeKey | None = None
        self.measured = 0

    # ------------------------------------------------------------------ keys
    def key(self, is_decode: bool, batch: int, query_len: int, seq_len: int) -> ForwardShapeKey:
        if is_decode:
            b = self.decode_bucket
            return ForwardShapeKey(True, batch, 1, -(-seq_len // b) * b)
        return ForwardShapeKey(False, batch, query_len, seq_len)

    def bytes_needed(self, k: ForwardShapeKey) -> int:
        kv_tok = self.h_kv * self.d * 2 * 2  # K and V, bf16
        if k.is_decode:
            pages = min(k.model_concurrency * -(-k.seq_len // 16), max(1, self.decode_pool_bytes // (16 * kv_tok)))
        else:
            pages = k.model_concurrency * -(-k.seq_len // 16)
        rows = k.model_concurrency * k.query_len
        return pages * 16 * kv_tok + rows * (2 * self.h_q + 2 * self.h_kv) * self.d * 2

    # ------------------------------------------------------------------ table
    def prefetch(self, keys) -> None:
        """Measure the keys not yet in the table, in order, each once; stop at
        the first one that would not fit in free device memory."""
        seen = set()
        for k in keys:
            if k in seen or k in self.records:
                continue
            seen.add(k)
            if self.bytes_needed(k) + self.memory_reserve_bytes > self.free_bytes():
                self.memory_exceeded_key = k
                break
            self.records[k] = self._measure(k)

    def get(self, k: ForwardShapeKey) -> ForwardLatencyRecord:
        if k not in self.records:
            self.prefetch([k])
        if k not in self.records:
            raise RuntimeError(f"shape {k} does not fit in device memory")
        return self.records[k]

    def __call__(self, is_decode: bool, batch: int, query_len: int, seq_len: int) -> float:
        return self.get(self.key(is_decode, batch, query_len, seq_len)).latency_ms

    # ------------------------------------------------------------------ measurement
    def free_bytes(self) -> int:
        return torch.cuda.mem_get_info(self.device)[0]

    def _measure(self, k: ForwardShapeKey) -> ForwardLatencyRecord:
        dev = self.device
        g = torch.Generator(device=dev)
        g.manual_seed((self.seed + k.model_concurrency * 1000003 + k.query_len * 10007 + k.seq_len * 2 +
                       int(k.is_decode)) & 0x7FFFFFFF)
        B, E, L = k.model_concurrency, k.query_len, k.seq_len
        P = L - E
        per_seq = -(-L // 16)
        kv_tok = self.h_kv * self.d * 2 * 2
        if k.is_decode:
            pool = min(B * per_seq, max(per_seq, self.decode_pool_bytes // (16 * kv_tok)))
            pt = torch.randint(0, pool, (B, per_seq), generator=g, device=dev, dtype=torch.int32)
        else:
            pool = B * per_seq
            pt = torch.randperm(pool, generator=g, device=dev).to(torch.int32).view(B, per_seq)
        bf = torch.bfloat16
        kc = torch.randn(pool, 16, self.h_kv, self.d, generator=g, device=dev, dtype=bf)
        vc = torch.randn(pool, 16, self.h_kv, self.d, generator=g, device=dev, dtype=bf)
        q = torch.randn(B * E, self.h_q, self.d, generator=g, device=dev, dtype=bf)
        kn = torch.randn(B * E, self.h_kv, self.d, generator=g, device=dev, dtype=bf)
        vn = torch.randn(B * E, self.h_kv, self.d, generator=g, device=dev, dtype=bf)
        qo = torch.arange(0, B * E + 1, E, dtype=torch.int32, device=dev)
        pl = torch.full((B,), P, dtype=torch.int32, device=dev)
        out = torch.empty_like(q)
        ws = cpe.alloc_workspace(B, B * E, self.h_q, self.h_kv, self.d, L, dev)

        def call():
            cpe.cpe_kv_append(kn, vn, kc, vc, pt, qo, pl)
            if k.is_decode:
                cpe.cpe_decode_attention(q, kc, vc, pt, pl, L, out=out, workspace=ws)
            else:
                cpe.cpe_extend_attention(q, kc, vc, pt, qo, pl, L, out=out, workspace=ws)

        for _ in range(self.warmup):
            call()
        n0 = cpe.cpe_launch_count()
        times = []
        for _ in range(self.reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            call()
            b.record()
            times.append((a, b))
        torch.cuda.synchronize(dev)
        st, detail = cpe.cpe_get_device_status()
        if st != cpe.CPE_OK:
            raise RuntimeError(f"device status {cpe.cpe_status_string(st)} ({detail}) measuring {k}")
        launches = (cpe.cpe_launch_count() - n0) // self.reps
        ms = statistics.median(x.elapsed_time(y) for x, y in times)
        self.measured += 1
        return ForwardLatencyRecord(ms, self.bytes_needed(k), launches)


def simulate_with_table(table: KernelLatencyTable, chunks, n_requests: int, output_len: int,
                        max_batched_tokens: int, scheduler=None) -> dict:
    """Dry run (keys only), prefetch of the unique keys, replay from the table."""
    keys = []

    def record(is_decode, batch, query_len, seq_len):
        keys.append(table.key(is_decode, batch, query_len, seq_len))
        return 0.0
    cpe.cpe_simulate_requests(chunks, n_requests, output_len, max_batched_tokens, record, scheduler)
    table.prefetch(keys)
    if table.memory_exceeded_key is not None:
        raise RuntimeError(f"shape {table.memory_exceeded_key} does not fit in device memory")
    out = cpe.cpe_simulate_requests(chunks, n_requests, output_len, max_batched_tokens,
                                    lambda *a: table.get(table.key(*a)).latency_ms, scheduler)
    out["forward_shapes"] = len(set(keys))
    out["forward_calls"] = len(keys)
    return out
