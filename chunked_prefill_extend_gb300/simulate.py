"""TTFT, TPOT and throughput of N concurrent requests under chunked prefill,
simulated with attention latencies measured on this GPU.

    python -m chunked_prefill_extend_gb300.simulate --input-len 32768 --chunk 4096 \\
        --output-len 256 --concurrency 16

The request's chunk plan comes from cpe_plan_chunks; the step schedule from
the decode-first scheduler with 15 % slack (cpe_simulate_requests); each unique
forward shape is measured once with this library's kernels (latency.py) and the
schedule is replayed from those records.  The latencies are the attention layer
alone (K/V append plus attention), not a full model forward.
"""
from __future__ import annotations

import argparse
import json
import time

import torch

from . import cpe
from .latency import KernelLatencyTable, simulate_with_table


def main(argv=None) -> dict:
    ap = argparse.ArgumentParser()
    ap.add_argument("--input-len", type=int, default=32768)
    ap.add_argument("--hit-rate", type=float, default=0.0, help="prefix-cache hit rate of the prompt")
    ap.add_argument("--chunk", type=int, default=4096, help="max_batched_tokens (chunk size and step budget)")
    ap.add_argument("--output-len", type=int, default=256)
    ap.add_argument("--concurrency", type=int, default=16)
    ap.add_argument("--h-q", type=int, default=32)
    ap.add_argument("--h-kv", type=int, default=8)
    ap.add_argument("--d", type=int, default=128)
    ap.add_argument("--reps", type=int, default=5)
    args = ap.parse_args(argv)
    if not torch.cuda.is_available():
        raise SystemExit("a CUDA device is required to measure the kernels")
    chunks, cached, effective = cpe.cpe_plan_chunks(args.input_len, args.hit_rate, args.chunk)
    plan = [(c.query_len, c.seq_len) for c in chunks]
    table = KernelLatencyTable(args.h_q, args.h_kv, args.d, reps=args.reps)
    t0 = time.perf_counter()
    res = simulate_with_table(table, plan, args.concurrency, args.output_len, args.chunk)
    line = {"input_len": args.input_len, "cached_prefix": cached, "effective_input_length": effective,
            "max_batched_tokens": args.chunk, "prefill_num_chunks": len(plan), "output_len": args.output_len,
            "concurrency": args.concurrency, "heads": f"{args.h_q}/{args.h_kv}", "d": args.d,
            "ttft_ms": res["ttft"], "tpot_ms": res["tpot"], "makespan_ms": res["makespan"],
            "request_throughput": res["request_throughput"], "output_throughput": res["output_throughput"],
            "steps": res["steps"], "forward_shapes": res["forward_shapes"], "forward_calls": res["forward_calls"],
            "measured_shapes": table.measured, "measure_seconds": time.perf_counter() - t0,
            "latency": "attention layer only (K/V append + attention), measured on this GPU"}
    print(json.dumps(line), flush=True)
    return line


if __name__ == "__main__":
    main()
