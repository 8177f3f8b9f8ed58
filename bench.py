#!/usr/bin/env python3
"""Benchmark of chunked-prefill extend attention on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload prefill-128k-c1024] [--impl ours|reference]

A step is one pass of the hot path over one batch of synthetic input:
  fp32-512, prefill-*   the whole chunked prefill of one request: the chunk plan, then
              for every chunk the KV append and the extend attention;
  mixed-256dec-2048     one mixed step: the mixed-step plan, the KV append, the
              split-KV decode rows and the prefill chunk.
Default workload: prefill-128k-c1024 (N=131072, C=1024, 128 chunks, GQA 64/8, d=128, bf16),
the long-context configuration whose per-chunk TFLOP/s the metric tracks.

Rank 0 prints one JSON line.  ``value`` is algorithmic TFLOP/s over all ranks
(4*d*H_q*(E*P + E(E+1)/2) per chunk, plus 4*d*H_q*L per decode row);
``roofline`` describes the dominant kernel; ``cpu_baseline`` times the float64
oracle on a bounded sample; ``e2e`` repeats the measurement with host inputs
and outputs copied inside the timed region.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
# The fp32 path's roofline: FP32 FMA lanes per SM and the maximum SM clock of
# a GB300 (the peak is SMs x lanes x 2 flop x clock)
FP32_LANES_PER_SM = 128
FP32_PEAK_CLOCK_MHZ = 2070
sys.path.insert(0, ROOT)

from chunked_prefill_extend_gb300 import workloads as W  # noqa: E402

L2_BYTES = 129 * 1024 * 1024


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16": p["bf16_tflops"], "bf16_sustained": p["bf16_tflops_sustained"],
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


def code_hash(path):
    """sha256 (first 16 hex digits) of a source file's code: // comments,
    trailing blanks and empty lines removed, so a comment edit keeps it."""
    import hashlib
    import re
    lines = []
    for line in open(path, encoding="utf-8").read().splitlines():
        line = re.sub(r"//.*$", "", line).rstrip()
        if line:
            lines.append(line)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()[:16]


def profiled_traffic(per_launch_flops):
    """DRAM bytes per extend launch from the committed ncu summary, scaled from
    the captured launch to this one by algorithmic work; None when the kernel
    code changed since the capture (the counters no longer describe it)."""
    import re
    try:
        h = code_hash(os.path.join(ROOT, "chunked_prefill_extend_gb300", "csrc", "extend_tc.cu"))
        text = open(os.path.join(ROOT, "profiles", "extend_tc_kernel_prefill-128k-c1024.md")).read()
    except OSError:
        return None
    m = re.search(r"traffic-bytes-per-launch: (\d+) \| captured-launch-flops: (\d+) \| "
                  r"extend_tc.cu-code-sha256-16: ([0-9a-f]+)", text)
    if not m or h != m.group(3):
        return None
    return float(m.group(1)) * per_launch_flops / float(m.group(2))


def chunk_flops(d, h_q, P, E):
    return 4.0 * d * h_q * (E * P + E * (E + 1) / 2.0)


# --------------------------------------------------------------------------- workloads

class Chunked:
    """Whole chunked prefill of one request."""

    def __init__(self, spec, device, cpe, rounds=None):
        self.spec, self.cpe, self.device = spec, cpe, device
        self.chunks, self.cached, _ = cpe.cpe_plan_chunks(spec.input_len, spec.hit_rate, spec.chunk)
        self.req = W.make_chunked(spec, self.cached, device=device)
        self.rounds = rounds or (0, len(self.chunks))
        if self.rounds[0] > 0:  # the cache must hold every earlier round's keys
            for c in self.chunks[:self.rounds[0]]:
                a = c.prefix_len - self.cached
                cpe.cpe_kv_append(self.req.k[a:a + c.query_len], self.req.v[a:a + c.query_len], self.req.k_cache,
                                  self.req.v_cache, self.req.page_table,
                                  torch.tensor([0, c.query_len], dtype=torch.int32, device=device),
                                  torch.tensor([c.prefix_len], dtype=torch.int32, device=device))
        self.chunks = self.chunks[self.rounds[0]:self.rounds[1]]
        self.idx = {c.index: (torch.tensor([0, c.query_len], dtype=torch.int32, device=device),
                              torch.tensor([c.prefix_len], dtype=torch.int32, device=device)) for c in self.chunks}
        self.out = torch.empty_like(self.req.q)
        # two workspaces, alternated between rounds: a round's tile list is
        # built while the previous round finishes
        self.wss = [cpe.alloc_workspace(1, spec.chunk, spec.h_q, spec.h_kv, spec.d, spec.input_len, device)
                    for _ in range(2)]
        self.ws = self.wss[0]
        self.views = {}
        self.flops = sum(chunk_flops(spec.d, spec.h_q, c.prefix_len, c.query_len) for c in self.chunks)
        self.tokens = sum(c.query_len for c in self.chunks)
        self.in_bytes = sum(t.numel() * t.element_size() for t in (self.req.q, self.req.k, self.req.v))
        self.kernel = "extend_tc_kernel" if spec.dtype == torch.bfloat16 else "extend_simt_kernel"
        self.bound = "tensor"
        self.small = l2_text(spec).startswith("flushed")

    def chunk_call(self, c, q, k, v, out):
        """One round: its K/V appended and its extend attention, in one call
        (cpe_mixed_step with no decode rows).  The round's row views of the
        request buffers are made once and reused."""
        key = (c.index, q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr())
        views = self.views.get(key)
        if views is None:
            a = c.prefix_len - self.cached
            views = self.views[key] = tuple(t[a:a + c.query_len] for t in (q, k, v, out))
        qo, pl = self.idx[c.index]
        self.cpe.cpe_mixed_step(views[0], views[1], views[2], self.req.k_cache, self.req.v_cache, self.req.page_table,
                                qo, pl, 0, c.seq_len, out=views[3], workspace=self.wss[c.index & 1])

    def step(self, ev=None, q=None, k=None, v=None, out=None):
        cpe, req = self.cpe, self.req
        q = req.q if q is None else q
        k = req.k if k is None else k
        v = req.v if v is None else v
        out = self.out if out is None else out
        chunks, _, _ = cpe.cpe_plan_chunks(self.spec.input_len, self.spec.hit_rate, self.spec.chunk)
        for c in chunks[self.rounds[0]:self.rounds[1]]:
            if ev is not None:
                ev[0].append(torch.cuda.Event(enable_timing=True))
                ev[0][-1].record()
            self.chunk_call(c, q, k, v, out)
            if ev is not None:
                ev[1].append(torch.cuda.Event(enable_timing=True))
                ev[1][-1].record()
        return out

    def e2e_setup(self, device):
        """Host side of the end-to-end step: each round's q, k and v rows packed
        in one pinned buffer (one upload per round), two device sets that
        consecutive steps alternate (a step's uploads overlap the previous
        step's work), and a pinned output.  Returns the bytes moved per step."""
        req = self.req
        self.e2e = []
        for c in self.chunks:
            a = c.prefix_len - self.cached
            rows = [t[a:a + c.query_len] for t in (req.q, req.k, req.v)]
            sizes = [r.numel() * r.element_size() for r in rows]

            def views(buf, rows=rows, sizes=sizes):
                out, off = [], 0
                for r, n in zip(rows, sizes):  # every offset is a multiple of 256 bytes
                    out.append(buf[off:off + n].view(r.dtype).view(r.shape))
                    off += n
                return out
            host = torch.empty(sum(sizes), dtype=torch.uint8, pin_memory=True)
            for hv, r in zip(views(host), rows):
                hv.copy_(r.cpu())
            devs = [torch.empty(sum(sizes), dtype=torch.uint8, device=device) for _ in range(2)]
            self.e2e.append((c, host, devs, [views(d) for d in devs], a))
        self.e2e_out = [torch.empty_like(self.out) for _ in range(2)]
        self.e2e_host_out = torch.empty(self.out.shape, dtype=self.out.dtype, pin_memory=True)
        self.e2e_out_views = [[(o[a:a + c.query_len], self.e2e_host_out[a:a + c.query_len])
                               for c, _, _, _, a in self.e2e] for o in self.e2e_out]
        return sum(h.numel() for _, h, _, _, _ in self.e2e), self.e2e_host_out.numel() * self.e2e_host_out.element_size()

    def step_e2e(self, s, h2d, d2h, free_ev):
        """One step from pinned host inputs to pinned host output through the
        public calls, on device set s: round t's rows go host->device on one
        stream and its output device->host on another, while other rounds
        compute.  free_ev: when set s's previous step is done with it.  Returns
        the event after this step's last download."""
        cpe, req = self.cpe, self.req
        main = torch.cuda.current_stream()
        cpe.cpe_plan_chunks(self.spec.input_len, self.spec.hit_rate, self.spec.chunk)
        if free_ev is not None:
            h2d.wait_event(free_ev)
        ev_in = []
        with torch.cuda.stream(h2d):
            for _, host, devs, _, _ in self.e2e:
                devs[s].copy_(host, non_blocking=True)
                e = torch.cuda.Event()
                e.record(h2d)
                ev_in.append(e)
        ev_out = []
        for (c, _, _, views, _), (o, _), e in zip(self.e2e, self.e2e_out_views[s], ev_in):
            main.wait_event(e)
            qo, pl = self.idx[c.index]
            q, k, v = views[s]
            cpe.cpe_mixed_step(q, k, v, req.k_cache, req.v_cache, req.page_table, qo, pl, 0, c.seq_len, out=o,
                               workspace=self.wss[c.index & 1])
            e2 = torch.cuda.Event()
            e2.record(main)
            ev_out.append(e2)
        with torch.cuda.stream(d2h):
            for (o, ho), e in zip(self.e2e_out_views[s], ev_out):
                d2h.wait_event(e)
                ho.copy_(o, non_blocking=True)
            done = torch.cuda.Event()
            done.record(d2h)
        return done

    def kernel_units(self):
        return self.flops / len(self.chunks), "flop"

    def oracle_sample(self, oracle, budget_s):
        """Time the oracle on sampled rows of sampled chunks; returns (flops, seconds, text)."""
        spec, req = self.spec, self.req
        kc, vc = req.k_cache.cpu(), req.v_cache.cpu()
        pt = torch.tensor([req.page_table_host], dtype=torch.int32)
        picks = sorted(set([0, len(self.chunks) // 2, len(self.chunks) - 1]))
        flops = 0.0
        t0 = time.perf_counter()
        n_rows = 0
        rows_per = 4
        while True:
            for t in picks:
                c = self.chunks[t]
                a = c.prefix_len - self.cached
                rows = W.sample_rows(c.query_len, 32, rows_per, 7 + t)
                q = req.q[a:a + c.query_len].cpu()
                oracle.extend_attention(q, kc, vc, pt, [0, c.query_len], [c.prefix_len], spec.h_q, spec.h_kv,
                                        rows=rows)
                for r in rows:
                    flops += 4.0 * spec.d * spec.h_q * (c.prefix_len + r + 1)
                n_rows += len(rows)
            if time.perf_counter() - t0 > budget_s * 0.3 or rows_per >= 256:
                break
            rows_per *= 2
        dt = time.perf_counter() - t0
        return flops, dt, f"{n_rows} query rows x {spec.h_q} heads from chunks {picks} (all keys of each row)"


class Mixed:
    """One mixed step: decode rows and one prefill chunk under one token budget."""

    def __init__(self, spec, device, cpe):
        self.spec, self.cpe, self.device = spec, cpe, device
        g = torch.Generator().manual_seed(spec.seed)
        ctx = torch.randint(spec.ctx_lo, spec.ctx_hi + 1, (spec.n_decode,), generator=g).tolist()
        plan = cpe.cpe_plan_mixed_step(spec.token_budget, ctx, spec.prefill_prefix, spec.prefill_remaining)
        self.mb = W.make_mixed(spec, plan["extend_len"], device=device)
        self.plan = cpe.cpe_plan_mixed_step(spec.token_budget, self.mb.ctx_len, spec.prefill_prefix,
                                            spec.prefill_remaining)
        self.qo = torch.tensor(self.plan["qo_indptr"], dtype=torch.int32, device=device)
        self.pl = torch.tensor(self.plan["prefix_len"], dtype=torch.int32, device=device)
        self.max_kv = max(self.plan["kv_len"])
        n = len(self.plan["prefix_len"])
        self.ws = cpe.alloc_workspace(n, self.mb.q.shape[0], spec.h_q, spec.h_kv, spec.d, self.max_kv, device)
        self.out = torch.empty_like(self.mb.q)
        E, P = self.plan["extend_len"], spec.prefill_prefix
        dec_L = self.plan["kv_len"][:self.plan["n_decode"]]
        self.flops = chunk_flops(spec.d, spec.h_q, P, E) + sum(4.0 * spec.d * spec.h_q * L for L in dec_L)
        self.decode_bytes = sum(2.0 * L * spec.h_kv * spec.d * 2 + 2.0 * spec.h_q * spec.d * 2 for L in dec_L)
        self.prefill_kv_bytes = 2.0 * (P + E) * spec.h_kv * spec.d * 2
        self.tokens = E + self.plan["n_decode"]
        self.in_bytes = sum(t.numel() * t.element_size() for t in (self.mb.q, self.mb.k_new, self.mb.v_new))
        self.kernel = "decode_kernel"
        self.bound = "hbm"
        self.small = False

    def step(self, ev=None, q=None, k=None, v=None, out=None):
        cpe, mb, spec = self.cpe, self.mb, self.spec
        q = mb.q if q is None else q
        k = mb.k_new if k is None else k
        v = mb.v_new if v is None else v
        out = self.out if out is None else out
        cpe.cpe_plan_mixed_step(spec.token_budget, mb.ctx_len, spec.prefill_prefix, spec.prefill_remaining)
        cpe.cpe_mixed_step(q, k, v, mb.k_cache, mb.v_cache, mb.page_table, self.qo, self.pl, self.plan["n_decode"],
                           self.max_kv, out=out, workspace=self.ws)
        return out

    def decode_only(self, ev):
        """The decode rows alone through cpe_decode_attention (for the HBM roofline)."""
        nd = self.plan["n_decode"]
        ev[0].append(torch.cuda.Event(enable_timing=True))
        ev[0][-1].record()
        self.cpe.cpe_decode_attention(self.mb.q[:nd], self.mb.k_cache, self.mb.v_cache, self.mb.page_table[:nd],
                                      self.pl[:nd], self.max_kv, out=self.out[:nd], workspace=self.ws)
        ev[1].append(torch.cuda.Event(enable_timing=True))
        ev[1][-1].record()

    def host_io(self):
        return [self.mb.q, self.mb.k_new, self.mb.v_new], self.out

    def oracle_sample(self, oracle, budget_s):
        spec, mb, plan = self.spec, self.mb, self.plan
        t0 = time.perf_counter()
        flops = 0.0
        picks = list(range(0, plan["n_decode"], max(1, plan["n_decode"] // 8)))[:8]
        kl = [plan["kv_len"][s] for s in picks]
        pg = mb.k_cache.shape[1]
        need = [-(-L // pg) for L in kl]
        ids = torch.cat([mb.page_table_host[s, :n].long() for s, n in zip(picks, need)])
        kc, vc = mb.k_cache[ids.to(mb.k_cache.device)].cpu(), mb.v_cache[ids.to(mb.v_cache.device)].cpu()
        pt = torch.full((len(picks), max(need)), -1, dtype=torch.int32)
        off = 0
        for r, n in enumerate(need):
            pt[r, :n] = torch.arange(off, off + n, dtype=torch.int32)
            off += n
        t0 = time.perf_counter()
        oracle.extend_attention(mb.q[picks].cpu(), kc, vc, pt, list(range(len(picks) + 1)),
                                [plan["prefix_len"][s] for s in picks], spec.h_q, spec.h_kv)
        flops += sum(4.0 * spec.d * spec.h_q * L for L in kl)
        dt = time.perf_counter() - t0
        return flops, dt, f"{len(picks)} decode rows x {spec.h_q} heads (all keys)"


class Scheduled(Mixed):
    """One scheduling step over running and waiting requests: the budget-laid
    varlen batch (decode rows, several prefill chunks) through cpe_mixed_step."""

    def __init__(self, spec, device, cpe):
        self.spec, self.cpe, self.device = spec, cpe, device
        self.running, self.waiting = W.scheduled_requests(spec)
        self.plan = cpe.cpe_plan_schedule(spec.token_budget, self.running, self.waiting)
        qo = self.plan["qo_indptr"]
        lens = [(p, qo[i + 1] - qo[i]) for i, p in enumerate(self.plan["prefix_len"])]
        self.mb = W.make_scheduled(spec, lens, device=device)
        self.qo = torch.tensor(qo, dtype=torch.int32, device=device)
        self.pl = torch.tensor(self.plan["prefix_len"], dtype=torch.int32, device=device)
        self.max_kv = max(self.plan["kv_len"])
        nd = self.plan["n_decode"]
        self.ws = cpe.alloc_workspace(len(lens), self.mb.q.shape[0], spec.h_q, spec.h_kv, spec.d, self.max_kv,
                                      device)
        self.out = torch.empty_like(self.mb.q)
        dec_L = self.plan["kv_len"][:nd]
        self.extend_flops = sum(chunk_flops(spec.d, spec.h_q, P, E) for P, E in lens[nd:])
        self.flops = self.extend_flops + sum(4.0 * spec.d * spec.h_q * L for L in dec_L)
        self.decode_bytes = sum(2.0 * L * spec.h_kv * spec.d * 2 + 2.0 * spec.h_q * spec.d * 2 for L in dec_L)
        self.prefill_kv_bytes = sum(2.0 * (P + E) * spec.h_kv * spec.d * 2 for P, E in lens[nd:])
        self.tokens = qo[-1]
        self.in_bytes = sum(t.numel() * t.element_size() for t in (self.mb.q, self.mb.k_new, self.mb.v_new))
        # the chunks alone, for the extend call's roofline
        r0 = qo[nd]
        self.q_ext = self.mb.q[r0:]
        self.out_ext = self.out[r0:]
        self.qo_ext = torch.tensor([x - r0 for x in qo[nd:]], dtype=torch.int32, device=device)
        self.pl_ext = self.pl[nd:]
        self.pt_ext = self.mb.page_table[nd:]
        self.lens = lens
        self.kernel = "extend_tc_kernel"
        self.bound = "tensor"
        self.small = False

    def step(self, ev=None, q=None, k=None, v=None, out=None):
        cpe, mb, spec = self.cpe, self.mb, self.spec
        q = mb.q if q is None else q
        k = mb.k_new if k is None else k
        v = mb.v_new if v is None else v
        out = self.out if out is None else out
        cpe.cpe_plan_schedule(spec.token_budget, self.running, self.waiting)
        cpe.cpe_mixed_step(q, k, v, mb.k_cache, mb.v_cache, mb.page_table, self.qo, self.pl, self.plan["n_decode"],
                           self.max_kv, out=out, workspace=self.ws)
        return out

    def extend_only(self, ev):
        """The prefill chunks alone through cpe_extend_attention (the tensor roofline)."""
        ev[0].append(torch.cuda.Event(enable_timing=True))
        ev[0][-1].record()
        self.cpe.cpe_extend_attention(self.q_ext, self.mb.k_cache, self.mb.v_cache, self.pt_ext, self.qo_ext,
                                      self.pl_ext, self.max_kv, out=self.out_ext, workspace=self.ws)
        ev[1].append(torch.cuda.Event(enable_timing=True))
        ev[1][-1].record()

    def oracle_sample(self, oracle, budget_s):
        spec, mb, plan = self.spec, self.mb, self.plan
        nd = plan["n_decode"]
        qo = plan["qo_indptr"]
        # four decode rows and two rows of every chunk, all heads, all keys
        picks = list(range(0, nd, max(1, nd // 4)))[:4]
        pg = mb.k_cache.shape[1]
        flops, dt = 0.0, 0.0
        for s in picks + list(range(nd, len(self.lens))):
            E = qo[s + 1] - qo[s]
            rows = [0] if E == 1 else [E // 3, E - 1]
            L = plan["kv_len"][s]
            n = -(-L // pg)
            ids = mb.page_table_host[s, :n].long().to(mb.k_cache.device)
            kc, vc = mb.k_cache[ids].cpu(), mb.v_cache[ids].cpu()
            pt = torch.arange(n, dtype=torch.int32).view(1, -1)
            q = mb.q[qo[s]:qo[s + 1]].cpu()
            t0 = time.perf_counter()
            oracle.extend_attention(q, kc, vc, pt, [0, E], [plan["prefix_len"][s]], spec.h_q, spec.h_kv, rows=rows)
            dt += time.perf_counter() - t0
            flops += sum(4.0 * spec.d * spec.h_q * (plan["prefix_len"][s] + r + 1) for r in rows)
        return flops, dt, f"{len(picks)} decode rows and 2 rows of each of {len(self.lens) - nd} chunks x {spec.h_q} " \
                          "heads (all keys of each row)"


def make_workload(args, device, cpe):
    spec = W.CONFIGS[args.workload]
    if isinstance(spec, W.ScheduledSpec):
        return Scheduled(spec, device, cpe)
    if isinstance(spec, W.MixedSpec):
        if args.decode_rows:
            spec = W.shrink(spec, n_decode=args.decode_rows)
        return Mixed(spec, device, cpe)
    if args.input_len:
        spec = W.shrink(spec, input_len=args.input_len)
    rounds = tuple(int(x) for x in args.rounds.split(":")) if args.rounds else None
    return Chunked(spec, device, cpe, rounds)


# --------------------------------------------------------------------------- helpers

class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.idx = device_index
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws, device):
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def flush_l2(buf):
    buf.add_(1)


# --------------------------------------------------------------------------- arms

def l2_text(spec):
    """How the timed steps keep L2 from serving a step's inputs from the one
    before: chunked workloads whose inputs and caches fit twice in L2 are
    flushed between steps, everything else is larger than L2."""
    if isinstance(spec, W.ChunkedSpec):
        es = 2 if spec.dtype == torch.bfloat16 else 4
        n_new = spec.input_len - math.floor(spec.input_len * spec.hit_rate)
        pages = -(-spec.input_len // spec.page_size)
        b = n_new * (spec.h_q + 2 * spec.h_kv) * spec.d * es + 2 * pages * spec.page_size * spec.h_kv * spec.d * es
        if b < 2 * L2_BYTES:
            return "flushed between steps (256 MiB write outside the per-step events)"
    return "inputs larger than L2 (no flush)"


def workload_config(name, args, ws):
    return {"workload": f"{name}: {W.WORKLOAD_TEXT[name]}" +
            (f" (input_len {args.input_len})" if args.input_len else "") +
            (f" (decode rows {args.decode_rows})" if args.decode_rows else "") +
            (f" (rounds {args.rounds})" if args.rounds else ""),
            "l2": l2_text(W.CONFIGS[name]), "parallelism": f"replicas x{ws}"}


def measure(wl, name, steps, warmup, peaks, ws, device, traffic_ok=False):
    """Warm-up, then `steps` timed steps of workload `wl` (events around each
    step, clocks sampled meanwhile), then its dominant kernel's roofline.
    Returns the fields of a bench line for this workload."""
    from chunked_prefill_extend_gb300 import cpe
    flush = torch.zeros(256 * 1024 * 1024 // 4, dtype=torch.float32, device=device) if wl.small else None
    for _ in range(warmup):
        wl.step()
        if flush is not None:
            flush_l2(flush)
    st, detail = cpe.cpe_get_device_status()
    if st != cpe.CPE_OK:
        raise RuntimeError(f"{name}: device status after warm-up: {cpe.cpe_status_string(st)} ({detail})")

    clocks = Clocks(device.index or 0)
    clocks.start()
    time.sleep(0.3)
    sev = []
    launches0 = cpe.cpe_launch_count()
    barrier(ws)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record()
    for _ in range(steps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        wl.step()  # no events between a step's calls: they would keep its launches from overlapping
        b.record()
        sev.append((a, b))
        if flush is not None:
            flush_l2(flush)
    t_end.record()
    torch.cuda.synchronize()
    barrier(ws)
    launches = cpe.cpe_launch_count() - launches0
    clk = clocks.stop()
    st, detail = cpe.cpe_get_device_status()
    if st != cpe.CPE_OK:
        raise RuntimeError(f"{name}: device status after timing: {cpe.cpe_status_string(st)} ({detail})")
    step_ms = [a.elapsed_time(b) for a, b in sev]
    region_ms = t_start.elapsed_time(t_end)
    my_ms = sum(step_ms) if flush is not None else region_ms
    total_ms = max_over_ranks(my_ms, ws, device)
    ms_per_step = total_ms / steps
    value = wl.flops * ws / (ms_per_step * 1e-3) / 1e12

    # dominant kernel, timed live with events on the launching stream
    if isinstance(wl, Scheduled):
        ext_ev, dev_ev = ([], []), ([], [])
        for _ in range(max(3, steps // 2)):
            wl.extend_only(ext_ev)
            wl.decode_only(dev_ev)
        torch.cuda.synchronize()
        kms = statistics.mean(a.elapsed_time(b) for a, b in zip(*ext_ev))
        dms = statistics.mean(a.elapsed_time(b) for a, b in zip(*dev_ev))
        achieved = wl.extend_flops / (kms * 1e-3) / 1e12
        pk = peaks["bf16_sustained"]
        dach = wl.decode_bytes / (dms * 1e-3) / 1e9
        roof = {"bound": "tensor", "achieved": achieved, "peak": pk, "unit": "TFLOP/s", "frac": achieved / pk,
                "traffic": None, "kernel": "extend attention call on the step's prefill chunks",
                "peak_source": peaks["source"] + " bf16_tflops_sustained", "units_per_launch": wl.extend_flops,
                "decode_rows": {"achieved": dach, "unit": "GB/s", "peak": peaks["hbm_gbs"],
                                "frac": dach / peaks["hbm_gbs"], "ms": dms},
                "per_chunk": [{"prefix_len": P, "query_len": E} for P, E in wl.lens[wl.plan["n_decode"]:]]}
    elif isinstance(wl, Mixed):
        # the step is one fused launch (decode rows on the CTAs the prefill
        # chunk leaves free); its HBM roofline counts the K/V it must read
        dev_ev = ([], [])
        for _ in range(max(3, steps // 2)):
            wl.decode_only(dev_ev)
        torch.cuda.synchronize()
        dms = statistics.mean(a.elapsed_time(b) for a, b in zip(*dev_ev))
        step_bytes = wl.decode_bytes + wl.prefill_kv_bytes
        achieved = step_bytes / (ms_per_step * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": None,
                "kernel": "mixed-step call (prep_kernel: schedule + K/V append; extend_tc_kernel with decode workers; merges)",
                "peak_source": peaks["source"] + " hbm_gbs", "units_per_launch": step_bytes,
                "decode_kernel_alone": {"achieved": wl.decode_bytes / (dms * 1e-3) / 1e9, "unit": "GB/s",
                                        "frac": wl.decode_bytes / (dms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                                        "ms": dms}}
    else:
        # one round's call, timed over the timed region: its mean duration
        # there is the step time over the rounds (the calls run back to back)
        nch = len(wl.chunks)
        kms = ms_per_step / nch
        per_launch = wl.flops / nch
        achieved = per_launch / (kms * 1e-3) / 1e12
        if wl.spec.dtype == torch.bfloat16:
            bound, pk, src = "tensor", peaks["bf16_sustained"], peaks["source"] + " bf16_tflops_sustained"
            kname = "one round's call: K/V append + extend attention (prep_kernel + extend_tc_kernel + merge)"
        else:  # fp32 data runs on the CUDA cores: FP32 FMA issue rate, SMs x 128 lanes x 2 flop x clock
            n_sms = torch.cuda.get_device_properties(device).multi_processor_count
            bound, pk = "alu", FP32_LANES_PER_SM * 2 * n_sms * FP32_PEAK_CLOCK_MHZ * 1e6 / 1e12
            src = (f"derived: {n_sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 flop (FMA) x "
                   f"{FP32_PEAK_CLOCK_MHZ} MHz (maximum SM clock)")
            kname = "one round's call: K/V append + extend attention (kv_append_kernel + extend_simt_kernel, fp32)"
        traffic = profiled_traffic(per_launch) if traffic_ok else None
        roof = {"bound": bound, "achieved": achieved, "peak": pk, "unit": "TFLOP/s", "frac": achieved / pk,
                "traffic": traffic, "kernel": kname, "peak_source": src, "units_per_launch": per_launch}
        # per round: a pass after the timed region with events around every
        # call (so each call runs alone); the median over its steps
        kev = ([], [])
        for _ in range(steps):
            wl.step(ev=kev)
            if flush is not None:
                flush_l2(flush)
        torch.cuda.synchronize()
        kms_list = [a.elapsed_time(b) for a, b in zip(*kev)]
        med = [statistics.median(kms_list[i::nch]) for i in range(nch)]
        curve = [(c.prefix_len, chunk_flops(wl.spec.d, wl.spec.h_q, c.prefix_len, c.query_len) / (t * 1e-3) / 1e12)
                 for c, t in zip(wl.chunks, med)]
        pick = sorted(set([0, len(curve) // 4, len(curve) // 2, 3 * len(curve) // 4, len(curve) - 1])) \
            if len(curve) > 8 else list(range(len(curve)))
        roof["per_chunk_tflops"] = {str(curve[i][0]): round(curve[i][1], 1) for i in pick}
        roof["per_chunk_reps"] = len(kms_list) // nch
        roof["aggregate_tflops"] = wl.flops / (sum(med) * 1e-3) / 1e12  # sum of flops / sum of median times
    return {"value": value, "ms_per_step": ms_per_step, "tokens_per_s": wl.tokens * ws / (ms_per_step * 1e-3),
            "flops_per_step": wl.flops, "roofline": roof, "clocks": clk, "gpu_launches": launches,
            "steps": steps, "warmup": warmup}


# the other workloads, timed after the headline in the same run
PER_CONFIG = ("prefill-4000-c512", "prefill-32k-hit50", "mixed-256dec-2048", "sched", "fp32-512")


def run_ours(args, ws, rank, local):
    from chunked_prefill_extend_gb300 import cpe
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    peaks = _peaks()
    wl = make_workload(args, device, cpe)
    full = not args.input_len and not args.rounds and not args.decode_rows
    m = measure(wl, args.workload, args.steps, args.warmup, peaks, ws, device,
                traffic_ok=args.workload == "prefill-128k-c1024" and full)

    # end to end through the public API with host buffers
    e2e = None if args.no_e2e else e2e_measure(wl, args, device, ws)

    line = {
        "metric": "extend-attn TFLOP/s & tokens/s per chunk; % bf16 TC peak / % HBM BW (1 GB300)",
        "value": m["value"], "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": m["ms_per_step"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if W.CONFIGS[args.workload].dtype == torch.bfloat16 else "f32", "data": "synthetic",
        "tokens_per_s": m["tokens_per_s"], "flops_per_step": m["flops_per_step"],
        "config": workload_config(args.workload, args, ws),
        "roofline": m["roofline"], "clocks": m["clocks"], "gpu_launches": m["gpu_launches"], "e2e": e2e,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args)
    if full and args.workload == "prefill-128k-c1024" and not args.no_per_config:
        del wl
        torch.cuda.empty_cache()
        per = {}
        for name in PER_CONFIG:
            a2 = argparse.Namespace(**{**vars(args), "workload": name})
            w2 = make_workload(a2, device, cpe)
            r = measure(w2, name, 20, 5, peaks, ws, device)
            r["config"] = workload_config(name, a2, ws)
            r["dtype"] = "bf16" if W.CONFIGS[name].dtype == torch.bfloat16 else "f32"
            per[name] = r
            del w2
            torch.cuda.empty_cache()
        line["per_config"] = per
    if rank == 0:
        print(json.dumps(line), flush=True)


def e2e_measure(wl, args, device, ws):
    """The same metric through the public API with pinned host inputs copied in
    and the output copied back inside the timed region (every step)."""
    h2d = torch.cuda.Stream(device=device)
    d2h = torch.cuda.Stream(device=device)
    if hasattr(wl, "e2e_setup"):
        bytes_in, bytes_out = wl.e2e_setup(device)
        done = [None, None]
        count = [0]

        def one_step():
            s = count[0] & 1
            done[s] = wl.step_e2e(s, h2d, d2h, done[s])
            count[0] += 1
        copies = ("pinned host buffers, each round's q/k/v rows in one; per-round uploads and downloads on two "
                  "side streams overlapping compute, consecutive steps on alternate device buffers")
    else:
        ins, out_dev = wl.host_io()
        host_in = [t.cpu().pin_memory() for t in ins]
        host_out = torch.empty(out_dev.shape, dtype=out_dev.dtype, pin_memory=True)
        dev_sets = [([torch.empty_like(t) for t in ins], torch.empty_like(out_dev)) for _ in range(2)]
        bytes_in = sum(t.numel() * t.element_size() for t in host_in)
        bytes_out = host_out.numel() * host_out.element_size()
        done = [None, None]
        count = [0]

        def one_step():
            s = count[0] & 1
            dev_in, dev_out = dev_sets[s]
            main = torch.cuda.current_stream()
            if done[s] is not None:
                h2d.wait_event(done[s])  # set s's previous step is done with it
            with torch.cuda.stream(h2d):
                for d, h in zip(dev_in, host_in):
                    d.copy_(h, non_blocking=True)
            main.wait_stream(h2d)
            wl.step(q=dev_in[0], k=dev_in[1], v=dev_in[2], out=dev_out)
            d2h.wait_stream(main)
            with torch.cuda.stream(d2h):
                host_out.copy_(dev_out, non_blocking=True)
                done[s] = torch.cuda.Event()
                done[s].record(d2h)
            count[0] += 1
        copies = ("pinned host buffers; upload, step, download, consecutive steps on alternate device buffers "
                  "(a step's upload and download overlap its neighbours' compute)")

    n = max(3, min(args.steps, 10))
    for _ in range(2):
        one_step()
    torch.cuda.current_stream().wait_stream(d2h)
    torch.cuda.synchronize()
    barrier(ws)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    h2d.wait_stream(torch.cuda.current_stream())  # the first upload starts inside the timed region
    for _ in range(n):
        one_step()
    torch.cuda.current_stream().wait_stream(d2h)  # every step's download is inside the timed region
    b.record()
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b) / n, ws, device)
    return {"value": wl.flops * ws / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": bytes_in, "d2h_bytes_per_step": bytes_out, "ms_per_step": ms, "copies": copies}


def cpu_baseline(wl, args):
    import oracle
    oracle.build()
    flops, dt, text = wl.oracle_sample(oracle, budget_s=20.0)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": text, "seconds": dt}


def run_reference(args, ws, rank, local):
    """The oracle (float64 CPU) as the reference arm, on a bounded sample per step."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    spec = W.CONFIGS[args.workload]
    # inputs generated on the CPU with the same seeded recipe (no GPU needed)
    if isinstance(spec, (W.MixedSpec, W.ScheduledSpec)):
        wl = _ref_mixed(spec)
    else:
        wl = _ref_chunked(spec)
    for _ in range(args.warmup):
        wl()
    t0 = time.perf_counter()
    fl = 0.0
    for _ in range(args.steps):
        fl += wl()
    dt = time.perf_counter() - t0
    value = fl / dt / 1e12
    line = {"metric": "extend-attn TFLOP/s & tokens/s per chunk; % bf16 TC peak / % HBM BW (1 GB300)",
            "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": workload_config(args.workload, args, ws),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": wl.text},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _ref_chunked(spec):
    import oracle
    # the sample: 2 query rows (all heads, all keys) from each of three chunks
    chunks = oracle.plan_chunks(spec.input_len, spec.hit_rate, spec.chunk)
    picks = sorted(set([0, len(chunks) // 2, len(chunks) - 1]))
    g = torch.Generator().manual_seed(spec.seed)
    N = spec.input_len
    pg = spec.page_size
    npages = -(-N // pg)
    kc = (torch.randn(npages, pg, spec.h_kv, spec.d, generator=g) * spec.std).to(spec.dtype)
    vc = (torch.randn(npages, pg, spec.h_kv, spec.d, generator=g) * spec.std).to(spec.dtype)
    pt = torch.arange(npages, dtype=torch.int32).view(1, -1)
    state = {"k": 0}

    def step():
        fl = 0.0
        for t in picks:
            c = chunks[t]
            q = (torch.randn(c.query_len, spec.h_q, spec.d, generator=g) * spec.std).to(spec.dtype)
            rows = [c.query_len - 1 - ((state["k"] * 7 + 3 * j) % c.query_len) for j in range(2)]
            oracle.extend_attention(q, kc, vc, pt, [0, c.query_len], [c.prefix_len], spec.h_q, spec.h_kv, rows=rows)
            fl += sum(4.0 * spec.d * spec.h_q * (c.prefix_len + r + 1) for r in rows)
        state["k"] += 1
        return fl
    step.text = f"2 query rows x {spec.h_q} heads from chunks {picks} per step (all keys of each row)"
    return step


def _ref_mixed(spec):
    import oracle
    g = torch.Generator().manual_seed(spec.seed)
    ctx = torch.randint(spec.ctx_lo, spec.ctx_hi + 1, (spec.n_decode,), generator=g).tolist()
    pg = spec.page_size
    picks = ctx[:4]
    npg = [-(-L // pg) for L in picks]
    kc = (torch.randn(sum(npg), pg, spec.h_kv, spec.d, generator=g) * spec.std).to(spec.dtype)
    vc = (torch.randn(sum(npg), pg, spec.h_kv, spec.d, generator=g) * spec.std).to(spec.dtype)
    pt = torch.full((len(picks), max(npg)), -1, dtype=torch.int32)
    off = 0
    for r, n in enumerate(npg):
        pt[r, :n] = torch.arange(off, off + n, dtype=torch.int32)
        off += n
    q = (torch.randn(len(picks), spec.h_q, spec.d, generator=g) * spec.std).to(spec.dtype)

    def step():
        oracle.extend_attention(q, kc, vc, pt, list(range(len(picks) + 1)), [L - 1 for L in picks], spec.h_q,
                                spec.h_kv)
        return sum(4.0 * spec.d * spec.h_q * L for L in picks)
    step.text = f"{len(picks)} decode rows x {spec.h_q} heads per step (all keys)"
    return step


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="prefill-128k-c1024", choices=sorted(W.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end measurement")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the other workloads timed after the default one")
    ap.add_argument("--input-len", type=int, default=0, help="shrink a chunked workload's request (profiling)")
    ap.add_argument("--decode-rows", type=int, default=0, help="shrink the mixed step's decode rows (profiling)")
    ap.add_argument("--rounds", default="", help="a:b, run only chunks [a, b) of a chunked workload (profiling)")
    args = ap.parse_args()
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, ws, rank, local)
    else:
        run_ours(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
