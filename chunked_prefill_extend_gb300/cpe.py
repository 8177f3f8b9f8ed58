"""Thin ctypes binding of libcpe (include/cpe.h).

Each function has the name of the C entry point it calls and only marshals
arguments: torch tensors become device pointers, the current torch stream
becomes the cudaStream_t, and a non-OK status becomes a ``CpeError``.  Every
step of the computation runs in libcpe's kernels; there is no other path.  If
``libcpe.so`` is missing the import fails: build it with
``python -m chunked_prefill_extend_gb300.build`` (or ``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import NamedTuple
from dataclasses import dataclass

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libcpe.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(f"libcpe.so not built ({_LIB_PATH}); run chunked_prefill_extend_gb300/build.py")
_lib = ctypes.CDLL(_LIB_PATH)

CPE_OK, CPE_ERR_INVALID_ARG, CPE_ERR_UNSUPPORTED, CPE_ERR_CAPACITY, CPE_ERR_CUDA, CPE_ERR_TIMEOUT, \
    CPE_ERR_DEVICE_ARG = range(7)
CPE_F32, CPE_BF16 = 0, 1

EXPORTS = ["cpe_plan_chunks", "cpe_plan_budget", "cpe_plan_mixed_step", "cpe_plan_schedule", "cpe_kv_append",
           "cpe_workspace_size", "cpe_extend_attention", "cpe_mixed_step", "cpe_decode_attention",
           "cpe_get_device_status", "cpe_set_wait_limit_ns", "cpe_status_string", "cpe_last_error",
           "cpe_launch_count", "cpe_decode_attention_noalloc", "cpe_decide_decode_first",
           "cpe_simulate_requests"]

_vp, _i32, _i64, _f32, _f64, _sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                    ctypes.c_double, ctypes.c_size_t)


class _Chunk(ctypes.Structure):
    _fields_ = [("index", _i32), ("prefix_len", _i32), ("query_len", _i32), ("seq_len", _i32),
                ("model_seq_len", _i32)]


_lib.cpe_plan_chunks.argtypes = [_i64, _f64, _i32, _i32, ctypes.POINTER(_Chunk), _i32,
                                 ctypes.POINTER(_i32), ctypes.POINTER(_i64), ctypes.POINTER(_i64)]
_lib.cpe_plan_budget.argtypes = [_i32, _i32, _vp, _vp, ctypes.POINTER(_i32)]
_lib.cpe_plan_mixed_step.argtypes = [_i32, _i32, _vp, _i32, _i32, _vp, _vp, _vp, ctypes.POINTER(_i32),
                                     ctypes.POINTER(_i32), ctypes.POINTER(_i32)]
_lib.cpe_plan_schedule.argtypes = [_i32, _i32, _vp, _vp, _i32, _vp, _vp, _vp, ctypes.POINTER(_i32), _vp, _vp, _vp,
                                   _vp, ctypes.POINTER(_i32), ctypes.POINTER(_i32)]
_LATENCY_FN = ctypes.CFUNCTYPE(ctypes.c_double, _vp, _i32, _i32, _i32, _i32)
_DECIDE_FN = ctypes.CFUNCTYPE(_i32, _vp, _i32, _i32, _i32, _i32, ctypes.POINTER(_i32), ctypes.POINTER(_i32))
_MERGE_FN = ctypes.CFUNCTYPE(ctypes.c_double, _vp, ctypes.c_double, ctypes.c_double)


class _SimResult(ctypes.Structure):
    _fields_ = [("ttft_ms", _f64), ("tpot_ms", _f64), ("makespan_ms", _f64), ("request_throughput", _f64),
                ("output_throughput", _f64), ("steps", _i64)]


_lib.cpe_decide_decode_first.argtypes = [_i32, _i32, _i32, _i32, _i32, ctypes.POINTER(_i32), ctypes.POINTER(_i32)]
_lib.cpe_simulate_requests.argtypes = [_i32, _vp, _vp, _i32, _i32, _i32, _LATENCY_FN, _vp, _DECIDE_FN, _MERGE_FN, _vp,
                                       _vp, _vp, ctypes.POINTER(_SimResult)]
_lib.cpe_kv_append.argtypes = [_vp, _vp, _vp, _vp, _i64, _vp, _i32, _vp, _vp, _i32, _i32, _i32, _i32,
                               _i32, ctypes.c_int, _vp]
_lib.cpe_workspace_size.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32]
_lib.cpe_workspace_size.restype = _sz
_lib.cpe_extend_attention.argtypes = [_vp, _vp, _vp, _i64, _vp, _i32, _vp, _vp, _i32, _i32, _i32, _i32,
                                      _i32, _i32, _i32, _f32, ctypes.c_int, _vp, _vp, _vp, _sz, _vp]
_lib.cpe_mixed_step.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _vp, _i32, _vp, _vp, _i32, _i32, _i32, _i32,
                                _i32, _i32, _i32, _i32, _f32, ctypes.c_int, _vp, _vp, _vp, _sz, _vp]
_lib.cpe_decode_attention.argtypes = [_vp, _vp, _vp, _i64, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32,
                                      _i32, _f32, ctypes.c_int, _vp, _vp, _vp, _sz, _vp]
_lib.cpe_decode_attention_noalloc.argtypes = [_vp, _vp, _vp, _i64, _vp, _i32, _vp, _i32, _i32, _i32, _i32,
                                              _i32, _i32, _f32, ctypes.c_int, _vp, _vp, _vp]
_lib.cpe_get_device_status.argtypes = [_vp, ctypes.POINTER(_i32)]
_lib.cpe_set_wait_limit_ns.argtypes = [_i64]
_lib.cpe_set_wait_limit_ns.restype = _i64
_lib.cpe_status_string.argtypes = [ctypes.c_int]
_lib.cpe_status_string.restype = ctypes.c_char_p
_lib.cpe_last_error.restype = ctypes.c_char_p
_lib.cpe_launch_count.restype = _i64


class CpeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.cpe_last_error().decode() or _lib.cpe_status_string(status).decode()
        super().__init__(f"{where}: {_lib.cpe_status_string(status).decode()} ({status}): {msg}")


def _check(st: int, where: str):
    if st != CPE_OK:
        raise CpeError(st, where)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return CPE_BF16
    if t.dtype == torch.float32:
        return CPE_F32
    raise TypeError(f"libcpe takes bfloat16 or float32 tensors, got {t.dtype}")


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream):
    """The stream handle: the given stream's, else the current device's current stream."""
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        return _raw_stream(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


@dataclass(frozen=True)
class Chunk:
    index: int
    prefix_len: int
    query_len: int
    seq_len: int
    model_seq_len: int


def cpe_plan_chunks(input_len: int, prefix_hit_rate: float, chunk_size: int, align_to: int = 0):
    """Chunk plan of one request -> (chunks, cached_len, effective_len)."""
    n = _i32(0)
    cached = _i64(0)
    eff = _i64(0)
    st = _lib.cpe_plan_chunks(input_len, prefix_hit_rate, chunk_size, align_to, None, 0, ctypes.byref(n),
                              ctypes.byref(cached), ctypes.byref(eff))
    if st not in (CPE_OK, CPE_ERR_CAPACITY):
        _check(st, "cpe_plan_chunks")
    buf = (_Chunk * max(1, n.value))()
    _check(_lib.cpe_plan_chunks(input_len, prefix_hit_rate, chunk_size, align_to, buf, n.value,
                                ctypes.byref(n), ctypes.byref(cached), ctypes.byref(eff)), "cpe_plan_chunks")
    chunks = [Chunk(c.index, c.prefix_len, c.query_len, c.seq_len, c.model_seq_len) for c in buf[:n.value]]
    return chunks, cached.value, eff.value


def cpe_plan_budget(token_budget: int, need):
    need_a = (_i32 * max(1, len(need)))(*need)
    out = (_i32 * max(1, len(need)))()
    used = _i32(0)
    _check(_lib.cpe_plan_budget(token_budget, len(need), need_a, out, ctypes.byref(used)), "cpe_plan_budget")
    return list(out[:len(need)]), used.value


def cpe_plan_mixed_step(token_budget: int, decode_ctx_len, prefill_prefix_len: int, prefill_remaining: int):
    n = len(decode_ctx_len)
    ctx = (_i32 * max(1, n))(*decode_ctx_len)
    qo = (_i32 * (n + 2))()
    pl = (_i32 * (n + 1))()
    kv = (_i32 * (n + 1))()
    ns, nd, ext = _i32(0), _i32(0), _i32(0)
    _check(_lib.cpe_plan_mixed_step(token_budget, n, ctx, prefill_prefix_len, prefill_remaining, qo, pl, kv,
                                    ctypes.byref(ns), ctypes.byref(nd), ctypes.byref(ext)), "cpe_plan_mixed_step")
    k = ns.value
    return {"qo_indptr": list(qo[:k + 1]), "prefix_len": list(pl[:k]), "kv_len": list(kv[:k]),
            "n_decode": nd.value, "extend_len": ext.value}


def cpe_plan_schedule(token_budget: int, running, waiting):
    """running: [(computed, need)], waiting: [(cached, prompt)], both in queue order."""
    nr, nw = len(running), len(waiting)
    n = nr + nw
    rc = (_i32 * max(1, nr))(*[c for c, _ in running])
    rn = (_i32 * max(1, nr))(*[x for _, x in running])
    wc = (_i32 * max(1, nw))(*[c for c, _ in waiting])
    wp = (_i32 * max(1, nw))(*[p for _, p in waiting])
    granted = (_i32 * max(1, n))()
    qo = (_i32 * (n + 1))()
    pl, kv, sr = (_i32 * max(1, n))(), (_i32 * max(1, n))(), (_i32 * max(1, n))()
    adm, ns, nd = _i32(0), _i32(0), _i32(0)
    _check(_lib.cpe_plan_schedule(token_budget, nr, rc, rn, nw, wc, wp, granted, ctypes.byref(adm), qo, pl, kv, sr,
                                  ctypes.byref(ns), ctypes.byref(nd)), "cpe_plan_schedule")
    k = ns.value
    return {"granted": list(granted[:n]), "n_admitted": adm.value, "qo_indptr": list(qo[:k + 1]),
            "prefix_len": list(pl[:k]), "kv_len": list(kv[:k]), "seq_request": list(sr[:k]), "n_decode": nd.value}


class SchedulerState(NamedTuple):
    """What a scheduler sees at each simulated step."""
    ready_decode: int
    pending_prefill: int
    chunk_query_len: int
    max_batched_tokens: int


class StepDecision(NamedTuple):
    p_step: int
    d_step: int


def cpe_decide_decode_first(max_batched_tokens: int, ready_decode: int, pending_prefill: int, chunk_query_len: int,
                            slack_percent: int = 115) -> StepDecision:
    p, d = _i32(0), _i32(0)
    _check(_lib.cpe_decide_decode_first(max_batched_tokens, ready_decode, pending_prefill, chunk_query_len,
                                        slack_percent, ctypes.byref(p), ctypes.byref(d)), "cpe_decide_decode_first")
    return StepDecision(p.value, d.value)


def cpe_simulate_requests(chunks, n_requests: int, output_len: int, max_batched_tokens: int, latency,
                          scheduler=None) -> dict:
    """Time simulation of n_requests requests with chunk plan ``chunks`` =
    [(query_len, seq_len)].  latency(is_decode, batch, query_len, seq_len) -> ms.
    scheduler: None (decode-first with 15 % slack) or an object with
    decide(SchedulerState) -> StepDecision and step_latency(prefill_ms, decode_ms)."""
    n = len(chunks)
    ql = (_i32 * max(1, n))(*[q for q, _ in chunks])
    sl = (_i32 * max(1, n))(*[x for _, x in chunks])
    lat = _LATENCY_FN(lambda ctx, d, b, q, x: float(latency(bool(d), b, q, x)))
    dec, mrg = _DECIDE_FN(), _MERGE_FN()
    if scheduler is not None:
        def _decide(ctx, ready, pending, qlen, B, p, d):
            try:
                r = scheduler.decide(SchedulerState(ready, pending, qlen, B))
                p[0], d[0] = int(r.p_step), int(r.d_step)
                return 0
            except Exception:  # reported to the caller as a failed scheduler
                return 1
        dec = _DECIDE_FN(_decide)
        mrg = _MERGE_FN(lambda ctx, a, b: float(scheduler.step_latency(a, b)))
    first = (_f64 * max(1, n_requests))()
    fin = (_f64 * max(1, n_requests))()
    res = _SimResult()
    _check(_lib.cpe_simulate_requests(n, ql, sl, n_requests, output_len, max_batched_tokens, lat, None, dec, mrg,
                                      None, first, fin, ctypes.byref(res)), "cpe_simulate_requests")
    return {"ttft": res.ttft_ms, "tpot": res.tpot_ms, "makespan": res.makespan_ms,
            "request_throughput": res.request_throughput, "output_throughput": res.output_throughput,
            "steps": res.steps, "first_token_time": list(first[:n_requests]), "finish_time": list(fin[:n_requests])}


def cpe_workspace_size(n_seqs: int, total_q: int, h_q: int, h_kv: int, d: int, max_kv_len: int) -> int:
    return int(_lib.cpe_workspace_size(n_seqs, total_q, h_q, h_kv, d, max_kv_len))


def alloc_workspace(n_seqs, total_q, h_q, h_kv, d, max_kv_len, device) -> torch.Tensor:
    """A device buffer of cpe_workspace_size() bytes (torch's allocator gives 256-byte alignment)."""
    n = cpe_workspace_size(n_seqs, total_q, h_q, h_kv, d, max_kv_len)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def cpe_kv_append(k_new, v_new, k_cache, v_cache, page_table, qo_indptr, prefix_len, stream=None):
    num_pages, page_size, h_kv, d = k_cache.shape
    _check(_lib.cpe_kv_append(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), num_pages,
                              _ptr(page_table), page_table.shape[1], _ptr(qo_indptr), _ptr(prefix_len),
                              prefix_len.numel(), k_new.shape[0], h_kv, d, page_size, _dtype(k_cache),
                              _stream(stream)), "cpe_kv_append")


def cpe_extend_attention(q, k_cache, v_cache, page_table, qo_indptr, prefix_len, max_kv_len, out=None,
                         lse=None, workspace=None, sm_scale=None, stream=None):
    """Extend output for all query rows.  Returns (out, lse)."""
    total_q, h_q, d = q.shape
    num_pages, page_size, h_kv, _ = k_cache.shape
    n_seqs = prefix_len.numel()
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = alloc_workspace(n_seqs, total_q, h_q, h_kv, d, max_kv_len, q.device)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d)
    _check(_lib.cpe_extend_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), num_pages, _ptr(page_table),
                                     page_table.shape[1], _ptr(qo_indptr), _ptr(prefix_len), n_seqs, total_q,
                                     max_kv_len, h_q, h_kv, d, page_size, sm_scale, _dtype(q), _ptr(out),
                                     _ptr(lse), _ptr(workspace), workspace.numel(), _stream(stream)),
           "cpe_extend_attention")
    return out, lse


def cpe_decode_attention(q, k_cache, v_cache, page_table, prefix_len, max_kv_len, out=None, lse=None,
                         workspace=None, sm_scale=None, stream=None):
    """Decode rows: q [n_seqs, H_q, d], one row per sequence, keys [0, prefix_len+1)."""
    n_seqs, h_q, d = q.shape
    num_pages, page_size, h_kv, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = alloc_workspace(n_seqs, n_seqs, h_q, h_kv, d, max_kv_len, q.device)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d)
    _check(_lib.cpe_decode_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), num_pages, _ptr(page_table),
                                     page_table.shape[1], _ptr(prefix_len), n_seqs, max_kv_len, h_q, h_kv, d,
                                     page_size, sm_scale, _dtype(q), _ptr(out), _ptr(lse), _ptr(workspace),
                                     workspace.numel(), _stream(stream)), "cpe_decode_attention")
    return out, lse


def cpe_mixed_step(q, k_new, v_new, k_cache, v_cache, page_table, qo_indptr, prefix_len, n_decode, max_kv_len,
                   out=None, lse=None, workspace=None, sm_scale=None, stream=None):
    """KV append + decode rows (split-KV) + prefill chunks (extend) in one call."""
    total_q, h_q, d = q.shape
    num_pages, page_size, h_kv, _ = k_cache.shape
    n_seqs = prefix_len.numel()
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = alloc_workspace(n_seqs, total_q, h_q, h_kv, d, max_kv_len, q.device)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d)
    _check(_lib.cpe_mixed_step(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), num_pages,
                               _ptr(page_table), page_table.shape[1], _ptr(qo_indptr), _ptr(prefix_len), n_seqs,
                               n_decode, total_q, max_kv_len, h_q, h_kv, d, page_size, sm_scale, _dtype(q),
                               _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(), _stream(stream)),
           "cpe_mixed_step")
    return out, lse


def cpe_decode_attention_noalloc(q, k_cache, v_cache, page_table, prefix_len, max_kv_len, out=None, lse=None,
                                 sm_scale=None, stream=None):
    """cpe_decode_attention without a workspace: for callers that cannot allocate
    device memory, the split partials live in the library's fixed 8 MiB device
    array (see include/cpe.h for its limits).  ``out`` must be given by such a
    caller; passing None lets torch allocate it here, for convenience only."""
    n_seqs, h_q, d = q.shape
    num_pages, page_size, h_kv, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d)
    _check(_lib.cpe_decode_attention_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), num_pages, _ptr(page_table),
                                             page_table.shape[1], _ptr(prefix_len), n_seqs, max_kv_len, h_q, h_kv,
                                             d, page_size, sm_scale, _dtype(q), _ptr(out), _ptr(lse),
                                             _stream(stream)), "cpe_decode_attention_noalloc")
    return out, lse


def cpe_get_device_status(stream=None):
    """Synchronise the stream; return (status, detail) of the device status word and clear it."""
    detail = _i32(0)
    st = _lib.cpe_get_device_status(_stream(stream), ctypes.byref(detail))
    return st, detail.value


def cpe_set_wait_limit_ns(ns: int) -> int:
    return int(_lib.cpe_set_wait_limit_ns(ns))


def cpe_status_string(status: int) -> str:
    return _lib.cpe_status_string(status).decode()


def cpe_last_error() -> str:
    return _lib.cpe_last_error().decode()


def cpe_launch_count() -> int:
    return int(_lib.cpe_launch_count())
