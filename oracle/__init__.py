"""Float64 CPU oracle for chunked-prefill extend attention (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's
``cpu_baseline`` / ``--impl reference`` legs may import this package.  It shares
no code with the CUDA path: the attention arithmetic is plain C in
``cpe_oracle.c`` (compiled with gcc), the planners are plain Python in
``plan.py``.  Every function cites the page it follows in its own source.

Inputs are the exact fp32 / bf16 values the GPU sees (torch CPU tensors), and
results come back as float64 numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np
import torch

from .plan import Chunk, budget_truncate, effective_input_length, plan_chunks, plan_mixed_step, plan_schedule

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cpe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

F32, BF16 = 0, 1

__all__ = ["Chunk", "budget_truncate", "effective_input_length", "plan_chunks", "plan_mixed_step", "plan_schedule",
           "build", "extend_attention", "extend_attention_two_stage", "causal_attention",
           "kv_append", "num_threads", "set_fault"]


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (OpenMP) into oracle/liboracle.so."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", _SRC,
                               "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i32p = ctypes.c_void_p
        attn_args = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, i32p,
                     ctypes.c_int, i32p, i32p, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                     ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_void_p,
                     ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_extend_attention.argtypes = attn_args
        lib.oracle_extend_attention_two_stage.argtypes = attn_args
        lib.oracle_causal_attention.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                                ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_kv_append.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_int64, i32p, ctypes.c_int,
                                         i32p, i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int]
        lib.oracle_set_fault.argtypes = [ctypes.c_int]
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def num_threads() -> int:
    """Threads the oracle's OpenMP loops use."""
    return int(_load().oracle_num_threads())


def set_fault(code: int) -> None:
    """Plant a deliberate mistake (tests of the pins only): 0 none, 1 diagonal
    key dropped, 2 wrong softmax scale, 3 wrong GQA head map."""
    _load().oracle_set_fault(int(code))


def _raw(t: torch.Tensor):
    """Contiguous CPU tensor and its dtype code; keeps the tensor alive."""
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.float32:
        return t, F32
    if t.dtype == torch.bfloat16:
        return t, BF16
    raise TypeError(f"oracle takes float32 or bfloat16, got {t.dtype}")


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a.cpu() if isinstance(a, torch.Tensor) else a,
                                           dtype=np.int32))


def _attn(fn, q, k_cache, v_cache, page_table, qo_indptr, prefix_len, h_q, h_kv, scale, rows):
    qt, dt = _raw(q)
    kt, dk = _raw(k_cache)
    vt, dv = _raw(v_cache)
    if not (dt == dk == dv):
        raise TypeError("q, k_cache and v_cache must share a dtype")
    d = qt.shape[-1]
    page_size = kt.shape[1]
    pt = _i32(page_table)
    qo = _i32(qo_indptr)
    pl = _i32(prefix_len)
    n_seqs = len(pl)
    total_q = int(qo[-1])
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    if rows is not None:
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nr = len(rows)
    else:
        nr = total_q
    out = np.zeros((nr, h_q, d), dtype=np.float64)
    lse = np.zeros((nr, h_q), dtype=np.float64)
    rc = fn(qt.data_ptr(), kt.data_ptr(), vt.data_ptr(), dt, pt.ctypes.data, pt.shape[1],
            qo.ctypes.data, pl.ctypes.data, n_seqs, total_q, h_q, h_kv, d, page_size,
            float(scale), rows.ctypes.data if rows is not None else None, nr,
            out.ctypes.data, lse.ctypes.data)
    if rc != 0:
        raise RuntimeError(f"oracle attention failed ({rc})")
    return out, lse


def extend_attention(q, k_cache, v_cache, page_table, qo_indptr, prefix_len, h_q, h_kv,
                     scale=None, rows=None):
    """Direct form of the extend output o_i (one softmax over keys [0, P+i]).

    q [total_q, H_q, d]; caches [num_pages, page_size, H_kv, d]; page_table
    [n_seqs, max_pages]; rows: optional global query rows to compute.
    Returns (out [rows, H_q, d], lse [rows, H_q]) as float64.
    """
    return _attn(_load().oracle_extend_attention, q, k_cache, v_cache, page_table, qo_indptr,
                 prefix_len, h_q, h_kv, scale, rows)


def extend_attention_two_stage(q, k_cache, v_cache, page_table, qo_indptr, prefix_len, h_q, h_kv,
                               scale=None, rows=None):
    """Stage 1 (prefix rectangle) + Stage 2 (causal triangle) + LSE merge."""
    return _attn(_load().oracle_extend_attention_two_stage, q, k_cache, v_cache, page_table,
                 qo_indptr, prefix_len, h_q, h_kv, scale, rows)


def causal_attention(q, k, v, h_q, h_kv, scale=None):
    """One-shot causal attention on contiguous q [N,H_q,d], k/v [N,H_kv,d]."""
    qt, dt = _raw(q)
    kt, _ = _raw(k)
    vt, _ = _raw(v)
    n, _, d = qt.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = np.zeros((n, h_q, d), dtype=np.float64)
    lse = np.zeros((n, h_q), dtype=np.float64)
    rc = _load().oracle_causal_attention(qt.data_ptr(), kt.data_ptr(), vt.data_ptr(), dt, n, h_q,
                                         h_kv, d, float(scale), out.ctypes.data, lse.ctypes.data)
    if rc != 0:
        raise RuntimeError(f"oracle causal attention failed ({rc})")
    return out, lse


def kv_append(k_new, v_new, k_cache, v_cache, page_table, qo_indptr, prefix_len):
    """Byte scatter of the new rows into the paged caches (in place, CPU tensors)."""
    for t in (k_new, v_new, k_cache, v_cache):
        if t.device.type != "cpu" or not t.is_contiguous():
            raise ValueError("kv_append oracle works in place on contiguous CPU tensors")
    num_pages, page_size, h_kv, d = k_cache.shape
    pt = _i32(page_table)
    qo = _i32(qo_indptr)
    pl = _i32(prefix_len)
    rc = _load().oracle_kv_append(k_new.data_ptr(), v_new.data_ptr(), k_cache.data_ptr(),
                                  v_cache.data_ptr(), num_pages, pt.ctypes.data, pt.shape[1],
                                  qo.ctypes.data, pl.ctypes.data, len(pl), h_kv, d, page_size,
                                  k_cache.element_size())
    if rc != 0:
        raise RuntimeError("oracle kv_append: position beyond the page table or bad page id")
