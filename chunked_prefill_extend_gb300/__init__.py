"""Chunked-prefill extend attention for GB300 (sm_103a).

The compute path is the C-ABI library ``libcpe.so`` built from ``csrc/``;
``chunked_prefill_extend_gb300.cpe`` is its thin ctypes binding.  Importing
the package itself loads nothing, so the seeded workload generators in
``workloads`` can be used without the CUDA library.
"""
__all__ = ["cpe", "workloads"]
