"""Chunked-prefill attention over a paged KV cache, for GB300 (sm_103a).

The compute lives in ``libppa.so`` (CUDA kernels behind a C ABI declared in
``include/ppa.h``); :mod:`paged_kv_prefix_gb300.binding` is a thin ctypes layer over it.
The library is loaded on first use, and a missing or stale build raises instead of
falling back to anything else.
"""

__all__ = ["binding", "workloads"]
