"""ctypes binding for ``libppa.so`` (C ABI in ``include/ppa.h``).

Argument marshalling only: every function here forwards to the C entry point of the same
name. Tensors are passed by ``data_ptr()``; streams default to torch's current CUDA stream.
There is no fallback: if the library is missing, :func:`lib` raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libppa.so")

PPA_OK = 0
PPA_ERR_INVALID = 1
PPA_ERR_UNSUPPORTED = 2
PPA_ERR_CUDA = 3
PPA_ERR_TIMEOUT = 4
PPA_ERR_BAD_PAGE = 5

PPA_KV_BF16 = 0
PPA_KV_FP8_E4M3 = 1

PPA_FLAG_CAUSAL = 1
PPA_FLAG_CLAMP_MM = 2
PPA_FLAG_NO_PRUNE = 4
PPA_FLAG_FP8_INKERNEL = 8
PPA_FLAG_KV_IN_CACHE = 16


class PpaDims(ctypes.Structure):
    _fields_ = [
        ("num_seqs", ctypes.c_int),
        ("total_q", ctypes.c_int),
        ("num_q_heads", ctypes.c_int),
        ("num_kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int),
        ("page_size", ctypes.c_int),
        ("num_pages", ctypes.c_int),
        ("max_pages_per_seq", ctypes.c_int),
        ("max_mm_ranges", ctypes.c_int),
        ("window_left", ctypes.c_int),
        ("window_right", ctypes.c_int),
        ("kv_dtype", ctypes.c_int),
        ("flags", ctypes.c_uint),
        ("sm_scale", ctypes.c_float),
        ("chunk_size", ctypes.c_int),
        ("chunk_lookback", ctypes.c_int),
        ("kv_split_tiles", ctypes.c_int),
        ("seq_causal", ctypes.c_void_p),  # device int32[num_seqs] or None
        ("max_cache_tokens", ctypes.c_int),
    ]


class PpaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (code {code})")


_lib: Optional[ctypes.CDLL] = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_DIMS = ctypes.POINTER(PpaDims)

_SIGNATURES = {
    "ppa_workspace_bytes": (ctypes.c_size_t, [_DIMS]),
    "ppa_prefill": (_I, [_DIMS, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "ppa_plan": (_I, [_DIMS, _P, _P, _P, _P, _P, _P]),
    "ppa_attend": (_I, [_DIMS, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "ppa_prefill_noalloc": (_I, [_DIMS, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                 _P]),
    "ppa_query_tiles": (None, [_DIMS, ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "ppa_tile_bounds": (_I, [_DIMS, _I, _I, _P, _P, _P, _P, _P, _P]),
    "ppa_append_kv": (_I, [_DIMS, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "ppa_debug_mask": (_I, [_DIMS, _I, _P, _P, _P, _P, _I, _I, _P]),
    "ppa_live_pairs": (_I, [_DIMS, _P, _P, _P, _P, _P]),
    "ppa_live_kv_tokens": (_I, [_DIMS, _P, _P, _P, _P, _P]),
    "ppa_debug_e4m3_to_bf16": (_I, [_P, _P, _I, _P]),
    "ppa_debug_prefill_stalled": (_I, [_DIMS, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                       _P, _P, ctypes.c_uint, _P]),
    "ppa_read_status": (_I, [_P, _P]),
    "ppa_status_string": (ctypes.c_char_p, [_I]),
    "ppa_version": (_I, []),
}


def lib() -> ctypes.CDLL:
    """Loads the in-tree ``libppa.so`` (built by ``paged_kv_prefix_gb300.build``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m paged_kv_prefix_gb300.build` "
                "(there is no CPU fallback)")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def status_string(code: int) -> str:
    return lib().ppa_status_string(int(code)).decode()


def _check(code: int, where: str) -> None:
    if code != PPA_OK:
        raise PpaError(code, where)


# --------------------------------------------------------------------------------------
# Same-name wrappers
# --------------------------------------------------------------------------------------
def ppa_workspace_bytes(dims: PpaDims) -> int:
    return int(lib().ppa_workspace_bytes(ctypes.byref(dims)))


def ppa_query_tiles(dims: PpaDims) -> tuple[int, int]:
    tq, tn = ctypes.c_int(0), ctypes.c_int(0)
    lib().ppa_query_tiles(ctypes.byref(dims), ctypes.byref(tq), ctypes.byref(tn))
    return tq.value, tn.value


def ppa_prefill(dims: PpaDims, q, k_new, v_new, k_cache, v_cache, block_table, cu_query_lens,
                context_lens, mm_ranges, k_scale, v_scale, out, workspace, device_status,
                stream=None, check: bool = True) -> int:
    code = lib().ppa_prefill(ctypes.byref(dims), _ptr(q), _ptr(k_new), _ptr(v_new),
                             _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                             _ptr(cu_query_lens), _ptr(context_lens), _ptr(mm_ranges),
                             _ptr(k_scale), _ptr(v_scale), _ptr(out), _ptr(workspace),
                             _ptr(device_status), _stream(stream))
    if check:
        _check(code, "ppa_prefill")
    return code


PPA_NOALLOC_WORKSPACE_BYTES = 2 << 20


def ppa_prefill_noalloc(dims: PpaDims, q, k_new, v_new, k_cache, v_cache, block_table,
                        cu_query_lens, context_lens, mm_ranges, k_scale, v_scale, out,
                        device_status, stream=None, check: bool = True) -> int:
    """ppa_prefill without a workspace argument, for callers that cannot allocate device
    memory; the scratch lives in the library's static device array (shared by all calls on
    a device, so calls must not overlap on the GPU)."""
    code = lib().ppa_prefill_noalloc(ctypes.byref(dims), _ptr(q), _ptr(k_new), _ptr(v_new),
                                     _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                     _ptr(cu_query_lens), _ptr(context_lens), _ptr(mm_ranges),
                                     _ptr(k_scale), _ptr(v_scale), _ptr(out),
                                     _ptr(device_status), _stream(stream))
    if check:
        _check(code, "ppa_prefill_noalloc")
    return code


def ppa_plan(dims: PpaDims, cu_query_lens, context_lens, mm_ranges, workspace, device_status,
             stream=None, check: bool = True) -> int:
    code = lib().ppa_plan(ctypes.byref(dims), _ptr(cu_query_lens), _ptr(context_lens),
                          _ptr(mm_ranges), _ptr(workspace), _ptr(device_status), _stream(stream))
    if check:
        _check(code, "ppa_plan")
    return code


def ppa_attend(dims: PpaDims, q, k_new, v_new, k_cache, v_cache, block_table, cu_query_lens,
               context_lens, mm_ranges, k_scale, v_scale, out, workspace, device_status,
               stream=None, check: bool = True) -> int:
    code = lib().ppa_attend(ctypes.byref(dims), _ptr(q), _ptr(k_new), _ptr(v_new),
                            _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                            _ptr(cu_query_lens), _ptr(context_lens), _ptr(mm_ranges),
                            _ptr(k_scale), _ptr(v_scale), _ptr(out), _ptr(workspace),
                            _ptr(device_status), _stream(stream))
    if check:
        _check(code, "ppa_attend")
    return code


def ppa_append_kv(dims: PpaDims, k_new, v_new, k_cache, v_cache, block_table, cu_query_lens,
                  context_lens, k_scale, v_scale, device_status, stream=None,
                  check: bool = True) -> int:
    code = lib().ppa_append_kv(ctypes.byref(dims), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                               _ptr(v_cache), _ptr(block_table), _ptr(cu_query_lens),
                               _ptr(context_lens), _ptr(k_scale), _ptr(v_scale),
                               _ptr(device_status), _stream(stream))
    if check:
        _check(code, "ppa_append_kv")
    return code


def ppa_tile_bounds(dims: PpaDims, tq: int, tn: int, cu_query_lens, context_lens, mm_ranges,
                    bounds_out, device_status, stream=None, check: bool = True) -> int:
    code = lib().ppa_tile_bounds(ctypes.byref(dims), tq, tn, _ptr(cu_query_lens),
                                 _ptr(context_lens), _ptr(mm_ranges), _ptr(bounds_out),
                                 _ptr(device_status), _stream(stream))
    if check:
        _check(code, "ppa_tile_bounds")
    return code


def ppa_debug_mask(dims: PpaDims, seq: int, cu_query_lens, context_lens, mm_ranges, bitmap_out,
                   max_rows: int, words_per_row: int, stream=None, check: bool = True) -> int:
    code = lib().ppa_debug_mask(ctypes.byref(dims), seq, _ptr(cu_query_lens), _ptr(context_lens),
                                _ptr(mm_ranges), _ptr(bitmap_out), max_rows, words_per_row,
                                _stream(stream))
    if check:
        _check(code, "ppa_debug_mask")
    return code


def ppa_live_pairs(dims: PpaDims, cu_query_lens, context_lens, mm_ranges, count_out, stream=None,
                   check: bool = True) -> int:
    code = lib().ppa_live_pairs(ctypes.byref(dims), _ptr(cu_query_lens), _ptr(context_lens),
                                _ptr(mm_ranges), _ptr(count_out), _stream(stream))
    if check:
        _check(code, "ppa_live_pairs")
    return code


def ppa_live_kv_tokens(dims: PpaDims, cu_query_lens, context_lens, mm_ranges, count_out,
                       stream=None, check: bool = True) -> int:
    code = lib().ppa_live_kv_tokens(ctypes.byref(dims), _ptr(cu_query_lens), _ptr(context_lens),
                                    _ptr(mm_ranges), _ptr(count_out), _stream(stream))
    if check:
        _check(code, "ppa_live_kv_tokens")
    return code


def ppa_debug_e4m3_to_bf16(codes, bf16_out, n: int, stream=None, check: bool = True) -> int:
    code = lib().ppa_debug_e4m3_to_bf16(_ptr(codes), _ptr(bf16_out), n, _stream(stream))
    if check:
        _check(code, "ppa_debug_e4m3_to_bf16")
    return code


def ppa_debug_prefill_stalled(dims: PpaDims, q, k_new, v_new, k_cache, v_cache, block_table,
                              cu_query_lens, context_lens, mm_ranges, k_scale, v_scale, out,
                              workspace, device_status, wait_limit_us: int, stream=None,
                              check: bool = True) -> int:
    """ppa_prefill with its device waits limited to ``wait_limit_us`` and the first CTA's
    query load withheld, so that the waits run out (tests of the timeout path)."""
    code = lib().ppa_debug_prefill_stalled(ctypes.byref(dims), _ptr(q), _ptr(k_new),
                                           _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                           _ptr(block_table), _ptr(cu_query_lens),
                                           _ptr(context_lens), _ptr(mm_ranges), _ptr(k_scale),
                                           _ptr(v_scale), _ptr(out), _ptr(workspace),
                                           _ptr(device_status), int(wait_limit_us),
                                           _stream(stream))
    if check:
        _check(code, "ppa_debug_prefill_stalled")
    return code


def ppa_read_status(device_status, stream=None) -> int:
    return int(lib().ppa_read_status(_ptr(device_status), _stream(stream)))


def ppa_status_string(code: int) -> str:
    return status_string(code)


def ppa_version() -> int:
    return int(lib().ppa_version())


# --------------------------------------------------------------------------------------
# Convenience: dims from a case, and a runner that owns workspace and status.
# --------------------------------------------------------------------------------------
def dims_for(case, flags_extra: int = 0) -> PpaDims:
    """``PpaDims`` describing a :class:`paged_kv_prefix_gb300.workloads.PrefillCase`."""
    flags = (PPA_FLAG_CAUSAL if case.causal else 0) | (PPA_FLAG_CLAMP_MM if case.clamp_mm else 0)
    return PpaDims(
        num_seqs=case.num_seqs, total_q=case.total_q, num_q_heads=case.num_q_heads,
        num_kv_heads=case.num_kv_heads, head_dim=case.head_dim, page_size=case.page_size,
        num_pages=case.num_pages, max_pages_per_seq=case.max_pages_per_seq,
        max_mm_ranges=case.max_mm_ranges, window_left=case.window_left,
        window_right=case.window_right,
        kv_dtype=PPA_KV_FP8_E4M3 if case.kv_dtype == "fp8_e4m3" else PPA_KV_BF16,
        flags=flags | flags_extra, sm_scale=case.sm_scale,
        chunk_size=getattr(case, "chunk_size", 0), chunk_lookback=getattr(case, "chunk_lookback", 0))


class DeviceCase:
    """A case's tensors on the GPU plus the output, workspace and status buffers."""

    def __init__(self, case, device="cuda", flags_extra: int = 0, kv_split_tiles: int = 0,
                 max_cache_tokens: int = 0):
        import torch
        self.case = case
        self.dims = dims_for(case, flags_extra)
        self.dims.kv_split_tiles = kv_split_tiles  # these two size the workspace below
        self.dims.max_cache_tokens = max_cache_tokens
        dev = torch.device(device)
        self.q = case.q.to(dev)
        self.k_new = case.k_new.to(dev)
        self.v_new = case.v_new.to(dev)
        self.k_cache = case.k_cache.to(dev)
        self.v_cache = case.v_cache.to(dev)
        self.block_table = case.block_table.to(dev)
        self.cu_query_lens = case.cu_query_lens.to(dev)
        self.context_lens = case.context_lens.to(dev)
        self.mm_ranges = None if case.mm_ranges is None else case.mm_ranges.to(dev)
        seq_causal = getattr(case, "seq_causal", None)
        self.seq_causal = None if seq_causal is None else seq_causal.to(dev)
        if self.seq_causal is not None:
            self.dims.seq_causal = self.seq_causal.data_ptr()
        self.k_scale = torch.tensor([case.k_scale], dtype=torch.float32, device=dev)
        self.v_scale = torch.tensor([case.v_scale], dtype=torch.float32, device=dev)
        self.out = torch.zeros_like(self.q)
        nbytes = max(256, ppa_workspace_bytes(self.dims))
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    def _new_kv(self):
        """k_new / v_new for the attention calls: NULL when the dims say the new tokens' K/V
        are read from the cache."""
        if self.dims.flags & PPA_FLAG_KV_IN_CACHE:
            return None, None
        return self.k_new, self.v_new

    def append(self, stream=None):
        """Writes the new tokens' K/V into the cache (ppa_append_kv)."""
        return ppa_append_kv(self.dims, self.k_new, self.v_new, self.k_cache, self.v_cache,
                             self.block_table, self.cu_query_lens, self.context_lens,
                             self.k_scale, self.v_scale, self.status, stream)

    def run(self, stream=None, out=None):
        k_new, v_new = self._new_kv()
        return ppa_prefill(self.dims, self.q, k_new, v_new, self.k_cache, self.v_cache,
                           self.block_table, self.cu_query_lens, self.context_lens,
                           self.mm_ranges, self.k_scale, self.v_scale,
                           self.out if out is None else out, self.workspace, self.status, stream)

    def plan(self, stream=None):
        return ppa_plan(self.dims, self.cu_query_lens, self.context_lens, self.mm_ranges,
                        self.workspace, self.status, stream)

    def attend(self, stream=None, out=None):
        k_new, v_new = self._new_kv()
        return ppa_attend(self.dims, self.q, k_new, v_new, self.k_cache, self.v_cache,
                          self.block_table, self.cu_query_lens, self.context_lens,
                          self.mm_ranges, self.k_scale, self.v_scale,
                          self.out if out is None else out, self.workspace, self.status, stream)

    def read_status(self, stream=None) -> int:
        return ppa_read_status(self.status, stream)
