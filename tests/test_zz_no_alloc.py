"""ppa_prefill_noalloc: the entry point for callers that cannot allocate device memory (for
example a plugin inside a host framework that owns the device memory pool and gives it no
allocator). Its scratch lives in the library's static device array instead of a
caller-allocated workspace. Its output must match ppa_prefill's, call after call, although
every call reuses the array the previous call left behind.

This file is named so that pytest collects it last."""
import numpy as np
import pytest
import torch

from paged_kv_prefix_gb300 import binding
from paged_kv_prefix_gb300 import workloads as wl
from tests.gpu_util import assert_close

pytestmark = pytest.mark.gpu


def _noalloc(dc, out):
    return binding.ppa_prefill_noalloc(dc.dims, dc.q, dc.k_new, dc.v_new, dc.k_cache,
                                       dc.v_cache, dc.block_table, dc.cu_query_lens,
                                       dc.context_lens, dc.mm_ranges, dc.k_scale, dc.v_scale,
                                       out, dc.status)


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    # Two different batches back to back: the second call finds the first call's plan in
    # the shared array and must not be affected by it.
    cases = [wl.mixed(544, True, seed=31, scale=1 / 16, num_seqs=5),
             wl.clamped_mm(seed=32, scale=1 / 32, num_seqs=2, num_ranges=2),
             # fp8: the fixed scratch holds no bf16 staging, so the kernel widens the rows
             wl.mixed(544, False, kv_dtype="fp8_e4m3", seed=33, scale=1 / 16, num_seqs=3)]
    for case in cases:
        dc = binding.DeviceCase(case)
        dc.run()
        torch.cuda.synchronize()
        assert dc.read_status() == binding.PPA_OK
        want = dc.out.float().cpu().numpy()
        out = torch.full_like(dc.out, float("nan"))
        _noalloc(dc, out)
        torch.cuda.synchronize()
        assert dc.read_status() == binding.PPA_OK
        assert_close(out.float().cpu().numpy(), want, f"noalloc {case.name}")


def test_noalloc_runs_split_kv_batches_unsplit():
    """kv_split_tiles does not fit the fixed scratch: the batch runs unsplit, same output."""
    case = wl.build_case("noalloc_split", [3000, 200], [1, 4], 8, 2, 128, 37, causal=True,
                         seed=34)
    dc = binding.DeviceCase(case, kv_split_tiles=4)
    dc.run()
    torch.cuda.synchronize()
    assert dc.read_status() == binding.PPA_OK
    out = torch.full_like(dc.out, float("nan"))
    assert _noalloc(dc, out) == binding.PPA_OK
    torch.cuda.synchronize()
    assert dc.read_status() == binding.PPA_OK
    assert_close(out.float().cpu().numpy(), dc.out.float().cpu().numpy(), "noalloc split")


def test_noalloc_rejects_a_batch_larger_than_its_scratch():
    case = wl.tiny()
    dc = binding.DeviceCase(case)
    dims = binding.dims_for(case)
    dims.total_q = 20_000_000  # needs ~6 MB of scratch; rejected on the host, nothing launched
    assert binding.ppa_workspace_bytes(dims) > binding.PPA_NOALLOC_WORKSPACE_BYTES
    code = binding.ppa_prefill_noalloc(dims, dc.q, dc.k_new, dc.v_new, dc.k_cache, dc.v_cache,
                                       dc.block_table, dc.cu_query_lens, dc.context_lens, None,
                                       dc.k_scale, dc.v_scale, dc.out, dc.status, check=False)
    assert code == binding.PPA_ERR_UNSUPPORTED
