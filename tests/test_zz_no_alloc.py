"""ppa_prefill_noalloc: the entry point for callers that cannot allocate device memory (for
example a plugin inside a host framework that owns the device memory pool and gives it no
allocator). Its scratch lives in the library's static device array instead of a
caller-allocated workspace. Its output must match ppa_prefill's, call after call, although
every call reuses the array the previous call left behind.

This file is named so that pytest collects it last."""
import numpy as np
import pytest
import torch

from oracle import ref
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
    # Several different batches back to back: each call finds the previous call's plan in the
    # shared array and must not be affected by it. Both entry points run the same kernels on
    # the same inputs (an fp8 cache is widened inside the attention kernel by both: the
    # fixed scratch holds no bf16 staging), so the outputs must be bitwise equal.
    cases = [wl.mixed(544, False, seed=31, scale=1 / 16, num_seqs=5),
             wl.clamped_mm(seed=32, scale=1 / 32, num_seqs=2, num_ranges=2),
             wl.mixed(544, False, kv_dtype="fp8_e4m3", seed=33, scale=1 / 16, num_seqs=3),
             wl.mixed(544, False, seed=31, scale=1 / 16, num_seqs=5)]
    for i, case in enumerate(cases):
        fp8 = case.kv_dtype != "bf16"
        dc = binding.DeviceCase(case, flags_extra=binding.PPA_FLAG_FP8_INKERNEL if fp8 else 0)
        dc.run()
        torch.cuda.synchronize()
        assert dc.read_status() == binding.PPA_OK
        out = torch.full_like(dc.out, float("nan"))
        _noalloc(dc, out)
        torch.cuda.synchronize()
        assert dc.read_status() == binding.PPA_OK
        assert torch.equal(out, dc.out), f"noalloc {case.name}: differs from ppa_prefill"
        if i == 0:  # and against the oracle directly
            assert_close(out.float().cpu().numpy(), ref.attention(case.numpy_inputs()),
                         f"noalloc {case.name} vs oracle")


def test_noalloc_runs_split_kv_batches_unsplit():
    """kv_split_tiles does not fit the fixed scratch: the batch runs unsplit, with the output
    of the unsplit ppa_prefill bit for bit, and of the split one within the tolerance."""
    case = wl.build_case("noalloc_split", [3000, 200], [1, 4], 8, 2, 128, 37, causal=True,
                         seed=34)
    split = binding.DeviceCase(case, kv_split_tiles=4)
    split.run()
    unsplit = binding.DeviceCase(case)
    unsplit.run()
    torch.cuda.synchronize()
    assert split.read_status() == binding.PPA_OK and unsplit.read_status() == binding.PPA_OK
    out = torch.full_like(split.out, float("nan"))
    assert _noalloc(split, out) == binding.PPA_OK
    torch.cuda.synchronize()
    assert split.read_status() == binding.PPA_OK
    assert torch.equal(out, unsplit.out)
    assert_close(out.float().cpu().numpy(), split.out.float().cpu().numpy(), "noalloc split")


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
