"""The attention kernel's bounded waits, exercised without a fault.

``ppa_debug_prefill_stalled`` runs a batch with every device wait limited to a few
milliseconds while the first CTA never loads its first query tile: the MMA issuer's wait for
it runs out. The kernel must report PPA_ERR_TIMEOUT through the status word, leave every
loop, wait for its copies in flight, retire its tensor-core work, free TMEM and return; the
context stays usable, and the next ordinary call on the same stream matches the oracle."""
import time

import pytest
import torch

from oracle import ref
from paged_kv_prefix_gb300 import binding
from paged_kv_prefix_gb300 import workloads as wl
from tests.gpu_util import assert_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("head_dim", [64, 128])
def test_expired_wait_reports_timeout_and_the_next_call_is_exact(head_dim):
    case = wl.build_case("stall", [0, 300, 1200], [500, 200, 90], 8, 2, head_dim, 37,
                         causal=True, seed=40 + head_dim)
    dc = binding.DeviceCase(case)
    t0 = time.perf_counter()
    code = binding.ppa_debug_prefill_stalled(
        dc.dims, dc.q, dc.k_new, dc.v_new, dc.k_cache, dc.v_cache, dc.block_table,
        dc.cu_query_lens, dc.context_lens, dc.mm_ranges, dc.k_scale, dc.v_scale, dc.out,
        dc.workspace, dc.status, 20_000)
    assert code == binding.PPA_OK
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert dc.read_status() == binding.PPA_ERR_TIMEOUT
    assert elapsed < 1.5, f"the stalled launch took {elapsed:.2f} s with a 20 ms wait limit"
    # the same stream, workspace and buffers: an ordinary call is exact again
    dc.out.zero_()
    dc.run()
    torch.cuda.synchronize()
    assert dc.read_status() == binding.PPA_OK
    assert_close(dc.out.float().cpu().numpy(), ref.attention(case.numpy_inputs()), case.name)


def test_stalled_entry_point_rejects_the_pair_kernel_and_a_zero_limit():
    case = wl.build_case("stall256", [0], [64], 4, 2, 256, 16, causal=True, seed=3)
    dc = binding.DeviceCase(case)
    args = (dc.dims, dc.q, dc.k_new, dc.v_new, dc.k_cache, dc.v_cache, dc.block_table,
            dc.cu_query_lens, dc.context_lens, dc.mm_ranges, dc.k_scale, dc.v_scale, dc.out,
            dc.workspace, dc.status)
    assert (binding.ppa_debug_prefill_stalled(*args, 1000, check=False)
            == binding.PPA_ERR_UNSUPPORTED)
    dc.dims.head_dim = 128
    assert binding.ppa_debug_prefill_stalled(*args, 0, check=False) == binding.PPA_ERR_INVALID
