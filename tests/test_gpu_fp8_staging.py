"""fp8 caches dequantised into workspace, with the staging sized by ppa_dims.max_cache_tokens.

Only the live cache key tiles are staged, packed in sequence order, so a bound on the cached
positions the queries attend to (the sum of context lengths, or the live positions when
windows hide the rest) sizes the workspace. The staged values and the attention are those of
the unbounded staging: outputs must be bitwise equal to it, and match the oracle. A bound
below what the batch needs is reported as PPA_ERR_INVALID and nothing is computed."""
import numpy as np
import pytest
import torch

from oracle import ref
from paged_kv_prefix_gb300 import binding
from paged_kv_prefix_gb300 import workloads as wl
from tests.gpu_util import assert_close

pytestmark = pytest.mark.gpu


def _run(case, **kw):
    dc = binding.DeviceCase(case, **kw)
    dc.out.fill_(float("nan"))
    if dc.dims.flags & binding.PPA_FLAG_KV_IN_CACHE:
        dc.append()
    dc.run()
    torch.cuda.synchronize()
    return dc, dc.read_status()


def _live_cache_tokens(case):
    dc = binding.DeviceCase(case)
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
    binding.ppa_live_kv_tokens(dc.dims, dc.cu_query_lens, dc.context_lens, dc.mm_ranges, cnt)
    return int(cnt.item())


@pytest.mark.parametrize("windowed", [False, True])
@pytest.mark.parametrize("page", [37, 544])
def test_bounded_staging_equals_unbounded_bitwise(windowed, page):
    case = wl.mixed(page, windowed, kv_dtype="fp8_e4m3", seed=50 + page, scale=1 / 8, num_seqs=5)
    full, st = _run(case)
    assert st == binding.PPA_OK
    bound = _live_cache_tokens(case) if windowed else int(case.context_lens.sum())
    packed, st = _run(case, max_cache_tokens=bound)
    assert st == binding.PPA_OK
    assert packed.workspace.numel() < full.workspace.numel()
    assert torch.equal(packed.out, full.out)
    assert_close(packed.out.float().cpu().numpy(), ref.attention(case.numpy_inputs()), case.name)


def test_bounded_staging_with_split_kv_and_ranges():
    mm = np.array([[[100, 900]], [[0, 0]], [[1000, 1990]], [[0, 0]]])
    case = wl.build_case("fp8_split", [2000, 700, 2500, 40], [1, 5, 3, 200], 8, 2, 128, 37,
                         causal=True, window_left=600, mm_ranges=mm, clamp_mm=True,
                         kv_dtype="fp8_e4m3", seed=51)
    dc, st = _run(case, kv_split_tiles=2, max_cache_tokens=_live_cache_tokens(case))
    assert st == binding.PPA_OK
    assert_close(dc.out.float().cpu().numpy(), ref.attention(case.numpy_inputs()), "split mm")


def test_bounded_staging_cache_sourced():
    case = wl.build_case("fp8_cached", [300, 0, 1200], [100, 70, 1], 8, 4, 256, 16, causal=True,
                         kv_dtype="fp8_e4m3", seed=52)
    bound = int(case.context_lens.sum()) + case.total_q  # cache positions c + n
    dc, st = _run(case, flags_extra=binding.PPA_FLAG_KV_IN_CACHE, max_cache_tokens=bound)
    assert st == binding.PPA_OK
    inp = case.numpy_inputs()
    inp["k_cache"], inp["v_cache"] = ref.append_kv(inp)
    inp["kv_in_cache"] = True
    assert_close(dc.out.float().cpu().numpy(), ref.attention(inp), case.name)


def test_too_small_a_bound_is_rejected_on_the_device():
    case = wl.mixed(544, False, kv_dtype="fp8_e4m3", seed=53, scale=1 / 8, num_seqs=5)
    dc, st = _run(case, max_cache_tokens=128)  # far below the batch's live cache positions
    assert st == binding.PPA_ERR_INVALID
    assert torch.isnan(dc.out.float()).all()  # nothing was computed
