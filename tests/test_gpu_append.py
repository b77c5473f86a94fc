"""KV append into the paged cache and cache-sourced attention (new tokens' K/V read back from
the cache) on the GPU, against the oracle: the appended caches bit-exact (bf16 values, fp8
codes), the attention output within the bf16 tolerance, and the same output as the path that
reads k_new / v_new."""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import ref
from paged_kv_prefix_gb300 import binding
from paged_kv_prefix_gb300 import workloads as wl
from tests.gpu_util import assert_close

pytestmark = pytest.mark.gpu

IN_CACHE = binding.PPA_FLAG_KV_IN_CACHE


def _ragged(D, page, kv="bf16", seed=0, window_left=0, mm=None):
    rng = np.random.default_rng(seed)
    ctx = [0, 1, 127, int(rng.integers(200, 500)), 64, 0]
    qlen = [5, 0, 130, int(rng.integers(50, 200)), 1, 77]
    return wl.build_case("append", ctx, qlen, 4, 2, D, page, causal=True, window_left=window_left,
                         mm_ranges=mm, clamp_mm=mm is not None, kv_dtype=kv, seed=seed)


def _appended_inputs(case):
    inp = case.numpy_inputs()
    k, v = ref.append_kv(inp)
    app = dict(inp)
    app["k_cache"], app["v_cache"], app["kv_in_cache"] = k, v, True
    return app


def _run_append(case, flags=0):
    dc = binding.DeviceCase(case, flags_extra=flags)
    dc.append()
    torch.cuda.synchronize()
    assert dc.read_status() == binding.PPA_OK
    return dc


def _cache_np(t, kv):
    return t.float().cpu().numpy() if kv == "bf16" else t.cpu().numpy()


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("page", [1, 5, 16, 37, 544])
def test_append_bit_exact(kv, D, page):
    case = _ragged(D, page, kv, seed=D + page)
    dc = _run_append(case)
    app = _appended_inputs(case)
    for which in ("k", "v"):
        got = _cache_np(getattr(dc, f"{which}_cache"), kv)
        want = app[f"{which}_cache"]
        if kv == "bf16":  # untouched slots keep their NaN poison
            assert np.array_equal(got, want, equal_nan=True), which
        else:
            assert np.array_equal(got, want), which


def test_append_fp8_saturates_like_the_oracle():
    case = _ragged(128, 16, "fp8_e4m3", seed=5)
    case = dataclasses.replace(case, k_scale=1e-3, v_scale=3e-3)  # |x| / scale well past 448
    dc = _run_append(case)
    app = _appended_inputs(case)
    got = dc.k_cache.cpu().numpy()
    assert np.array_equal(got, app["k_cache"])
    assert (got == 0x7E).any() and (got == 0xFE).any()  # saturated codes of both signs
    assert np.array_equal(dc.v_cache.cpu().numpy(), app["v_cache"])


FP8_PATHS = [0, binding.PPA_FLAG_FP8_INKERNEL]


@pytest.mark.parametrize("kv,fp8_path", [("bf16", 0), ("fp8_e4m3", FP8_PATHS[0]),
                                         ("fp8_e4m3", FP8_PATHS[1])],
                         ids=["bf16", "fp8_prepass", "fp8_inkernel"])
@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("page", [5, 16, 544])
def test_cache_sourced_attention_parity(kv, fp8_path, D, page):
    case = _ragged(D, page, kv, seed=3 * D + page, window_left=int(page % 2) * 90)
    dc = _run_append(case, IN_CACHE | fp8_path)
    dc.run()
    torch.cuda.synchronize()
    assert dc.read_status() == binding.PPA_OK
    want = ref.attention(_appended_inputs(case))
    assert_close(dc.out.float().cpu().numpy(), want, f"cache-sourced {kv} D{D} P{page}")


def test_cache_sourced_with_multimodal_ranges():
    mm = np.array([[[0, 0]], [[0, 0]], [[10, 90]], [[100, 300]], [[0, 0]], [[3, 40]]])
    case = _ragged(128, 16, "bf16", seed=9, window_left=50, mm=mm)
    dc = _run_append(case, IN_CACHE)
    dc.run()
    torch.cuda.synchronize()
    assert dc.read_status() == binding.PPA_OK
    assert_close(dc.out.float().cpu().numpy(), ref.attention(_appended_inputs(case)), "mm")


@pytest.mark.parametrize("D", [64, 128, 256])
def test_cache_sourced_equals_the_new_token_tensors_bitwise(D):
    """bf16: the appended rows hold the same values, so both paths compute the same thing."""
    case = _ragged(D, 37, "bf16", seed=D)
    ref_dc = binding.DeviceCase(case)
    ref_dc.run()
    dc = _run_append(case, IN_CACHE)
    dc.plan()
    dc.attend()
    torch.cuda.synchronize()
    assert ref_dc.read_status() == binding.PPA_OK and dc.read_status() == binding.PPA_OK
    assert torch.equal(dc.out.float(), ref_dc.out.float())


def test_short_block_table_rows_are_rejected_on_the_device():
    """Rows must cover c + n positions for the append and for cache-sourced attention."""
    case = wl.build_case("short", [40], [30], 4, 2, 64, 16, causal=True, seed=11)
    dc = binding.DeviceCase(case, flags_extra=IN_CACHE)
    before = dc.k_cache.clone()
    dc.dims.max_pages_per_seq = 4  # covers 64 positions, the sequence needs 70
    dc.block_table = dc.block_table[:, :4].contiguous()
    binding.ppa_append_kv(dc.dims, dc.k_new, dc.v_new, dc.k_cache, dc.v_cache, dc.block_table,
                          dc.cu_query_lens, dc.context_lens, dc.k_scale, dc.v_scale, dc.status)
    assert dc.read_status() == binding.PPA_ERR_INVALID
    assert torch.equal(dc.k_cache.view(torch.int16), before.view(torch.int16))
    dc.status.zero_()
    dc.out.fill_(7.0)
    dc.run()
    assert dc.read_status() == binding.PPA_ERR_INVALID
    assert bool((dc.out == 7.0).all())  # the plan scheduled nothing


def test_null_new_tensors_need_the_flag():
    case = wl.tiny()
    dc = binding.DeviceCase(case)
    code = binding.ppa_prefill(dc.dims, dc.q, None, None, dc.k_cache, dc.v_cache, dc.block_table,
                               dc.cu_query_lens, dc.context_lens, None, dc.k_scale, dc.v_scale,
                               dc.out, dc.workspace, dc.status, check=False)
    assert code == binding.PPA_ERR_UNSUPPORTED
